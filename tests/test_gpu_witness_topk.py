"""GPU parity of the integer / selection kernels against the oracle, through
the C ABI: witness merge and witness table (bit-exact), top-K of given score
rows (bit-exact ids and scores)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import dsa as odsa
from oracle import witness as ow
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "witness_examples.json")))


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _dev(a, dtype=torch.int32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def test_printed_examples(B):
    c = GOLD["merge"][0]
    ids = _dev(np.array([c["learned"]], dtype=np.int32))
    B.witness_merge(ids, _dev(np.array([c["L"]])), c["keep"], c["S"], c["max_replacements"])
    assert ids.cpu().numpy()[0].tolist() == c["expected"]
    c = GOLD["serving"][0]
    ids = _dev(np.array([c["learned"]], dtype=np.int32))
    topk = len(c["learned"])
    B.witness_merge(ids, _dev(np.array([c["L"]])), topk - c["S"], c["S"], c["S"])
    assert ids.cpu().numpy()[0].tolist() == c["expected"]
    c = GOLD["witness_indices"][0]
    out = torch.empty((1, c["S"]), dtype=torch.int32, device="cuda")
    B.witness_indices(_dev(np.array([c["learned"]])), _dev(np.array([c["L"]])), c["S"], out)
    assert out.cpu().numpy()[0].tolist() == c["expected"]
    assert B.device_error() == 0


@pytest.mark.parametrize("seed,rows,topk,S,keep_mode", [
    (1, 64, 2048, 16, "serving"), (2, 128, 2048, 32, "serving"), (3, 37, 100, 64, "serving"),
    (4, 50, 33, 7, "random"), (5, 300, 8, 4, "random"), (6, 20, 64, 64, "random"), (7, 9, 5, 40, "serving"),
    (8, 5000, 64, 16, "serving"), (9, 6000, 37, 64, "random")])     # many rows: one warp per row
def test_merge_random_rows(B, seed, rows, topk, S, keep_mode):
    learned, ctx = wl.witness_rows(seed, rows, topk, L_min=-2, L_max=5000)
    rng = np.random.default_rng(seed + 100)
    if keep_mode == "serving":
        keep, maxr = max(topk - S, 0), S
    else:
        keep, maxr = int(rng.integers(0, topk + 1)), int(rng.integers(0, S + 3))
    ids = _dev(learned)
    B.witness_merge(ids, _dev(ctx), keep, S, maxr)
    ref = ow.apply_topology_witnesses(learned, topk, ctx, keep, S, maxr)
    assert np.array_equal(ids.cpu().numpy(), ref)
    tab = torch.empty((rows, S), dtype=torch.int32, device="cuda")
    B.witness_indices(_dev(learned), _dev(ctx), S, tab)
    assert np.array_equal(tab.cpu().numpy(), ow.topology_witness_indices(learned, topk, ctx, S))
    assert B.device_error() == 0


@pytest.mark.parametrize("S", [3, 16, 64])
def test_merge_large_contexts_at_segment_edges(B, S):
    """Context lengths up to 2^31 - 1 and entries at the segment edges e_s - 1,
    e_s, e_s + 1 (where floor(x S_eff / L) changes): bit-exact occupancy and
    witnesses against the oracle's integer arithmetic."""
    rng = np.random.default_rng(90 + S)
    rows, topk = 40, 96
    ctx = rng.integers(2 ** 30, 2 ** 31, rows).astype(np.int64)
    ctx[0] = 2 ** 31 - 1
    ctx[1] = S + 1
    learned = np.full((rows, topk), -1, dtype=np.int64)
    for r in range(rows):
        L = int(ctx[r])
        s_eff = min(S, L)
        edges = [(s * L + s_eff - 1) // s_eff for s in range(s_eff)]
        pick = rng.choice(s_eff, size=min(s_eff, 12), replace=False)
        vals = []
        for s in pick:
            for d in (-1, 0, 1):
                x = edges[s] + d
                if 0 <= x < L:
                    vals.append(x)
        vals += [L - 1, L, L + 5] if L < 2 ** 31 - 6 else [L - 1]
        vals = vals[:topk - 8]
        learned[r, :len(vals)] = vals
    learned = learned.astype(np.int32)
    ctx = ctx.astype(np.int32)
    ids = _dev(learned)
    B.witness_merge(ids, _dev(ctx), topk - S if topk > S else 0, S, S)
    ref = ow.apply_topology_witnesses(learned, topk, ctx, topk - S if topk > S else 0, S, S)
    assert np.array_equal(ids.cpu().numpy(), ref)
    tab = torch.empty((rows, S), dtype=torch.int32, device="cuda")
    B.witness_indices(_dev(learned), _dev(ctx), S, tab)
    assert np.array_equal(tab.cpu().numpy(), ow.topology_witness_indices(learned, topk, ctx, S))
    assert B.device_error() == 0


def test_decode_shaped_rows_with_padding(B):
    """64 rows x 2048 with 5% of slots set to -1, S = 16, serving form."""
    wp = wl.decode_bf16(M=64, H=2, D=8, L=32768, K=2048)
    rng = np.random.default_rng(9)
    learned = np.stack([rng.choice(32768, 2048, replace=False) for _ in range(64)]).astype(np.int32)
    learned[wp.extras["pad_mask"]] = -1
    ctx = np.full(64, 32768, dtype=np.int32)
    ids = _dev(learned)
    B.witness_merge(ids, _dev(ctx), 2048 - 16, 16, 16)
    ref = ow.apply_topology_witnesses(learned, 2048, ctx, 2048 - 16, 16, 16)
    assert np.array_equal(ids.cpu().numpy(), ref)


def test_refused_calls_leave_the_buffer(B):
    learned = np.array([[0, 5, 9, -1]], dtype=np.int32)
    ids = _dev(learned)
    for args, name in [((_dev(np.array([16])), 2, 65, 2), "SEGMENTS_OUT_OF_RANGE"),
                       ((_dev(np.array([16])), 5, 4, 2), "KEEP_OUT_OF_RANGE"),
                       ((_dev(np.zeros(0)), 2, 4, 2), "ROWS_MISMATCH")]:
        with pytest.raises(B.IdxError) as e:
            B.witness_merge(ids, *args)
        assert e.value.name == name
    assert ids.cpu().numpy().tolist() == learned.tolist()


@pytest.mark.parametrize("seed,M,L,K,ties", [
    (1, 16, 5000, 32, False), (2, 16, 5000, 2048, False), (3, 8, 40000, 2048, False), (4, 33, 3000, 100, True),
    (5, 7, 9000, 4096, True), (6, 12, 300, 1, True), (7, 5, 131072, 2048, False), (8, 40, 64, 64, True),
    (9, 6, 32768, 2048, False), (10, 6, 32769, 2048, True), (11, 4, 100000, 4096, True), (12, 9, 70000, 3, False),
    (13, 3, 32768, 2048, True)])
def test_topk_scores_bit_exact(B, seed, M, L, K, ties):
    s, lens = wl.score_rows(seed, M, L, ties=ties)
    lens[0] = 0
    lens[-1] = L
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, B.idx_topk_scores_workspace_size(M, L, K)), dtype=torch.uint8, device="cuda")
    B.idx_topk_scores(_dev(s, torch.float32), _dev(lens), L, K, ids, sc, ws=ws)
    g_ids, g_sc = ids.cpu().numpy(), sc.cpu().numpy()
    for m in range(M):
        o_ids, o_sc = odsa.topk(s[m, :lens[m]].astype(np.float64), K)
        assert g_ids[m].tolist() == o_ids.tolist(), m
        o32 = o_sc.astype(np.float32) + np.float32(0.0)    # the kernel reports -0.0 as +0.0
        assert np.array_equal(g_sc[m].view(np.uint32), o32.view(np.uint32)), m
    assert B.device_error() == 0


def test_topk_all_equal_and_two_valued_rows(B):
    """All scores equal (the sample threshold cannot separate anything: exact
    fallback) and two-valued rows: ties resolve to the lowest ids."""
    M, L, K = 4, 50000, 2048
    s = np.zeros((M, L), dtype=np.float32)
    s[1] = 1.0
    s[2, ::3] = 2.0
    s[3] = -0.0
    lens = np.full(M, L, dtype=np.int32)
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, B.idx_topk_scores_workspace_size(M, L, K)), dtype=torch.uint8, device="cuda")
    B.idx_topk_scores(_dev(s, torch.float32), _dev(lens), L, K, ids, sc, ws=ws)
    g = ids.cpu().numpy()
    for m in range(M):
        o_ids, _ = odsa.topk(s[m].astype(np.float64), K)
        assert g[m].tolist() == o_ids.tolist(), m
    assert B.device_error() == 0


def test_topk_heavy_ties_among_candidates(B):
    """The ~2500 best keys share three values (buckets of ~800 equal keys: the
    candidates go through the radix cut and the bitonic sort); the rest are
    distinct and lower.  Ties resolve to the lowest ids."""
    M, L, K = 3, 40000, 2048
    rng = np.random.default_rng(21)
    s = rng.random((M, L), dtype=np.float32)
    for m in range(M):
        top = rng.choice(L, 2500, replace=False)
        s[m, top] = rng.choice(np.array([10.0, 11.0, 12.0], dtype=np.float32), 2500)
    lens = np.full(M, L, dtype=np.int32)
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, B.idx_topk_scores_workspace_size(M, L, K)), dtype=torch.uint8, device="cuda")
    B.idx_topk_scores(_dev(s, torch.float32), _dev(lens), L, K, ids, sc, ws=ws)
    g_ids, g_sc = ids.cpu().numpy(), sc.cpu().numpy()
    for m in range(M):
        o_ids, o_sc = odsa.topk(s[m].astype(np.float64), K)
        assert g_ids[m].tolist() == o_ids.tolist(), m
        assert np.array_equal(g_sc[m], o_sc.astype(np.float32)), m
    assert B.device_error() == 0


def _many_rows(seed, M, L, K, ties):
    """Score rows for the many-long-rows top-K: random (or small-integer) rows of
    ragged lengths plus special rows (empty, shorter than K, all equal, -0.0 /
    +0.0, two-valued, heavy ties among the best ~1.2 K)."""
    s, lens = wl.score_rows(seed, M, L, ties=ties)
    rng = np.random.default_rng(seed + 100)
    lens[0], lens[1], lens[2], lens[3] = 0, 1, min(K - 1, L), min(K, L)
    lens[4] = min(K + 1, L)
    lens[5:12] = L
    s[5] = 0.0
    s[6] = -0.0
    s[6, ::7] = 0.0
    s[7] = 1.0
    s[7, ::3] = 2.0
    top = rng.choice(L, min(L, K + K // 5), replace=False)
    s[8] = rng.random(L, dtype=np.float32)
    s[8, top] = rng.choice(np.array([10.0, 11.0, 12.0], dtype=np.float32), top.size)
    s[9] = np.float32(3.0)
    s[9, rng.choice(L, 5, replace=False)] = np.float32(4.0)
    # a plateau of exact zeros under the top-K (rows whose heads all clip):
    # ~1.25 K positives (the K-th key above the plateau), ~0.75 K positives (the
    # K-th key on it: the smallest ids among the zeros complete the top-K)
    for row, npos in ((10, min(L // 3, K + K // 4)), (11, min(L // 3, (3 * K) // 4))):
        s[row] = -rng.random(L, dtype=np.float32) - np.float32(1.0)
        z = rng.choice(L, L // 3, replace=False)
        s[row, z] = np.float32(0.0)
        s[row, rng.choice(z, npos, replace=False)] = rng.random(npos, dtype=np.float32) + np.float32(0.5)
        lens[row] = L
    # a plateau of -inf (dropped entries) with finite scores above and below K
    s[12] = -np.inf
    s[12, rng.choice(L, min(L, K + 10), replace=False)] = rng.standard_normal(min(L, K + 10), dtype=np.float32)
    s[13] = -np.inf
    s[13, rng.choice(L, max(1, K // 2), replace=False)] = rng.standard_normal(max(1, K // 2), dtype=np.float32)
    lens[12] = lens[13] = L
    return s, lens


@pytest.mark.parametrize("seed,L,K,ties", [(41, 65536, 2048, False), (42, 65536, 2048, True), (43, 9000, 100, False),
                                           (44, 20001, 1, True), (45, 18432, 2048, False),
                                           (46, 16387, 2048, False)])
def test_topk_many_long_rows(B, seed, L, K, ties):
    """More rows than two per SM, longer than 4096: the one-block-per-row top-K
    (threshold, one stream, shared-memory sort), bit-exact against the oracle's
    lexicographic top-K on every row."""
    M = 2 * torch.cuda.get_device_properties(0).multi_processor_count + 16
    s, lens = _many_rows(seed, M, L, K, ties)
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, B.idx_topk_scores_workspace_size(M, L, K)), dtype=torch.uint8, device="cuda")
    B.idx_topk_scores(_dev(s, torch.float32), _dev(lens), L, K, ids, sc, ws=ws)
    g_ids, g_sc = ids.cpu().numpy(), sc.cpu().numpy()
    for m in range(M):
        o_ids, o_sc = odsa.topk(s[m, :lens[m]].astype(np.float64), K)
        assert g_ids[m].tolist() == o_ids.tolist(), m
        o32 = o_sc.astype(np.float32) + np.float32(0.0)    # the kernel reports -0.0 as +0.0
        assert np.array_equal(g_sc[m].view(np.uint32), o32.view(np.uint32)), m
    assert B.device_error() == 0
