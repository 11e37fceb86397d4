"""DoSA pruning on the GPU: dosa_topk must equal idx_topk bit for bit (ids and
score bits) on the same inputs, on every path (cold / strided / caller seeds,
bf16 / FP8 keys, shared / per-row keys, overflow and too-few-seed fallbacks,
exact ties at tau); and both agree with the fp64 oracle up to the score
tolerance."""
import numpy as np
import pytest
import torch

from helpers import EPS, check_topk_row
from oracle import dsa as odsa
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _unpruned(B, p, K):
    ids = torch.empty((p.q.shape[0], K), dtype=torch.int32, device="cuda")
    sc = torch.empty((p.q.shape[0], K), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.idx_topk_workspace_size(p, K), dtype=torch.uint8, device="cuda")
    B.idx_topk(p, K, ids, sc, ws)
    return ids.cpu().numpy(), sc.cpu().numpy()


def _pruned(B, p, K, seed_ids=None, **kw):
    dp = B.make_dosa_params(**kw)
    M = p.q.shape[0]
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    st = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    stats = torch.zeros(B.DOSA_STATS_FIELDS, dtype=torch.int64, device="cuda")
    sld = 0 if seed_ids is None else seed_ids.shape[1]
    ws = torch.empty(B.dosa_topk_workspace_size(p, K, dp, sld), dtype=torch.uint8, device="cuda")
    B.dosa_topk(p, K, dp, ids, sc, ws, seed_ids=seed_ids, row_status=st, stats=stats)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy(), st.cpu().numpy(), stats.cpu().numpy()


def _same(a_ids, a_sc, b_ids, b_sc):
    assert np.array_equal(a_ids, b_ids)
    assert np.array_equal(a_sc.view(np.uint32), b_sc.view(np.uint32))


def _check_oracle(wp, ids, sc, rows):
    for m in rows:
        s_ref, a_ref = odsa.row_scores(wp, m)
        check_topk_row(ids[m], sc[m], s_ref, a_ref, wp.K, EPS[wp.dtype])


@pytest.mark.parametrize("q_noise", [0.1, None])
def test_prefill_cold_seeds(B, q_noise):
    wp = wl.prefill_bf16(seed=11, n_queries=40, H=64, D=128, L=6000, K=256, n_seed=1024, R=16, q_noise=q_noise)
    p = B.problem_to_device(wp)
    u_ids, u_sc = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, stats = _pruned(B, p, wp.K, n_seed=1024, retained_heads=16, candidate_capacity=6000)
    _same(u_ids, u_sc, d_ids, d_sc)
    assert (st == 0).all(), st
    assert stats[0] == wp.pairs() and stats[1] == 1024 * wp.M
    assert stats[3] <= stats[2]
    _check_oracle(wp, d_ids, d_sc, [0, 17, 39])
    assert B.device_error() == 0


def test_near_parallel_heads_are_pruned(B):
    """Heads sharing one direction (tiny residuals): the anchor bound is tight,
    so most non-seed keys are dropped, and the output is still exact."""
    wp = wl.prefill_bf16(seed=12, n_queries=24, H=64, D=128, L=8000, K=256, n_seed=1024, R=16, q_noise=0.001)
    wp.w = np.abs(wp.w)      # every head adds: the threshold is a real score quantile
    p = B.problem_to_device(wp)
    u_ids, u_sc = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, stats = _pruned(B, p, wp.K, n_seed=1024, retained_heads=16, candidate_capacity=8000)
    _same(u_ids, u_sc, d_ids, d_sc)
    assert (st == 0).all()
    assert stats[2] < 0.5 * (stats[0] - stats[1]), stats
    assert stats[3] <= stats[2]


@pytest.mark.parametrize("H,R", [(32, 16), (64, 20), (16, 8)])
def test_decode_strided_seeds(B, H, R):
    wp = wl.decode_bf16(seed=H + R, M=6, H=H, D=128, L=3000, K=128)
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, stats = _pruned(B, p, wp.K, n_seed=512, retained_heads=R, candidate_capacity=3000)
    _same(*u, d_ids, d_sc)
    assert (st == 0).all()
    assert B.device_error() == 0


def test_ragged_fp8(B):
    wp = wl.ragged_fp8(seed=8, M=7, H=64, D=128, L_min=300, L_max=5000, K=128, R=20)
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, _ = _pruned(B, p, wp.K, n_seed=1024, retained_heads=20, candidate_capacity=5000)
    _same(*u, d_ids, d_sc)
    _check_oracle(wp, d_ids, d_sc, [0, 6])
    assert B.device_error() == 0


def test_caller_seeds_with_duplicates_and_junk(B):
    wp = wl.decode_bf16(seed=5, M=4, H=32, D=128, L=2000, K=64)
    p = B.problem_to_device(wp)
    rng = np.random.default_rng(5)
    seeds = rng.integers(-5, 2100, (4, 700)).astype(np.int32)      # duplicates, negatives, beyond L
    u = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, stats = _pruned(B, p, wp.K, seed_ids=torch.from_numpy(seeds).cuda(), retained_heads=16,
                                     candidate_capacity=2000)
    _same(*u, d_ids, d_sc)
    distinct = sum(len(set(x for x in row if 0 <= x < 2000)) for row in seeds)
    assert stats[1] == distinct


def test_overflow_and_too_few_seeds_fall_back(B):
    wp = wl.decode_bf16(seed=6, M=5, H=32, D=128, L=2500, K=100)
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, stats = _pruned(B, p, wp.K, n_seed=300, retained_heads=16, candidate_capacity=4)
    _same(*u, d_ids, d_sc)
    # overflow: found by the bound scan (2) or predicted by the planner, which then skips the scan (3)
    assert np.isin(st, (2, 3)).all() and stats[4] == 5
    assert (st == 3).any() and stats[5] == (st == 3).sum()
    d_ids, d_sc, st, stats = _pruned(B, p, wp.K, n_seed=50, retained_heads=16, candidate_capacity=4000)
    _same(*u, d_ids, d_sc)             # n_seed < K: every row on the unpruned path
    assert (st == 1).all()


def test_exact_ties_at_tau(B):
    """Keys duplicated many times so that scores tie exactly at the threshold."""
    wp = wl.decode_bf16(seed=9, M=3, H=32, D=128, L=1500, K=200)
    rng = np.random.default_rng(9)
    for m in range(3):
        base = m * 1500
        src = rng.integers(0, 1500, 60)
        for k in range(1500):
            wp.keys[base + k] = wp.keys[base + src[k % 60]]
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, _ = _pruned(B, p, wp.K, n_seed=400, retained_heads=16, candidate_capacity=1500)
    _same(*u, d_ids, d_sc)


def test_unsupported_shape_takes_the_exact_path(B):
    wp = wl.tiny_fp32()
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    d_ids, d_sc, st, _ = _pruned(B, p, wp.K, n_seed=64, retained_heads=2)
    _same(*u, d_ids, d_sc)
    assert (st == 1).all()


def _as_fp8_keys(wp):
    """The same problem with its keys quantised per token to e4m3 codes and a scale."""
    k = wp.keys_f32()
    amax = np.abs(k).max(axis=1)
    sc = np.where(amax > 0, amax / np.float32(wl.E4M3_MAX), np.float32(1.0)).astype(np.float32)
    codes = wl.f32_to_e4m3_bits(np.clip(k / sc[:, None], -wl.E4M3_MAX, wl.E4M3_MAX))
    return wl.IndexerProblem(wp.name + "_fp8", "fp8", wp.q, wp.w, codes, wp.key_len, None, wp.K, key_scale=sc,
                             extras=dict(wp.extras))


def _stream_counts_hold(on_stats, off_stats):
    """Every candidate is scored once on its row or once for its group: a group key was kept by two to four
    rows; both modes see the same candidates and survivors."""
    cands, group, solo = int(on_stats[2]), int(on_stats[6]), int(on_stats[7])
    assert group > 0 and solo > 0, on_stats
    assert solo + 2 * group <= cands <= solo + 4 * group, on_stats
    assert on_stats[2] == off_stats[2] and on_stats[3] == off_stats[3], (on_stats, off_stats)
    assert off_stats[6] == 0 and off_stats[7] == 0


@pytest.mark.parametrize("H,n_queries", [(64, 40), (32, 23), (16, 18)])
def test_shared_stream_groups_of_four(B, H, n_queries):
    """DoSA page section 4: groups of four queries share one exact pass over the keys that at least two of
    them kept.  Runs of three queries share a direction, so a group holds keys that several rows kept (shared)
    and keys that one row kept (its own list); a partial last group when n_queries % 4 != 0.  The output stays bit-identical to the unpruned top-K."""
    wp = wl.prefill_bf16(seed=13 + H, n_queries=n_queries, H=H, D=128, L=8000, K=256, n_seed=1024, R=min(16, H // 2),
                         q_noise=0.001, q_run=3, positive_w=True)
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    R = min(16, H // 2)
    on = _pruned(B, p, wp.K, n_seed=1024, retained_heads=R, candidate_capacity=8000, group_stream=1)
    off = _pruned(B, p, wp.K, n_seed=1024, retained_heads=R, candidate_capacity=8000, group_stream=0)
    _same(*u, on[0], on[1])
    _same(*u, off[0], off[1])
    assert (on[2] == 0).all() and (off[2] == 0).all()
    _stream_counts_hold(on[3], off[3])
    assert B.device_error() == 0


def test_shared_stream_fp8_keys(B):
    """The shared stream over e4m3 keys with a per-token scale (H 32: four queries' hi and lo rows fill
    N = 256)."""
    wp = _as_fp8_keys(wl.prefill_bf16(seed=31, n_queries=21, H=32, D=128, L=6000, K=192, n_seed=1024, R=16,
                                      q_noise=0.001, q_run=3, positive_w=True))
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    on = _pruned(B, p, wp.K, n_seed=1024, retained_heads=16, candidate_capacity=6000, group_stream=1)
    off = _pruned(B, p, wp.K, n_seed=1024, retained_heads=16, candidate_capacity=6000, group_stream=0)
    _same(*u, on[0], on[1])
    _same(*u, off[0], off[1])
    assert (on[2] == 0).all()
    _stream_counts_hold(on[3], off[3])
    _check_oracle(wp, on[0], on[1], [0, 20])
    assert B.device_error() == 0


def test_shared_stream_per_row_seeds_and_fallback_rows(B):
    """Caller seeds per row over shared keys: a key can be a seed of one row of a group and a candidate of the
    others, and the shared pass must not hand it back to the row that already has it.  Rows 5 and 6 get fewer
    than K seeds and take the unpruned path; their groups still share among the other rows."""
    wp = wl.prefill_bf16(seed=41, n_queries=16, H=64, D=128, L=7000, K=200, n_seed=1024, R=16, q_noise=0.001,
                         q_run=4, positive_w=True)
    rng = np.random.default_rng(41)
    seeds = np.full((wp.M, 1500), -1, dtype=np.int32)
    for m in range(wp.M):
        n = 100 if m in (5, 6) else 1500
        seeds[m, :n] = rng.choice(int(wp.key_len[m]), n, replace=False)
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    sd = torch.from_numpy(seeds).cuda()
    on = _pruned(B, p, wp.K, seed_ids=sd, retained_heads=16, candidate_capacity=7000, group_stream=1)
    off = _pruned(B, p, wp.K, seed_ids=sd, retained_heads=16, candidate_capacity=7000, group_stream=0)
    _same(*u, on[0], on[1])
    _same(*u, off[0], off[1])
    assert on[2][5] == 1 and on[2][6] == 1
    assert (np.delete(on[2], [5, 6]) == 0).all()
    _stream_counts_hold(on[3], off[3])
    assert B.device_error() == 0


def test_bound_with_more_than_16_retained_heads(B):
    """Shared bf16 keys with R = 20: the bound keeps 32 prepared rows per query (8 queries per tile);
    with R <= 16 it takes the group layout (16 rows per query, one block of aggregates).  Both
    layouts must leave the output equal to the unpruned top-K; 21 queries end on a partial group."""
    wp = wl.prefill_bf16(seed=51, n_queries=21, H=64, D=128, L=5000, K=200, n_seed=1024, R=20, q_noise=0.001,
                         q_run=3, positive_w=True)
    p = B.problem_to_device(wp)
    u = _unpruned(B, p, wp.K)
    for R in (20, 16, 9):
        d_ids, d_sc, st, stats = _pruned(B, p, wp.K, n_seed=1024, retained_heads=R, candidate_capacity=5000)
        _same(*u, d_ids, d_sc)
        assert (st == 0).all(), (R, st)
        assert stats[2] < stats[0] - stats[1], (R, stats)
    assert B.device_error() == 0
