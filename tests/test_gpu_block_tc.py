"""GPU parity of the tensor-core block-selection route (block size 128, D = 128):
bit-exact block indices against the oracle and against the CUDA-core route
(block_select_static computes every block score in the page's order), on
shapes that span several 256-row tiles with ragged tails, unsorted positions,
exact ties between blocks, queries whose bounds decide nothing (every block
rescored), and the certified-bound statistics."""
import numpy as np
import pytest
import torch

from oracle import block_select as obs
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _run(B, q, k, pos, top, init, local, static=False, stats=None):
    Q, n_kv, D = q.shape
    L = k.shape[0]
    cfg = B.block_sparse_config(128, top, init, local)
    W = max(top, init + local, 1)
    out = torch.full((Q, n_kv, W), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((Q, n_kv), -7, dtype=torch.int32, device="cuda")
    qd = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    kd = torch.from_numpy(np.ascontiguousarray(k, dtype=np.float32)).cuda()
    pd = torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda()
    if static:
        B.block_select_static(qd, kd, pd, cfg, out, cnt)
    else:
        ws = torch.empty(max(1, B.block_select_workspace_size(Q, n_kv, max(L, 1), cfg)), dtype=torch.uint8,
                         device="cuda")
        B.block_select(qd, kd, pd, cfg, out, cnt, ws, stats=stats)
    torch.cuda.synchronize()
    return out.cpu().numpy(), cnt.cpu().numpy()


def _lists(o, c):
    Q, n_kv, _ = o.shape
    res = []
    for i in range(Q):
        row = []
        for h in range(n_kv):
            assert (o[i, h, c[i, h]:] == -1).all()
            row.append(o[i, h, :c[i, h]].tolist())
        res.append(row)
    return res


def _check_oracle(got, q, k, pos, top, init, local, queries):
    for i in queries:
        ref = obs.block_sparse_select(q[i], k, int(pos[i]), 128, top, init, local)
        assert got[i] == ref, i


@pytest.mark.parametrize("seed,Q,n_kv,L,top,init,local", [
    (11, 70, 5, 5000, 12, 2, 1),       # 350 rows: two tiles, the second ragged; L not a multiple of 128
    (12, 40, 8, 20000, 32, 1, 2),      # the MiniMax configuration, short context
    (13, 1, 1, 9000, 4, 0, 0),         # one row
    (14, 33, 3, 30000, 200, 0, 0),     # a large budget: many certain blocks, long candidate lists
    (15, 25, 7, 16384, 512, 1, 1),     # the largest budget of the route
])
def test_tc_route_against_oracle(B, seed, Q, n_kv, L, top, init, local):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((Q, n_kv, 128)).astype(np.float32)
    k = rng.standard_normal((L, 128)).astype(np.float32)
    pos = rng.integers(0, L + 300, Q).astype(np.int32)   # unsorted, some past the end
    pos[0] = min(5, L - 1)
    o, c = _run(B, q, k, pos, top, init, local)
    got = _lists(o, c)
    _check_oracle(got, q, k, pos, top, init, local, range(Q))
    o2, c2 = _run(B, q, k, pos, top, init, local, static=True)
    assert np.array_equal(o, o2) and np.array_equal(c, c2)
    assert B.device_error() == 0


def test_tc_route_exact_ties(B):
    """Duplicated key rows make whole blocks tie on their maxima; the order
    (score desc, block asc) must still come out bit for bit."""
    rng = np.random.default_rng(21)
    Q, n_kv, L = 48, 4, 24000
    q = rng.standard_normal((Q, n_kv, 128)).astype(np.float32)
    k = rng.standard_normal((L, 128)).astype(np.float32)
    src = k[:128].copy()
    for b in rng.choice(L // 128, 40, replace=False):   # 40 blocks identical to block 0
        k[b * 128:(b + 1) * 128] = src
    k[rng.integers(0, L, L // 10)] = k[7]                # scattered duplicate rows
    pos = rng.integers(200, L, Q).astype(np.int32)
    o, c = _run(B, q, k, pos, 32, 1, 2)
    got = _lists(o, c)
    _check_oracle(got, q, k, pos, 32, 1, 2, range(0, Q, 3))
    o2, c2 = _run(B, q, k, pos, 32, 1, 2, static=True)
    assert np.array_equal(o, o2) and np.array_equal(c, c2)


def test_tc_route_undecided_pairs(B):
    """Zero queries (every block scores 0: nothing is decided by the bounds) and
    a context made of one repeated block (all maxima equal) send pairs down the
    path that rescores every non-forced block."""
    rng = np.random.default_rng(22)
    Q, n_kv, L = 12, 4, 40000
    q = rng.standard_normal((Q, n_kv, 128)).astype(np.float32)
    q[::3] = 0.0
    k = rng.standard_normal((L, 128)).astype(np.float32)
    pos = np.linspace(1000, L - 1, Q).astype(np.int32)
    st = B.block_select_stats_tensor()
    o, c = _run(B, q, k, pos, 32, 1, 2, stats=st)
    got = _lists(o, c)
    _check_oracle(got, q, k, pos, 32, 1, 2, range(Q))
    s = B.block_select_stats_read(st)
    assert s["fallback_pairs"] >= 3 * n_kv      # zero queries past the first (8 blocks: nothing to score)
    kr = np.tile(rng.standard_normal((128, 128)).astype(np.float32), (L // 128 + 1, 1))[:L]
    o, c = _run(B, q, kr, pos, 32, 1, 2)
    got = _lists(o, c)
    _check_oracle(got, q, kr, pos, 32, 1, 2, range(0, Q, 2))


def test_tc_route_matches_core_route_many_queries(B):
    """1000 random queries (unsorted) x 8 heads over 50000 keys: the two routes agree."""
    rng = np.random.default_rng(23)
    Q, n_kv, L = 1000, 8, 50000
    q = rng.standard_normal((Q, n_kv, 128)).astype(np.float32)
    k = rng.standard_normal((L, 128)).astype(np.float32)
    pos = rng.integers(0, L, Q).astype(np.int32)
    o, c = _run(B, q, k, pos, 32, 1, 2)
    o2, c2 = _run(B, q, k, pos, 32, 1, 2, static=True)
    assert np.array_equal(c, c2)
    assert np.array_equal(o, o2)


def test_tc_route_workload_stats(B):
    """The MiniMax workload: bounded blocks, few rescored, none undecided, and
    the measured error well inside the certified bound."""
    bp = wl.block_select()
    st = B.block_select_stats_tensor()
    o, c = _run(B, bp.index_q, bp.index_k, bp.query_pos, bp.top_blocks, bp.init_blocks, bp.local_blocks, stats=st)
    s = B.block_select_stats_read(st)
    assert s["pairs"] > 0 and s["fallback_pairs"] == 0
    assert s["blocks_rescored"] < 0.05 * s["blocks_bounded"]
    assert 0.0 < s["max_bound_use"] < 0.5
    got = _lists(o, c)
    _check_oracle(got, bp.index_q, bp.index_k, bp.query_pos, bp.top_blocks, bp.init_blocks, bp.local_blocks,
                  [3, 300, 777, 1023])
    o2, c2 = _run(B, bp.index_q, bp.index_k, bp.query_pos, bp.top_blocks, bp.init_blocks, bp.local_blocks,
                  static=True)
    assert np.array_equal(o, o2) and np.array_equal(c, c2)


def test_page_order_one_ulp_tie_both_routes(B):
    """Query 815, head 4 of the MiniMax workload: blocks 548 and 156 score
    41.377743 and 41.37774 in the page's sequential fp32 sum (one ulp apart),
    and a fused multiply-add chain swaps them.  Both routes must keep the
    page's order (products and sums rounded one by one)."""
    bp = wl.block_select()
    sc = obs.block_scores(bp.index_q[815, 4], bp.index_k, int(bp.query_pos[815]), 128)
    assert np.float32(sc[548]).view(np.int32) - np.float32(sc[156]).view(np.int32) == 1
    q = bp.index_q[815:816]
    pos = bp.query_pos[815:816]
    ref = obs.block_sparse_select(q[0], bp.index_k, int(pos[0]), 128, 32, 1, 2)
    assert 548 in ref[4] and 156 not in ref[4]
    for static in (False, True):
        o, c = _run(B, q, bp.index_k, pos, 32, 1, 2, static=static)
        assert _lists(o, c)[0] == ref, "static" if static else "tensor"


def _positions(B, blocks, counts, pos, L, bs):
    Q, n_kv, W = blocks.shape
    out = torch.full((Q, n_kv, max(1, W * bs)), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((Q, n_kv), -7, dtype=torch.int32, device="cuda")
    B.block_positions(torch.from_numpy(np.ascontiguousarray(blocks, dtype=np.int32)).cuda(),
                      None if counts is None else torch.from_numpy(np.asarray(counts, dtype=np.int32)).cuda(),
                      torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda(), L, bs, out, cnt)
    torch.cuda.synchronize()
    return out.cpu().numpy(), cnt.cpu().numpy()


def test_block_positions_against_oracle(B):
    """positions_of_blocks on arbitrary block lists: unsorted, repeated, -1 entries, blocks past
    the keys, positions past L, counts given or not."""
    rng = np.random.default_rng(31)
    Q, n_kv, W, L, bs = 40, 3, 12, 3000, 128
    blocks = rng.integers(-1, (L + bs - 1) // bs + 3, (Q, n_kv, W)).astype(np.int32)
    blocks[0, 0, :] = 5                                   # one block repeated
    counts = rng.integers(0, W + 1, (Q, n_kv)).astype(np.int32)
    pos = rng.integers(0, L + 100, Q).astype(np.int32)
    pos[1] = 0
    for use_counts in (True, False):
        o, c = _positions(B, blocks, counts if use_counts else None, pos, L, bs)
        for i in range(Q):
            for h in range(n_kv):
                n = counts[i, h] if use_counts else W
                ref = obs.positions_of_blocks([int(b) for b in blocks[i, h, :n] if b >= 0], int(pos[i]), L, bs)
                assert c[i, h] == len(ref)
                assert o[i, h, :c[i, h]].tolist() == ref
                assert (o[i, h, c[i, h]:] == -1).all()
    o, c = _positions(B, blocks, counts, pos, L, 0)        # block size 0: nothing covered
    assert (c == 0).all()


def test_block_positions_of_workload_selection(B):
    """The MiniMax selection of sampled queries, expanded to positions."""
    bp = wl.block_select()
    o, c = _run(B, bp.index_q, bp.index_k, bp.query_pos, bp.top_blocks, bp.init_blocks, bp.local_blocks)
    po, pc = _positions(B, o, c, bp.query_pos, bp.index_k.shape[0], 128)
    for i in (0, 1, 500, 1023):
        for h in range(8):
            ref = obs.positions_of_blocks(o[i, h, :c[i, h]].tolist(), int(bp.query_pos[i]), bp.index_k.shape[0], 128)
            assert po[i, h, :pc[i, h]].tolist() == ref
    # a full selection covers top_blocks * 128 positions except in the last, partial block
    assert (pc[100:] >= 31 * 128).all()


def test_block_select_events_same_result(B):
    """block_select_events records its six events and returns what block_select returns."""
    rng = np.random.default_rng(41)
    Q, n_kv, L = 30, 8, 9000
    q = torch.from_numpy(rng.standard_normal((Q, n_kv, 128)).astype(np.float32)).cuda()
    k = torch.from_numpy(rng.standard_normal((L, 128)).astype(np.float32)).cuda()
    pos = torch.from_numpy(rng.integers(0, L, Q).astype(np.int32)).cuda()
    cfg = B.block_sparse_config(128, 32, 1, 2)
    ws = torch.empty(B.block_select_workspace_size(Q, n_kv, L, cfg), dtype=torch.uint8, device="cuda")
    out1 = torch.empty((Q, n_kv, 32), dtype=torch.int32, device="cuda")
    out2 = torch.empty_like(out1)
    c1 = torch.empty((Q, n_kv), dtype=torch.int32, device="cuda")
    c2 = torch.empty_like(c1)
    B.block_select(q, k, pos, cfg, out1, c1, ws)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record()
    B.block_select_events(q, k, pos, cfg, out2, c2, ws, ev, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(c1, c2)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0.0 for t in times)


def test_tc_route_adversarial_bounds(B):
    """Inputs aimed at the certified bound of the tensor-core block maxima
    ("ferrox_core/block_sparse.rs", dot and select_for_head: the selection
    rests on the exact sequential f32 block maxima): query and key elements
    spread over many binades (fp16 under a per-row / per-block power-of-two
    scale loses the small ones), keys k = 1000 u + v with u orthogonal to one
    query head (large products cancelling to a small dot), and copies of the
    block at the selection cut (exact ties and one-ulp nudges).  Every
    selection must equal the oracle's and the CUDA-core route's, and the
    measured error of every rescored block must stay inside its bound."""
    rng = np.random.default_rng(31)
    Q, n_kv, L, D = 16, 4, 20000, 128
    q = rng.standard_normal((Q, n_kv, D)).astype(np.float32)
    q[::2] *= (2.0 ** rng.integers(-12, 13, (Q // 2, n_kv, D))).astype(np.float32)
    k = rng.standard_normal((L, D)).astype(np.float32)
    k[:L // 4] *= (2.0 ** rng.integers(-20, 21, (L // 4, D))).astype(np.float32)
    pos = np.linspace(8000, L - 1, Q).astype(np.int32)
    # cancellation: blocks 70..89 orthogonal to query 1 head 0, 100..119 to query 3 head 1
    for (qi, h, b0) in ((1, 0, 70), (3, 1, 100), (5, 2, 40)):
        qv = q[qi, h].astype(np.float64)
        for b in range(b0, b0 + 20):
            r = rng.standard_normal((128, D))
            u = r - np.outer(r @ qv / (qv @ qv), qv)
            k[b * 128:(b + 1) * 128] = (1000.0 * u + rng.standard_normal((128, D))).astype(np.float32)
    # copies of the block at the cut of query 0, head 0 (32 places, 3 forced)
    sc = obs.block_scores(q[0, 0], k, int(pos[0]), 128)
    n_blocks = sc.shape[0]
    free = [b for b in range(1, n_blocks - 2)]
    order = sorted(free, key=lambda b: (-float(sc[b]), b))
    cut = order[28]
    src = k[cut * 128:(cut + 1) * 128].copy()
    for b in rng.choice([x for x in free if x != cut], 4, replace=False):
        k[b * 128:(b + 1) * 128] = src                           # exact ties with the cut block
    nudged = src.copy()
    nudged.view(np.uint32)[:, 0] ^= 1                              # one-ulp changes of one element
    b = [x for x in free if x != cut][5]
    k[b * 128:(b + 1) * 128] = nudged
    st = B.block_select_stats_tensor()
    o, c = _run(B, q, k, pos, 32, 1, 2, stats=st)
    got = _lists(o, c)
    _check_oracle(got, q, k, pos, 32, 1, 2, range(Q))
    o2, c2 = _run(B, q, k, pos, 32, 1, 2, static=True)
    assert np.array_equal(o, o2) and np.array_equal(c, c2)
    s = B.block_select_stats_read(st)
    print("adversarial bound stats", s)
    assert s["blocks_rescored"] > 0
    assert 0.0 <= s["max_bound_use"] < 1.0
    assert B.device_error() == 0
