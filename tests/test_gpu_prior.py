"""GPU parity of the top-K with a prior selection (idx_topk_prior): ids and
scores bit-identical to the unpruned idx_topk on every row, the rows checked
against the fp64 oracle where it is cheap, and every fallback route
(no usable prior, candidate overflow) exercised."""
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
    M = p.q.shape[0]
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.idx_topk_workspace_size(p, K), dtype=torch.uint8, device="cuda")
    B.idx_topk(p, K, ids, sc, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy()


def _prior(B, p, K, prior, cap):
    M = p.q.shape[0]
    ids = torch.full((M, K), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    st = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    stats = torch.zeros(3, dtype=torch.int64, device="cuda")
    pr = torch.from_numpy(np.ascontiguousarray(prior, dtype=np.int32)).cuda()
    ws = torch.empty(B.idx_topk_prior_workspace_size(p, K, pr.shape[1], cap), dtype=torch.uint8, device="cuda")
    ws.random_(0, 255)                            # stale workspace contents must not matter
    B.idx_topk_prior(p, K, pr, cap, ids, sc, ws, row_status=st, stats=stats)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy(), st.cpu().numpy(), stats.cpu().numpy()


def _oracle_prior(prev, K):
    """The previous step's top-K by the oracle (the prior input)."""
    out = np.full((prev.M, K), -1, dtype=np.int32)
    for m in range(prev.M):
        t = np.asarray(odsa.row_topk(prev, m, K)[0])
        t = t[t >= 0][:K]
        out[m, :len(t)] = t
    return out


def _same(a, b):
    assert np.array_equal(a[0], b[0]), "ids"
    assert np.array_equal(a[1].view(np.int32), b[1].view(np.int32)), "scores"


@pytest.mark.parametrize("maker,K", [
    (lambda: wl.decode_bf16(seed=7, M=16, H=32, L=4096, K=256), 256),
    (lambda: wl.ragged_fp8(seed=9, M=12, H=64, L_min=1500, L_max=9000, K=512), 512),
])
def test_prior_matches_unpruned(B, maker, K):
    wp = maker()
    prev = wl.previous_step(wp, seed=8, noise=0.3)
    prior = _oracle_prior(prev, K)
    p = B.problem_to_device(wp)
    ref = _unpruned(B, p, K)
    ids, sc, st, stats = _prior(B, p, K, prior, cap=8 * K)
    _same((ids, sc), ref)
    assert (st == 0).all() and stats[0] == wp.M and stats[2] == 0
    assert stats[1] < 0.5 * wp.pairs()          # the prior cut the candidates
    for m in range(0, wp.M, 5):
        s_ref, a_ref = odsa.row_scores(wp, m)
        check_topk_row(ids[m], sc[m], s_ref, a_ref, K, EPS[wp.dtype])
    assert B.device_error() == 0


def test_prior_fallback_routes(B):
    """Bad priors (padding, out-of-range ids, repeats, too few), rows shorter
    than K, a prior wider than K, and a capacity too small for a poor prior."""
    K = 128
    wp = wl.decode_bf16(seed=12, M=10, H=32, L=2048, K=K)
    wp.key_len[3] = 100                           # shorter than K
    wp.key_len[4] = 0
    p = B.problem_to_device(wp)
    ref = _unpruned(B, p, K)
    prev = wl.previous_step(wp, seed=13, noise=0.3)
    good = _oracle_prior(prev, K)
    wide = np.concatenate([good, np.random.default_rng(1).integers(0, 2048, (10, K))], axis=1).astype(np.int32)
    bad = good.copy()
    bad[0, :] = -1                                # no prior
    bad[1, :] = 5000                              # all out of range
    bad[2, :] = bad[2, 0]                         # one id repeated
    bad[5, 1:] = -1                               # a single id
    ids, sc, st, stats = _prior(B, p, K, bad, cap=4 * K)
    _same((ids, sc), ref)
    assert st[0] == 1 and st[1] == 1 and st[2] == 1 and st[5] == 1 and st[6] == 0
    # 100 keys < K: the answer is every key, and the prior (the previous step's 99) misses the newest
    assert st[3] == 1
    ids, sc, st, stats = _prior(B, p, K, wide, cap=4 * K)
    _same((ids, sc), ref)
    poor = np.random.default_rng(2).choice(2048, (10, K)).astype(np.int32)   # random, may repeat
    ids, sc, st, stats = _prior(B, p, K, poor, cap=K)
    _same((ids, sc), ref)
    assert (st != 0).sum() >= 5                   # overflow or repeats: the unpruned path


def test_prior_shared_keys(B):
    """Causal rows over one key sequence (prefill layout): same result."""
    K = 256
    wp = wl.prefill_bf16(seed=14, n_queries=48, H=64, L=6000, K=K)
    p = B.problem_to_device(wp)
    ref = _unpruned(B, p, K)
    prev = wl.previous_step(wp, seed=15, noise=0.2)
    prior = _oracle_prior(prev, K)
    ids, sc, st, stats = _prior(B, p, K, prior, cap=8 * K)
    _same((ids, sc), ref)
    assert (st == 0).sum() >= 40


def test_prior_full_size_ragged_fp8(B):
    """128 rows, L ~ U[4096, 131072] FP8 keys, H64, K2048, the top-K of the two previous
    steps as the prior: bit-identical to idx_topk on every row, run after run, with
    stale workspaces (the prior is an input, computed by the unpruned top-K of the
    previous steps' queries)."""
    wp = wl.ragged_fp8()
    K = wp.K
    p = B.problem_to_device(wp)
    ref = _unpruned(B, p, K)
    priors = []
    for seed in (8, 9):
        prev = wl.previous_step(wp, seed=seed, noise=0.3)
        q = torch.from_numpy(np.ascontiguousarray(prev.q).view(np.int16)).cuda().view(torch.bfloat16)
        pq = B.Problem(q, p.w, p.keys, torch.from_numpy(prev.key_len).cuda(), p.max_key_len, p.key_off, p.key_scale)
        ids = torch.empty((wp.M, K), dtype=torch.int32, device="cuda")
        B.idx_topk(pq, K, ids, None, torch.empty(B.idx_topk_workspace_size(pq, K), dtype=torch.uint8, device="cuda"))
        priors.append(ids)
    prior = torch.cat(priors, dim=1).cpu().numpy()
    for rep in range(3):
        ids, sc, st, stats = _prior(B, p, K, prior, cap=4 * K)
        _same((ids, sc), ref)
    assert (st == 0).sum() >= 120 and stats[1] < 0.05 * wp.pairs()
    assert B.device_error() == 0


def test_prior_events_same_result(B):
    """idx_topk_prior_events records its six events and returns what idx_topk_prior returns."""
    K = 128
    wp = wl.decode_bf16(seed=21, M=8, H=32, L=3000, K=K)
    prev = wl.previous_step(wp, seed=22, noise=0.3)
    prior = torch.from_numpy(_oracle_prior(prev, K)).cuda()
    p = B.problem_to_device(wp)
    ws = torch.empty(B.idx_topk_prior_workspace_size(p, K, K, 4 * K), dtype=torch.uint8, device="cuda")
    i1 = torch.empty((8, K), dtype=torch.int32, device="cuda")
    s1 = torch.empty((8, K), dtype=torch.float32, device="cuda")
    i2, s2 = torch.empty_like(i1), torch.empty_like(s1)
    B.idx_topk_prior(p, K, prior, 4 * K, i1, s1, ws)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record()
    B.idx_topk_prior_events(p, K, prior, 4 * K, i2, s2, ws, ev, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(s1.view(torch.int32), s2.view(torch.int32))
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0.0 for i in range(5))
