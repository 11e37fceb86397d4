"""Parity at the full workload sizes, in the launch configuration the
benchmark times, against the oracle run on every host core: every row of the
decode batch (64) and of the ragged FP8 batch (128), every 16th query of the
causal prefill (256 of 4096) and every (query, KV head) selection of the
MiniMax workload (1024 x 8) -- scores within tolerance, top-K sets equal away
from the K-th score, block indices bit-exact -- plus every row of the integer
witness merge bit-exact, and the DoSA-pruned top-K bit-identical to the
unpruned one on every row, with the number of rows that stayed on the pruned
path asserted (the near-parallel-heads prefill: at least 99%)."""
import numpy as np
import pytest
import torch

from helpers import EPS, check_topk_row, oracle_pool, row_check_task, sub_problem
from oracle import dsa as odsa
from oracle import witness as ow
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _topk(B, p, K):
    M = p.q.shape[0]
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.idx_topk_workspace_size(p, K), dtype=torch.uint8, device="cuda")
    B.idx_topk(p, K, ids, sc, ws)
    return ids, sc


def _dosa(B, p, K, **kw):
    M = p.q.shape[0]
    dp = B.make_dosa_params(**kw)
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    st = torch.empty((M,), dtype=torch.int32, device="cuda")
    stats = torch.zeros(B.DOSA_STATS_FIELDS, dtype=torch.int64, device="cuda")
    ws = torch.empty(B.dosa_topk_workspace_size(p, K, dp), dtype=torch.uint8, device="cuda")
    B.dosa_topk(p, K, dp, ids, sc, ws, row_status=st, stats=stats)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy(), st.cpu().numpy(), stats.cpu().numpy()


def test_decode_bf16_full(B):
    """64 rows x 32768 own keys, H32, K2048; witnesses S=16 after 5% padding."""
    wp = wl.decode_bf16()
    p = B.problem_to_device(wp)
    ids, sc = _topk(B, p, wp.K)
    g_ids, g_sc = ids.cpu().numpy(), sc.cpu().numpy()
    _check_rows_pooled(wp, g_ids, g_sc, range(wp.M), EPS["bf16"])
    learned = g_ids.copy()
    learned[wp.extras["pad_mask"]] = -1
    t = torch.from_numpy(learned).cuda()
    S = wp.extras["S"]
    B.witness_merge(t, p.key_len, wp.K - S, S, S)
    ref = ow.apply_topology_witnesses(learned, wp.K, wp.key_len, wp.K - S, S, S)
    assert np.array_equal(t.cpu().numpy(), ref)
    assert B.device_error() == 0


def _check_rows_pooled(wp, g_ids, g_sc, rows, eps):
    """check_topk_row on `rows` by the oracle on every host core."""
    rows = list(rows)
    if wp.key_off is None:
        sub = sub_problem(wp, rows)
        tasks = [(None, i, g_ids[m], g_sc[m], eps) for i, m in enumerate(rows)]
    else:
        sub = None
        tasks = [(sub_problem(wp, [m]), 0, g_ids[m], g_sc[m], eps) for m in rows]
    pool = oracle_pool(sub)
    try:
        done = pool.map(row_check_task, tasks, chunksize=1)
    finally:
        pool.close()
        pool.join()
    assert len(done) == len(rows)


def _pruned_rows(st, stats, M):
    """Rows that stayed on the pruned path; consistent with the counters."""
    pruned = int((st == 0).sum())
    assert pruned == M - int(stats[4]), (pruned, stats)
    return pruned


@pytest.mark.parametrize("q_noise", [None, 0.05])
def test_prefill_full_pruned_equals_unpruned(B, q_noise):
    """4096 causal queries over 65536 keys, H64, K2048, 12288 seeds, R16; every
    16th query against the oracle."""
    wp = wl.prefill_bf16(q_noise=q_noise)
    p = B.problem_to_device(wp)
    ids, sc = _topk(B, p, wp.K)
    u_ids, u_sc = ids.cpu().numpy(), sc.cpu().numpy()
    d_ids, d_sc, st, stats = _dosa(B, p, wp.K, n_seed=12288, retained_heads=16)
    assert np.array_equal(u_ids, d_ids)
    assert np.array_equal(u_sc.view(np.uint32), d_sc.view(np.uint32))
    assert stats[0] == wp.pairs()
    pruned = _pruned_rows(st, stats, wp.M)
    print(f"prefill q_noise={q_noise}: {pruned} of {wp.M} rows pruned, {int(stats[5])} skipped the scan, "
          f"{int(stats[2])} candidates, {int(stats[3])} survivors")
    _check_rows_pooled(wp, u_ids, u_sc, range(0, wp.M, 16), EPS["bf16"])
    assert B.device_error() == 0


def test_prefill_aligned_full_pruned_equals_unpruned(B):
    """The near-parallel-heads prefill (the benchmark's DoSA workload): the bound
    prunes, so the identity covers the pruned path itself on nearly every row."""
    wp = wl.prefill_bf16(seed=3, q_noise=0.001, q_run=16, positive_w=True)
    p = B.problem_to_device(wp)
    ids, sc = _topk(B, p, wp.K)
    u_ids, u_sc = ids.cpu().numpy(), sc.cpu().numpy()
    d_ids, d_sc, st, stats = _dosa(B, p, wp.K, n_seed=12288, retained_heads=16)
    assert np.array_equal(u_ids, d_ids)
    assert np.array_equal(u_sc.view(np.uint32), d_sc.view(np.uint32))
    pruned = _pruned_rows(st, stats, wp.M)
    print(f"aligned prefill: {pruned} of {wp.M} rows pruned, {int(stats[2])} candidates, "
          f"{int(stats[3])} survivors, {int(stats[6])} group keys")
    assert pruned >= 0.99 * wp.M
    assert stats[2] > 0 and stats[3] > 0
    assert stats[2] < 0.5 * (stats[0] - stats[1])      # the bound dropped most non-seed pairs
    assert B.device_error() == 0


def test_ragged_fp8_full(B):
    """128 rows, L_r ~ U[4096, 131072], FP8 keys; DoSA R=20 == unpruned; witnesses S=32."""
    wp = wl.ragged_fp8()
    p = B.problem_to_device(wp)
    ids, sc = _topk(B, p, wp.K)
    u_ids, u_sc = ids.cpu().numpy(), sc.cpu().numpy()
    _check_rows_pooled(wp, u_ids, u_sc, range(wp.M), EPS["fp8"])
    d_ids, d_sc, st, stats = _dosa(B, p, wp.K, n_seed=8192, retained_heads=20)
    assert np.array_equal(u_ids, d_ids)
    assert np.array_equal(u_sc.view(np.uint32), d_sc.view(np.uint32))
    pruned = _pruned_rows(st, stats, wp.M)
    print(f"ragged FP8: {pruned} of {wp.M} rows pruned, {int(stats[5])} skipped the scan")
    S = wp.extras["S"]
    t = torch.from_numpy(u_ids.copy()).cuda()
    B.witness_merge(t, p.key_len, wp.K - S, S, S)
    ref = ow.apply_topology_witnesses(u_ids, wp.K, wp.key_len, wp.K - S, S, S)
    assert np.array_equal(t.cpu().numpy(), ref)
    assert B.device_error() == 0
