"""GPU parity of the indexer score and top-K against the fp64 oracle, through
the C ABI, on the workload shapes (scaled so the oracle finishes quickly, plus
sampled rows of the full sizes)."""
import numpy as np
import pytest
import torch

from helpers import EPS, check_scores, check_topk_row
from oracle import dsa as odsa
from oracle import witness as ow
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _run_score(B, wp):
    p = B.problem_to_device(wp)
    ld = max(1, p.max_key_len)
    scores = torch.full((wp.M, ld), float("nan"), dtype=torch.float32, device="cuda")
    B.idx_score(p, scores, ld)
    return scores.cpu().numpy()


def _run_topk(B, wp, K=None):
    p = B.problem_to_device(wp)
    K = wp.K if K is None else K
    ids = torch.empty((wp.M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((wp.M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.idx_topk_workspace_size(p, K), dtype=torch.uint8, device="cuda")
    B.idx_topk(p, K, ids, sc, ws)
    return ids.cpu().numpy(), sc.cpu().numpy()


def _problems():
    yield wl.tiny_fp32()
    yield wl.tiny_fp32(seed=10, M=5, H=3, D=7, L=1000, K=50)
    yield wl.decode_bf16(M=3, H=32, D=128, L=1000, K=64)
    yield wl.decode_bf16(M=2, H=16, D=128, L=333, K=2048)
    yield wl.decode_bf16(M=3, H=8, D=40, L=700, K=30)
    yield wl.prefill_bf16(n_queries=9, H=64, D=128, L=1500, K=100)
    yield wl.ragged_fp8(M=4, H=64, D=128, L_min=100, L_max=1500, K=128)


@pytest.mark.parametrize("wp", list(_problems()), ids=lambda w: f"{w.name}-M{w.M}-H{w.H}-D{w.D}")
def test_score_and_topk_match_oracle(B, wp):
    scores = _run_score(B, wp)
    ids, sc = _run_topk(B, wp)
    eps = EPS[wp.dtype]
    for m in range(wp.M):
        L = int(wp.key_len[m])
        s_ref, a_ref = odsa.row_scores(wp, m)
        check_scores(scores[m, :L], s_ref, a_ref, eps)
        check_topk_row(ids[m], sc[m], s_ref, a_ref, wp.K, eps)
    assert B.device_error() == 0


def test_tiny_fp32_workload_end_to_end(B):
    """8 rows, H4, D16, L512, K32 fp32; top-K then witnesses S=4, keep=28, B=4."""
    wp = wl.tiny_fp32()
    p = B.problem_to_device(wp)
    K, S = wp.K, wp.extras["S"]
    ids = torch.empty((wp.M, K), dtype=torch.int32, device="cuda")
    ws = torch.empty(B.idx_topk_workspace_size(p, K), dtype=torch.uint8, device="cuda")
    B.idx_topk(p, K, ids, None, ws)
    learned = ids.cpu().numpy().copy()
    B.witness_merge(ids, p.key_len, K - S, S, S)
    merged = ids.cpu().numpy()
    ref = ow.apply_topology_witnesses(learned, K, wp.key_len, K - S, S, S)
    assert np.array_equal(merged, ref)
    for m in range(wp.M):
        s_ref, a_ref = odsa.row_scores(wp, m)
        check_topk_row(learned[m], None, s_ref, a_ref, K, EPS["f32"])
