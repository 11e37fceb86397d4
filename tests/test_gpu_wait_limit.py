"""The bounded-wait failure path of the tensor-core pipelines, made to run out
on purpose without faulting anything.

With the pipeline wait limit at 0 every wait that is not already complete
gives up at once: the score kernel's warps stop, the kernel waits for the key
copies and MMAs it has in flight (those drain waits keep their fixed limit),
frees its tensor memory and returns.  The host must see IDX_DEVERR_WAIT_TIMEOUT
in the device error word, the context must stay usable, and with the default
limit restored the next calls must give the same bits as before.
"""
import numpy as np
import pytest
import torch

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
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("make", [
    lambda: wl.decode_bf16(seed=31, M=8, L=4096, K=256),                 # per-row bf16 keys
    lambda: wl.prefill_bf16(seed=32, n_queries=64, L=4096, K=256),        # shared keys, 4 queries per tile
    lambda: wl.ragged_fp8(seed=33, M=4, L_min=2000, L_max=6000, K=256),   # FP8 keys, query-split warp
])
def test_wait_timeout_is_reported_and_recovered(B, make):
    wp = make()
    p = B.problem_to_device(wp)
    assert B.device_error() == 0
    ids0, sc0 = _topk(B, p, wp.K)
    assert B.device_error() == 0
    scores = torch.empty((wp.M, p.max_key_len), dtype=torch.float32, device="cuda")
    try:
        B.set_wait_limit_ns(0)
        B.idx_score(p, scores, p.max_key_len)      # the launch itself succeeds
        err = B.device_error()                     # synchronises: the kernel returned
    finally:
        B.set_wait_limit_ns(B.DEFAULT_WAIT_LIMIT_NS)
    assert err & B.DEVERR_WAIT_TIMEOUT, f"device error word {err}"
    # the context is usable and the default limit is back: same bits as before
    for _ in range(2):
        ids1, sc1 = _topk(B, p, wp.K)
        assert B.device_error() == 0
        assert np.array_equal(ids0, ids1)
        assert np.array_equal(sc0.view(np.uint32), sc1.view(np.uint32))
