"""block_select_static: the entry point for callers that cannot allocate
device memory (a host framework that owns every allocation, or a path where a
cudaMalloc could stall or fail).  It must give exactly the block indices of
block_select, which takes a caller workspace, on consecutive calls that share
its fixed scratch array; sizes beyond that array are refused up front.

This file is named so that pytest collects it last."""
import ctypes

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


def _run_both(B, bp):
    dev = "cuda"
    q = torch.from_numpy(bp.index_q).to(dev)
    k = torch.from_numpy(bp.index_k).to(dev)
    pos = torch.from_numpy(bp.query_pos).to(dev)
    cfg = B.block_sparse_config(bp.block_size, bp.top_blocks, bp.init_blocks, bp.local_blocks)
    Q, n_kv, _ = bp.index_q.shape
    W = max(bp.top_blocks, bp.init_blocks + bp.local_blocks)
    ref = torch.empty((Q, n_kv, W), dtype=torch.int32, device=dev)
    ref_cnt = torch.empty((Q, n_kv), dtype=torch.int32, device=dev)
    ws = torch.empty(B.block_select_workspace_size(Q, n_kv, bp.index_k.shape[0], cfg), dtype=torch.uint8, device=dev)
    B.block_select(q, k, pos, cfg, ref, ref_cnt, ws)
    got = torch.full((Q, n_kv, W), -7, dtype=torch.int32, device=dev)
    got_cnt = torch.full((Q, n_kv), -7, dtype=torch.int32, device=dev)
    B.block_select_static(q, k, pos, cfg, got, got_cnt)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), ref_cnt.cpu().numpy(), got.cpu().numpy(), got_cnt.cpu().numpy()


def test_static_scratch_matches_the_workspace_entry_point_twice(B):
    # two different problems in a row: the second must not see the first's scratch
    for seed, L, Q in [(41, 32768, 256), (42, 20000, 160)]:
        bp = wl.block_select(seed=seed, Q=Q, n_kv=8, D=128, L=L, block_size=128, top_blocks=32, init_blocks=1,
                             local_blocks=2)
        ref, ref_cnt, got, got_cnt = _run_both(B, bp)
        assert np.array_equal(ref, got)
        assert np.array_equal(ref_cnt, got_cnt)
    assert B.device_error() == 0


def test_sizes_beyond_the_fixed_scratch_are_refused(B):
    cfg = B.block_sparse_config(1, 4, 1, 1)
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    # 2 queries x 8 heads x 2^20 one-token blocks > 2^23 words
    st = B.lib().block_select_static(one, one, one, 2, 8, 128, 1 << 20, ctypes.byref(cfg), one, 4, nul, nul)
    assert st == 6
    assert b"exceed" in B.lib().idx_last_error_string()
