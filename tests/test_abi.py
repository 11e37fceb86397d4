"""The C ABI: the library builds, loads and exports every function that
include/idx.h declares; host-side refusals happen before any launch (these
calls pass no device memory, so they run without a GPU)."""
import ctypes
import os

import pytest

from helpers import header_functions

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_attention_indexer_idx_gb300 import build
    build.build()
    from sparse_attention_indexer_idx_gb300 import binding
    return binding.lib()


def test_exports_every_declared_function(L):
    names = header_functions(os.path.join(ROOT, "include", "idx.h"))
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    from sparse_attention_indexer_idx_gb300 import binding
    assert set(binding.EXPORTS) == set(names)


def test_witness_refusals_before_launch(L):
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    assert L.witness_merge(nul, 1, 4, nul, 1, 2, 0, 2, nul) == 0            # S = 0: off switch
    assert L.witness_merge(nul, 1, 4, nul, 1, 2, 65, 2, nul) == 2           # S > 64
    assert L.witness_merge(nul, 1, 4, nul, 1, 5, 4, 2, nul) == 3            # keep > topk
    assert L.witness_merge(nul, 2, 4, nul, 1, 2, 4, 2, nul) == 1            # rows mismatch
    assert L.witness_merge(nul, 1, 4, nul, 1, 4, 4, 2, nul) == 0            # B = 0: no-op
    assert L.witness_merge(nul, 0, 4, nul, 0, 2, 4, 2, nul) == 0            # zero rows
    assert L.witness_indices(nul, 1, 4, nul, 1, 0, nul, nul) == 2           # no off switch here
    assert b"num_segments" in L.idx_last_error_string()


def test_problem_refusals_before_launch(L):
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    p = B.idx_problem(None, B.IDX_F32, None, 1, 4, 16, None, B.IDX_F32, None, 10, None, None, 10)
    assert L.idx_score(ctypes.byref(p), nul, 10, nul) == 4                  # NULL q/w/key_len
    p2 = B.idx_problem(1, B.IDX_BF16, 1, 1, 4, 16, 1, B.IDX_FP8_E4M3, None, 10, None, 1, 10)
    assert L.idx_score(ctypes.byref(p2), ctypes.c_void_p(1), 10, nul) == 4  # FP8 without scale
    p3 = B.idx_problem(1, B.IDX_F32, 1, 1, 4, 16, 1, B.IDX_BF16, None, 10, None, 1, 10)
    assert L.idx_score(ctypes.byref(p3), ctypes.c_void_p(1), 10, nul) == 5  # mixed dtypes
    p4 = B.idx_problem(1, B.IDX_F32, 1, 1, 4, 16, 1, B.IDX_F32, None, 10, None, 1, 11)
    assert L.idx_score(ctypes.byref(p4), ctypes.c_void_p(1), 11, nul) == 4  # shared keys, len > n_keys
    p5 = B.idx_problem(1, B.IDX_F32, 1, 1, 4, 16, 1, B.IDX_F32, None, 10, None, 1, 10)
    assert L.idx_topk(ctypes.byref(p5), 0, ctypes.c_void_p(1), nul, ctypes.c_void_p(1), 1 << 20, nul) == 4  # K = 0
    assert L.idx_topk(ctypes.byref(p5), 4097, ctypes.c_void_p(1), nul, ctypes.c_void_p(1), 1 << 20, nul) == 4
    assert L.idx_topk(ctypes.byref(p5), 8, ctypes.c_void_p(1), nul, ctypes.c_void_p(1), 1, nul) == 6  # workspace
    assert L.idx_topk_workspace_size(ctypes.byref(p5), 8) >= 40


def test_block_select_refusals_before_launch(L):
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    cfg = B.block_sparse_config(128, 32, 1, 2)
    one = ctypes.c_void_p(256)
    assert L.block_select(one, one, one, 4, 2, 128, 1024, ctypes.byref(cfg), one, 31, nul, nul, one, 1 << 20, nul) == 4
    bad = B.block_sparse_config(128, -1, 1, 2)
    assert L.block_select(one, one, one, 4, 2, 128, 1024, ctypes.byref(bad), one, 32, nul, nul, one, 1 << 20, nul) == 4
    assert L.block_select(one, one, one, 4, 2, 128, 1024, ctypes.byref(cfg), one, 32, nul, nul, one, 0, nul) == 6
    assert L.block_select_workspace_size(4, 2, 1024, ctypes.byref(cfg)) >= 4 * 2 * 8 * 4


def test_block_select_events_refusals(L):
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    cfg = B.block_sparse_config(128, 32, 1, 2)
    one = ctypes.c_void_p(256)
    ev = (ctypes.c_void_p * 6)()
    # fewer than 6 events, or none, is refused before anything runs
    assert L.block_select_events(one, one, one, 4, 2, 128, 1024, ctypes.byref(cfg), one, 32, nul, nul, one, 1 << 20,
                                 ev, 5, nul) == 4
    assert L.block_select_events(one, one, one, 4, 2, 128, 1024, ctypes.byref(cfg), one, 32, nul, nul, one, 1 << 20,
                                 nul, 6, nul) == 4
    # the same argument checks as block_select
    assert L.block_select_events(one, one, one, 4, 2, 128, 1024, ctypes.byref(cfg), one, 31, nul, nul, one, 1 << 20,
                                 ev, 6, nul) == 4


def test_block_positions_refusals(L):
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    # out_width below W * block_size, W above IDX_MAX_K, n_kv of 0
    assert L.block_positions(one, nul, 4, 2, 32, one, 1024, 128, one, 4095, nul, nul) == 4
    assert L.block_positions(one, nul, 4, 2, 4097, one, 1024, 1, one, 1 << 20, nul, nul) == 4
    assert L.block_positions(one, nul, 4, 0, 32, one, 1024, 128, one, 4096, nul, nul) == 4
    # no rows: nothing to do
    assert L.block_positions(one, nul, 0, 2, 32, one, 1024, 128, one, 4096, nul, nul) == 0


def test_topk_prior_refusals(L):
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    p = B.idx_problem(one, B.IDX_BF16, one, 4, 32, 128, one, B.IDX_BF16, None, 1 << 20, None, one, 4096)
    # K out of range, prior_ld < 1, capacity below K, NULL prior
    assert L.idx_topk_prior(ctypes.byref(p), 0, one, 16, 64, one, nul, nul, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_prior(ctypes.byref(p), 16, one, 0, 64, one, nul, nul, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_prior(ctypes.byref(p), 16, one, 16, 8, one, nul, nul, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_prior(ctypes.byref(p), 16, nul, 16, 64, one, nul, nul, nul, one, 1 << 30, nul) == 4
    # workspace too small
    assert L.idx_topk_prior(ctypes.byref(p), 16, one, 16, 64, one, nul, nul, nul, one, 16, nul) == 6
    assert L.idx_topk_prior_workspace_size(ctypes.byref(p), 16, 16, 64) > 4 * 4096 * 4
