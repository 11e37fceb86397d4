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


def test_dosa_refusals_and_layout(L):
    """dosa_topk refuses bad arguments before any launch; the workspace layout
    is host arithmetic: every region lies inside the workspace size."""
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    big = 1 << 40
    # 64 queries over 65536 shared bf16 keys (key_off NULL), H64 D128
    p = B.idx_problem(one, B.IDX_BF16, one, 64, 64, 128, one, B.IDX_BF16, None, 65536, None, one, 65536)
    dp = B.make_dosa_params(n_seed=4096, retained_heads=16)

    def call(K=256, params=dp, seeds=nul, seed_ld=0, out=one, ws_bytes=big, prob=p):
        pp = ctypes.byref(params) if params is not None else None
        return L.dosa_topk(ctypes.byref(prob), K, pp, seeds, seed_ld, out, nul, nul, nul, one, ws_bytes, nul)

    assert call(params=None) == 4                                   # NULL params
    assert call(K=0) == 4 and call(K=4097) == 4                     # K outside [1, 4096]
    for field, bad in (("n_seed", -1), ("retained_heads", 0), ("n_sample", 0), ("candidate_capacity", -1),
                       ("act_freq_min", 1.5), ("act_freq_min", float("nan")), ("margin_gamma", -1.0)):
        q = B.make_dosa_params(n_seed=4096, retained_heads=16)
        setattr(q, field, bad)
        assert call(params=q) == 4, field
    assert call(seeds=one, seed_ld=0) == 4                          # caller seeds without a row stride
    assert call(out=nul) == 4                                       # NULL output ids
    need = L.dosa_topk_workspace_size(ctypes.byref(p), 256, ctypes.byref(dp), 0)
    assert need > 64 * 65536 // 8                                   # at least the candidate bitmaps
    assert call(ws_bytes=need - 1) == 6                             # workspace too small
    p0 = B.idx_problem(one, B.IDX_BF16, one, 0, 64, 128, one, B.IDX_BF16, None, 65536, None, one, 65536)
    assert call(prob=p0, ws_bytes=0) == 0                           # no rows: nothing to do
    # the size grows with the rows
    p2 = B.idx_problem(one, B.IDX_BF16, one, 128, 64, 128, one, B.IDX_BF16, None, 65536, None, one, 65536)
    assert L.dosa_topk_workspace_size(ctypes.byref(p2), 256, ctypes.byref(dp), 0) > need

    lay = B.dosa_ws_layout()
    assert L.dosa_workspace_layout(ctypes.byref(p), 256, ctypes.byref(dp), 0, None) == 4
    assert L.dosa_workspace_layout(ctypes.byref(p), 0, ctypes.byref(dp), 0, ctypes.byref(lay)) == 4
    assert L.dosa_workspace_layout(ctypes.byref(p), 256, ctypes.byref(dp), 0, ctypes.byref(lay)) == 0
    offs = [getattr(lay, n) for n in ("seed_list", "seed_count", "rep_count", "rep_scores", "tau", "status",
                                      "plan_head", "plan_beta", "plan_dnorm", "wfold", "coef", "qprep")]
    assert all(0 <= o < need for o in offs)
    assert len(set(offs)) == len(offs)                              # distinct regions
    assert lay.seed_rows == 1                                       # shared keys: one seed list for all rows
    assert lay.seed_ld >= 4096 and lay.rep_ld >= 65536


def test_topk_scores_refusals(L):
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    # ld below max_len, negative rows, K outside [1, 4096], NULL lengths
    assert L.idx_topk_scores(one, 100, one, 4, 128, 16, one, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_scores(one, 128, one, -1, 128, 16, one, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_scores(one, 128, one, 4, 128, 0, one, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_scores(one, 128, one, 4, 128, 4097, one, nul, one, 1 << 30, nul) == 4
    assert L.idx_topk_scores(one, 128, nul, 4, 128, 16, one, nul, one, 1 << 30, nul) == 4
    need = L.idx_topk_scores_workspace_size(4, 1 << 16, 16)
    if need > 0:
        assert L.idx_topk_scores(one, 1 << 16, one, 4, 1 << 16, 16, one, nul, one, need - 1, nul) == 6
    assert L.idx_topk_scores(nul, 0, nul, 0, 0, 16, nul, nul, nul, 0, nul) == 0      # no rows


def test_block_select_static_refusals(L):
    """The fixed-array entry point checks Q x n_kv x blocks against its 2^23
    block scores by division, so sizes whose product would wrap are refused
    too; all before any device work."""
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    cfg = B.block_sparse_config(128, 32, 1, 2)
    assert L.block_select_static(one, one, one, 4, 2, 128, 1024, None, one, 32, nul, nul) == 4      # NULL config
    assert L.block_select_static(one, one, one, 4, 2, 128, 1024, ctypes.byref(cfg), one, 31, nul, nul) == 4
    assert L.block_select_static(one, one, one, 4, 2, 512, 1024, ctypes.byref(cfg), one, 32, nul, nul) == 5
    big = 1 << 23
    assert L.block_select_static(one, one, one, big, 2, 128, 1024, ctypes.byref(cfg), one, 32, nul, nul) == 6
    # Q * n_kv * blocks far past 2^63 (a product computed first would wrap)
    assert L.block_select_static(one, one, one, 1 << 40, 1 << 20, 128, 1 << 62, ctypes.byref(cfg), one, 32,
                                 nul, nul) == 6
    assert L.block_select_static(one, one, one, 0, 2, 128, 1024, ctypes.byref(cfg), one, 32, nul, nul) == 0


def test_problem_size_bounds(L):
    """Problems whose derived sizes would leave 64-bit arithmetic are refused."""
    from sparse_attention_indexer_idx_gb300 import binding as B
    nul = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    huge_m = B.idx_problem(one, B.IDX_F32, one, (1 << 40) + 1, 4, 16, one, B.IDX_F32, one, 1 << 20, None, one, 16)
    assert L.idx_score(ctypes.byref(huge_m), one, 16, nul) == 5
    wide = B.idx_problem(one, B.IDX_F32, one, 1 << 30, 4, 16, one, B.IDX_F32, one, 1 << 40, None, one, 1 << 30)
    assert L.idx_score(ctypes.byref(wide), one, 1 << 30, nul) == 5
    many_keys = B.idx_problem(one, B.IDX_F32, one, 4, 4, 16, one, B.IDX_F32, one, (1 << 46) + 1, None, one, 16)
    assert L.idx_score(ctypes.byref(many_keys), one, 16, nul) == 5
    assert b"too large" in L.idx_last_error_string()


def test_binding_checks_buffers():
    """The binding checks each output buffer's dtype and size before the call
    (the C ABI takes plain pointers): a short or mistyped buffer raises."""
    import torch
    from sparse_attention_indexer_idx_gb300 import binding as B
    with pytest.raises(ValueError, match="expected torch.int32"):
        B._buf(torch.zeros(8, dtype=torch.int64), torch.int32, 8, "out_ids")
    with pytest.raises(ValueError, match="the call needs 8"):
        B._buf(torch.zeros(7, dtype=torch.int32), torch.int32, 8, "out_ids")
    with pytest.raises(ValueError, match="CUDA tensor"):
        B._buf(torch.zeros(8, dtype=torch.int32), torch.int32, 8, "out_ids")
    assert B._buf(None, torch.int32, 8, "out_scores") is None


def test_binding_row_span():
    from sparse_attention_indexer_idx_gb300 import binding as B
    assert B._rows_need(0, 100, 50) == 0
    assert B._rows_need(4, 100, 0) == 0
    assert B._rows_need(1, 100, 50) == 50
    assert B._rows_need(4, 100, 100) == 400
    assert B._rows_need(4, 128, 100) == 3 * 128 + 100
