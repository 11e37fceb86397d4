"""Thin Python binding of libidx (ctypes).  Argument marshalling only: every
step of the computation runs in the library's CUDA kernels.

The functions carry the C names (idx_score, idx_topk, idx_topk_scores,
dosa_topk, witness_merge, witness_indices, block_select) and take torch CUDA
tensors; torch provides device memory and streams, nothing else.  A non-zero
status raises IdxError with the library's message.  If libidx.so has not been
built the import fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libidx.so")

IDX_OK = 0
STATUS_NAMES = {1: "ROWS_MISMATCH", 2: "SEGMENTS_OUT_OF_RANGE", 3: "KEEP_OUT_OF_RANGE", 4: "INVALID_ARG",
                5: "UNSUPPORTED", 6: "WORKSPACE_TOO_SMALL", 7: "CUDA"}
IDX_F32, IDX_BF16, IDX_FP8_E4M3 = 0, 1, 2
IDX_MAX_SEGMENTS, IDX_MAX_K = 64, 4096
DEVERR_WAIT_TIMEOUT, DEVERR_BAD_ROW, DEVERR_CAPACITY = 1, 2, 4


class IdxError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))


class idx_problem(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int32), ("w", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
                ("keys", ctypes.c_void_p), ("k_dtype", ctypes.c_int32), ("key_scale", ctypes.c_void_p),
                ("n_keys", ctypes.c_int64), ("key_off", ctypes.c_void_p), ("key_len", ctypes.c_void_p),
                ("max_key_len", ctypes.c_int32)]


class dosa_params(ctypes.Structure):
    _fields_ = [("n_seed", ctypes.c_int32), ("retained_heads", ctypes.c_int32), ("n_sample", ctypes.c_int32),
                ("act_freq_min", ctypes.c_float), ("margin_gamma", ctypes.c_float),
                ("candidate_capacity", ctypes.c_int32), ("group_stream", ctypes.c_int32)]


class dosa_stats(ctypes.Structure):
    _fields_ = [("pairs", ctypes.c_ulonglong), ("seeds", ctypes.c_ulonglong), ("candidates", ctypes.c_ulonglong),
                ("survivors", ctypes.c_ulonglong), ("fallback_rows", ctypes.c_ulonglong),
                ("skipped_rows", ctypes.c_ulonglong), ("group_keys", ctypes.c_ulonglong),
                ("solo_keys", ctypes.c_ulonglong)]

DOSA_STATS_FIELDS = len(dosa_stats._fields_)   # int64 counters of a device dosa_stats


class dosa_ws_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("seed_list", "seed_count", "rep_count", "rep_scores", "tau", "status",
                                             "plan_head", "plan_beta", "plan_dnorm", "wfold", "coef", "qprep",
                                             "seed_ld", "rep_ld", "seed_rows")] + \
               [("group_layout", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class topk_prior_stats(ctypes.Structure):
    _fields_ = [("rows_filtered", ctypes.c_ulonglong), ("candidates", ctypes.c_ulonglong),
                ("dense_rows", ctypes.c_ulonglong)]


class block_select_stats(ctypes.Structure):
    _fields_ = [("pairs", ctypes.c_ulonglong), ("blocks_bounded", ctypes.c_ulonglong),
                ("blocks_rescored", ctypes.c_ulonglong), ("fallback_pairs", ctypes.c_ulonglong),
                ("max_bound_use", ctypes.c_float), ("reserved", ctypes.c_float)]


def block_select_stats_tensor(device="cuda") -> torch.Tensor:
    """Zeroed device storage for one block_select_stats (40 bytes)."""
    return torch.zeros(5, dtype=torch.int64, device=device)


def block_select_stats_read(t: torch.Tensor) -> dict:
    """block_select_stats storage -> dict (copies to the host)."""
    h = t.detach().cpu()
    u = h.tolist()
    f = h[4:5].view(torch.float32).tolist()
    return {"pairs": u[0], "blocks_bounded": u[1], "blocks_rescored": u[2], "fallback_pairs": u[3],
            "max_bound_use": f[0]}


class block_sparse_config(ctypes.Structure):
    _fields_ = [("block_size", ctypes.c_int32), ("top_blocks", ctypes.c_int32), ("init_blocks", ctypes.c_int32),
                ("local_blocks", ctypes.c_int32)]


EXPORTS = {
    "idx_last_error_string": (ctypes.c_char_p, []),
    "idx_device_error": (ctypes.c_uint32, []),
    "idx_set_wait_limit_ns": (ctypes.c_int32, [ctypes.c_uint64]),
    "idx_score": (ctypes.c_int32, [ctypes.POINTER(idx_problem), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    "idx_topk_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(idx_problem), ctypes.c_int32]),
    "idx_topk": (ctypes.c_int32, [ctypes.POINTER(idx_problem), ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "idx_topk_scores_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]),
    "idx_topk_scores": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "dosa_topk_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(idx_problem), ctypes.c_int32,
                                                   ctypes.POINTER(dosa_params), ctypes.c_int32]),
    "dosa_topk": (ctypes.c_int32, [ctypes.POINTER(idx_problem), ctypes.c_int32, ctypes.POINTER(dosa_params),
                                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.c_void_p]),
    "dosa_workspace_layout": (ctypes.c_int32, [ctypes.POINTER(idx_problem), ctypes.c_int32,
                                               ctypes.POINTER(dosa_params), ctypes.c_int32,
                                               ctypes.POINTER(dosa_ws_layout)]),
    "witness_merge": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_void_p]),
    "witness_indices": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "block_select_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                                                      ctypes.POINTER(block_sparse_config)]),
    "block_select": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                      ctypes.POINTER(block_sparse_config), ctypes.c_void_p, ctypes.c_int32,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_void_p]),
    "block_select_events": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                             ctypes.POINTER(block_sparse_config), ctypes.c_void_p, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "idx_topk_prior_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(idx_problem), ctypes.c_int32, ctypes.c_int32,
                                                        ctypes.c_int32]),
    "idx_topk_prior": (ctypes.c_int32, [ctypes.POINTER(idx_problem), ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "idx_topk_prior_events": (ctypes.c_int32, [ctypes.POINTER(idx_problem), ctypes.c_int32, ctypes.c_void_p,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                               ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "block_positions": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "block_select_static": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                             ctypes.POINTER(block_sparse_config), ctypes.c_void_p, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libidx.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libidx.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(st: int) -> None:
    if st != IDX_OK:
        raise IdxError(st, lib().idx_last_error_string().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _buf(t: Optional[torch.Tensor], dtype: torch.dtype, numel: int, name: str):
    """A caller's device buffer that the library writes or reads as `numel`
    elements of `dtype` (the C ABI takes plain pointers, so this is the last
    place where a short or mistyped buffer can be caught)."""
    if t is None:
        return None
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, the call needs {numel}")
    return _ptr(t)


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


_DT = {torch.float32: IDX_F32, torch.bfloat16: IDX_BF16, torch.uint8: IDX_FP8_E4M3,
       torch.float8_e4m3fn: IDX_FP8_E4M3}


@dataclass
class Problem:
    """Device tensors of one indexer batch (see idx_problem in include/idx.h)."""
    q: torch.Tensor                     # [M, H, D] float32 or bfloat16
    w: torch.Tensor                     # [M, H] float32
    keys: torch.Tensor                  # [n_keys, D] float32 / bfloat16 / uint8 (e4m3 codes)
    key_len: torch.Tensor               # [M] int32
    max_key_len: int
    key_off: Optional[torch.Tensor] = None   # [M] int64 or None (shared keys)
    key_scale: Optional[torch.Tensor] = None  # [n_keys] float32 for FP8 keys

    def c(self) -> idx_problem:
        M, H, D = self.q.shape
        return idx_problem(_ptr(self.q), _DT[self.q.dtype], _ptr(self.w), M, H, D, _ptr(self.keys),
                           _DT[self.keys.dtype], _ptr(self.key_scale), self.keys.shape[0], _ptr(self.key_off),
                           _ptr(self.key_len), int(self.max_key_len))


def device_error() -> int:
    """Synchronise and return (then clear) the library's device error word."""
    return int(lib().idx_device_error())


DEFAULT_WAIT_LIMIT_NS = 2_000_000_000


def set_wait_limit_ns(ns: int) -> None:
    """Limit of every pipeline wait in the library's kernels (current device)."""
    _check(lib().idx_set_wait_limit_ns(int(ns)))


def _rows_need(M: int, ld: int, width: int) -> int:
    """Elements that M rows of `width` values at row stride `ld` span."""
    return 0 if M <= 0 or width <= 0 else (M - 1) * ld + width


def idx_score(p: Problem, scores: torch.Tensor, ld: Optional[int] = None, stream=None) -> torch.Tensor:
    cp = p.c()
    ld = int(ld if ld is not None else scores.shape[-1])
    need = _rows_need(p.q.shape[0], ld, int(p.max_key_len))
    _check(lib().idx_score(ctypes.byref(cp), _buf(scores, torch.float32, need, "scores"), ld, _stream(stream)))
    return scores


def idx_topk_workspace_size(p: Problem, K: int) -> int:
    cp = p.c()
    return int(lib().idx_topk_workspace_size(ctypes.byref(cp), K))


def idx_topk(p: Problem, K: int, out_ids: torch.Tensor, out_scores: Optional[torch.Tensor], ws: torch.Tensor,
             stream=None):
    cp = p.c()
    MK = p.q.shape[0] * K
    _check(lib().idx_topk(ctypes.byref(cp), K, _buf(out_ids, torch.int32, MK, "out_ids"),
                          _buf(out_scores, torch.float32, MK, "out_scores"), _ptr(ws), ws.numel() * ws.element_size(),
                          _stream(stream)))
    return out_ids, out_scores


def idx_topk_prior_workspace_size(p: Problem, K: int, prior_ld: int, capacity: int) -> int:
    cp = p.c()
    return int(lib().idx_topk_prior_workspace_size(ctypes.byref(cp), K, prior_ld, capacity))


def idx_topk_prior(p: Problem, K: int, prior_ids: torch.Tensor, capacity: int, out_ids: torch.Tensor,
                   out_scores: Optional[torch.Tensor], ws: torch.Tensor, row_status: Optional[torch.Tensor] = None,
                   stats: Optional[torch.Tensor] = None, stream=None):
    """Top-K with the previous step's selection prior_ids [M, prior_ld] as a prior.
    stats: torch.zeros(3, dtype=torch.int64) storage for topk_prior_stats, or None."""
    cp = p.c()
    M = p.q.shape[0]
    _check(lib().idx_topk_prior(ctypes.byref(cp), K, _buf(prior_ids, torch.int32, M * prior_ids.shape[1], "prior_ids"),
                                prior_ids.shape[1], capacity, _buf(out_ids, torch.int32, M * K, "out_ids"),
                                _buf(out_scores, torch.float32, M * K, "out_scores"),
                                _buf(row_status, torch.int32, M, "row_status"), _buf(stats, torch.int64, 3, "stats"),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
    return out_ids, out_scores


def idx_topk_prior_events(p: Problem, K: int, prior_ids: torch.Tensor, capacity: int, out_ids: torch.Tensor,
                          out_scores: Optional[torch.Tensor], ws: torch.Tensor, events, stream=None):
    """idx_topk_prior recording 6 torch.cuda.Event (already created) between its stages."""
    cp = p.c()
    M = p.q.shape[0]
    handles = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(e.cuda_event) for e in events[:6]])
    _check(lib().idx_topk_prior_events(ctypes.byref(cp), K,
                                       _buf(prior_ids, torch.int32, M * prior_ids.shape[1], "prior_ids"),
                                       prior_ids.shape[1], capacity, _buf(out_ids, torch.int32, M * K, "out_ids"),
                                       _buf(out_scores, torch.float32, M * K, "out_scores"), None, None, _ptr(ws),
                                       ws.numel() * ws.element_size(), handles, 6, _stream(stream)))
    return out_ids, out_scores


def idx_topk_scores_workspace_size(M: int, max_len: int, K: int) -> int:
    return int(lib().idx_topk_scores_workspace_size(M, max_len, K))


def idx_topk_scores(scores: torch.Tensor, lens: torch.Tensor, max_len: int, K: int, out_ids: torch.Tensor,
                    out_scores: Optional[torch.Tensor] = None, ld: Optional[int] = None,
                    ws: Optional[torch.Tensor] = None, stream=None):
    M = lens.shape[0]
    ld = int(ld if ld is not None else scores.shape[-1])
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().idx_topk_scores(_buf(scores, torch.float32, _rows_need(M, ld, int(max_len)), "scores"), ld,
                                 _buf(lens, torch.int32, M, "lens"), M, int(max_len), K,
                                 _buf(out_ids, torch.int32, M * K, "out_ids"),
                                 _buf(out_scores, torch.float32, M * K, "out_scores"), _ptr(ws), ws_bytes,
                                 _stream(stream)))
    return out_ids, out_scores


def make_dosa_params(n_seed=12288, retained_heads=16, n_sample=128, act_freq_min=0.5, margin_gamma=2.0 ** -10,
                     candidate_capacity=16384, group_stream=1) -> dosa_params:
    return dosa_params(n_seed, retained_heads, n_sample, act_freq_min, margin_gamma, candidate_capacity,
                       group_stream)


def dosa_topk_workspace_size(p: Problem, K: int, dp: dosa_params, seed_ld: int = 0) -> int:
    cp = p.c()
    return int(lib().dosa_topk_workspace_size(ctypes.byref(cp), K, ctypes.byref(dp), seed_ld))


def dosa_topk(p: Problem, K: int, dp: dosa_params, out_ids: torch.Tensor, out_scores: Optional[torch.Tensor],
              ws: torch.Tensor, seed_ids: Optional[torch.Tensor] = None, row_status: Optional[torch.Tensor] = None,
              stats: Optional[torch.Tensor] = None, stream=None):
    cp = p.c()
    M = p.q.shape[0]
    seed_ld = int(seed_ids.shape[1]) if seed_ids is not None else 0
    _check(lib().dosa_topk(ctypes.byref(cp), K, ctypes.byref(dp), _buf(seed_ids, torch.int32, M * seed_ld, "seed_ids"),
                           seed_ld, _buf(out_ids, torch.int32, M * K, "out_ids"),
                           _buf(out_scores, torch.float32, M * K, "out_scores"),
                           _buf(row_status, torch.int32, M, "row_status"),
                           _buf(stats, torch.int64, DOSA_STATS_FIELDS, "stats"), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream)))
    return out_ids, out_scores


def dosa_workspace_layout(p: Problem, K: int, dp: dosa_params, seed_ld: int = 0) -> dict:
    """Byte offsets (and row strides) of dosa_topk's intermediate arrays in its workspace."""
    cp = p.c()
    out = dosa_ws_layout()
    _check(lib().dosa_workspace_layout(ctypes.byref(cp), K, ctypes.byref(dp), seed_ld, ctypes.byref(out)))
    return {n: int(getattr(out, n)) for n, _ in dosa_ws_layout._fields_}


def witness_merge(topk_ids: torch.Tensor, context_lens: torch.Tensor, keep: int, num_segments: int,
                  max_replacements: int, rows: Optional[int] = None, topk: Optional[int] = None, stream=None):
    rows = topk_ids.shape[0] if rows is None else rows
    topk = topk_ids.shape[1] if topk is None else topk
    _check(lib().witness_merge(_ptr(topk_ids), rows, topk, _ptr(context_lens), context_lens.shape[0], keep,
                               num_segments, max_replacements, _stream(stream)))
    return topk_ids


def witness_indices(learned: torch.Tensor, context_lens: torch.Tensor, num_segments: int, out: torch.Tensor,
                    stream=None):
    rows, topk = learned.shape
    _check(lib().witness_indices(_ptr(learned), rows, topk, _ptr(context_lens), context_lens.shape[0], num_segments,
                                 _ptr(out), _stream(stream)))
    return out


def block_select_workspace_size(Q: int, n_kv: int, L: int, cfg: block_sparse_config) -> int:
    return int(lib().block_select_workspace_size(Q, n_kv, L, ctypes.byref(cfg)))


def block_select(index_q: torch.Tensor, index_k: torch.Tensor, query_pos: torch.Tensor, cfg: block_sparse_config,
                 out: torch.Tensor, out_count: Optional[torch.Tensor], ws: Optional[torch.Tensor], stream=None,
                 stats: Optional[torch.Tensor] = None):
    """stats: block_select_stats_tensor() storage or None."""
    Q, n_kv, D = index_q.shape
    L = index_k.shape[0]
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    if stats is not None and stats.numel() * stats.element_size() < ctypes.sizeof(block_select_stats):
        raise ValueError("stats needs 40 bytes")
    _check(lib().block_select(_ptr(index_q), _ptr(index_k), _ptr(query_pos), Q, n_kv, D, L, ctypes.byref(cfg),
                              _ptr(out), out.shape[-1], _ptr(out_count), _ptr(stats), _ptr(ws), ws_bytes,
                              _stream(stream)))
    return out, out_count


def block_select_events(index_q: torch.Tensor, index_k: torch.Tensor, query_pos: torch.Tensor,
                        cfg: block_sparse_config, out: torch.Tensor, out_count: Optional[torch.Tensor],
                        ws: Optional[torch.Tensor], events, stream=None, stats: Optional[torch.Tensor] = None):
    """block_select recording 6 torch.cuda.Event (already created: recorded once)
    between its kernels on `stream` (profiling)."""
    Q, n_kv, D = index_q.shape
    L = index_k.shape[0]
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    handles = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(e.cuda_event) for e in events[:6]])
    _check(lib().block_select_events(_ptr(index_q), _ptr(index_k), _ptr(query_pos), Q, n_kv, D, L, ctypes.byref(cfg),
                                     _ptr(out), out.shape[-1], _ptr(out_count), _ptr(stats), _ptr(ws), ws_bytes,
                                     handles, 6, _stream(stream)))
    return out, out_count


def block_positions(blocks: torch.Tensor, counts: Optional[torch.Tensor], query_pos: torch.Tensor, L: int,
                    block_size: int, out: torch.Tensor, out_count: Optional[torch.Tensor], stream=None):
    """blocks [Q, n_kv, W] int32 (as block_select writes them) -> covered positions
    [Q, n_kv, out_width] (ascending, -1 padded)."""
    Q, n_kv, W = blocks.shape
    _check(lib().block_positions(_ptr(blocks), _ptr(counts), Q, n_kv, W, _ptr(query_pos), L, block_size, _ptr(out),
                                 out.shape[-1], _ptr(out_count), _stream(stream)))
    return out, out_count


def problem_to_device(wp, device="cuda") -> Problem:
    """Copy a workloads.IndexerProblem (numpy, storage formats) to the device
    without changing a byte."""
    import numpy as np
    if wp.dtype == "f32":
        q = torch.from_numpy(np.ascontiguousarray(wp.q)).to(device)
        keys = torch.from_numpy(np.ascontiguousarray(wp.keys)).to(device)
    else:
        q = torch.from_numpy(np.ascontiguousarray(wp.q).view(np.int16)).to(device).view(torch.bfloat16)
        if wp.dtype == "bf16":
            keys = torch.from_numpy(np.ascontiguousarray(wp.keys).view(np.int16)).to(device).view(torch.bfloat16)
        else:
            keys = torch.from_numpy(np.ascontiguousarray(wp.keys)).to(device)
    w = torch.from_numpy(np.ascontiguousarray(wp.w, dtype=np.float32)).to(device)
    key_len = torch.from_numpy(np.ascontiguousarray(wp.key_len, dtype=np.int32)).to(device)
    key_off = None if wp.key_off is None else torch.from_numpy(np.ascontiguousarray(wp.key_off, dtype=np.int64)).to(device)
    key_scale = None if wp.key_scale is None else torch.from_numpy(np.ascontiguousarray(wp.key_scale)).to(device)
    return Problem(q, w, keys, key_len, int(np.max(wp.key_len)) if len(wp.key_len) else 0, key_off, key_scale)


def block_select_static(index_q: torch.Tensor, index_k: torch.Tensor, query_pos: torch.Tensor,
                        cfg: block_sparse_config, out: torch.Tensor, out_count: Optional[torch.Tensor], stream=None):
    """block_select without a workspace: the scratch is a fixed array inside the
    library (for callers that cannot allocate device memory)."""
    Q, n_kv, D = index_q.shape
    L = index_k.shape[0]
    _check(lib().block_select_static(_ptr(index_q), _ptr(index_k), _ptr(query_pos), Q, n_kv, D, L,
                                     ctypes.byref(cfg), _ptr(out), out.shape[-1], _ptr(out_count), _stream(stream)))
    return out, out_count
