"""Comparison helpers shared by the GPU parity tests (test-side only)."""
import re

import numpy as np

# Tolerance of a score, relative to a(k) = sum_h |w_h| ReLU(q_h.k): 1e-3 for
# fp32 / bf16 inputs, 2e-2 for FP8 keys.
EPS = {"f32": 1e-3, "bf16": 1e-3, "fp8": 2e-2}


def header_functions(path):
    """Names of the functions declared in a C header."""
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+([A-Za-z_][A-Za-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return", "sizeof")))


def check_scores(s_gpu, s_ref, a_ref, eps):
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    err = np.abs(s_gpu - s_ref)
    tol = eps * (a_ref + 1e-30)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} scores out of tolerance, e.g. id {bad[0]}: gpu {s_gpu[bad[0]]} ref {s_ref[bad[0]]} a {a_ref[bad[0]]}"


def check_topk_row(g_ids, g_sc, s_ref, a_ref, K, eps):
    """GPU top-K row vs the oracle's full score row (ids 0..L-1).

    * ids distinct, in range, -1 padding exactly when L < K;
    * reported scores within tolerance of the oracle score of that id;
    * order: non-increasing score, ties by ascending id;
    * the id set equals the oracle's except for keys whose oracle score lies
      within tolerance of the oracle's K-th score.
    """
    L = s_ref.shape[0]
    n = min(L, K)
    g_ids = np.asarray(g_ids)
    assert (g_ids[n:] == -1).all(), "padding"
    real = g_ids[:n]
    assert (real >= 0).all() and (real < L).all(), "id range"
    assert len(set(real.tolist())) == n, "distinct"
    if g_sc is not None:
        g_sc = np.asarray(g_sc, dtype=np.float64)
        assert np.isneginf(g_sc[n:]).all()
        check_scores(g_sc[:n], s_ref[real], a_ref[real], eps)
        for j in range(n - 1):
            assert g_sc[j] > g_sc[j + 1] or (g_sc[j] == g_sc[j + 1] and real[j] < real[j + 1]), f"order at {j}"
    if n == 0:
        return
    order = np.lexsort((np.arange(L), -s_ref))
    o_ids = order[:n]
    kth = o_ids[-1]
    s_k, a_k = s_ref[kth], a_ref[kth]
    diff = set(real.tolist()) ^ set(o_ids.tolist())
    for x in diff:
        assert abs(s_ref[x] - s_k) <= eps * (a_ref[x] + a_k) + 1e-30, f"id {x} differs and is not near the K-th score"


# ---------------------------------------------------------------------------
# The oracle on every host core: a pool of spawned worker processes (spawned,
# so that no worker inherits the test process's CUDA context), each running
# its BLAS on one thread.  A worker holds one problem (the pool initializer's);
# a task names a row of it, or carries a one-row problem of its own.

_POOL_PROBLEM = None


def _pool_init(problem):
    global _POOL_PROBLEM
    _POOL_PROBLEM = problem


def oracle_pool(problem=None):
    import multiprocessing as mp
    import os
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return mp.get_context("spawn").Pool(n, initializer=_pool_init, initargs=(problem,))


def row_check_task(task):
    """(problem or None, row, gpu ids, gpu scores, eps): check_topk_row of that
    row against oracle.dsa (None: the worker's problem)."""
    from oracle import dsa as odsa
    prob, m, ids, sc, eps = task
    wp = _POOL_PROBLEM if prob is None else prob
    s_ref, a_ref = odsa.row_scores(wp, m)
    check_topk_row(ids, sc, s_ref, a_ref, wp.K, eps)
    return m


def block_select_task(i):
    """oracle.block_select's selection of query i of the worker's problem."""
    from oracle import block_select as obs
    bp = _POOL_PROBLEM
    return i, obs.block_sparse_select(bp.index_q[i], bp.index_k, int(bp.query_pos[i]), bp.block_size,
                                      bp.top_blocks, bp.init_blocks, bp.local_blocks)


def sub_problem(wp, rows):
    """Rows `rows` of an indexer problem as a problem of their own; per-row keys
    are gathered, a shared key sequence is cut to what those rows see."""
    from sparse_attention_indexer_idx_gb300 import workloads as wl
    rows = np.asarray(rows, dtype=np.int64)
    key_len = np.asarray(wp.key_len)[rows].astype(np.int32)
    scale = None
    if wp.key_off is None:
        n = int(key_len.max())
        keys, key_off = wp.keys[:n], None
        if wp.key_scale is not None:
            scale = wp.key_scale[:n]
    else:
        offs = np.asarray(wp.key_off)[rows]
        keys = np.concatenate([wp.keys[o:o + l] for o, l in zip(offs, key_len)])
        if wp.key_scale is not None:
            scale = np.concatenate([wp.key_scale[o:o + l] for o, l in zip(offs, key_len)])
        key_off = np.concatenate([[0], np.cumsum(key_len.astype(np.int64))[:-1]]).astype(np.int64)
    extras = {k: v for k, v in wp.extras.items() if k != "pad_mask"}
    return wl.IndexerProblem(wp.name, wp.dtype, wp.q[rows], wp.w[rows], keys, key_len, key_off, wp.K,
                             key_scale=scale, extras=extras)
