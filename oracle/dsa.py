"""Oracle for the DSA indexer score and the exact top-K (fp64).

Test infrastructure only (see the package docstring).

Sources:
  * "DoSA：用安全上界减少 Indexer 的完整打分", section 3 (the indexer score
    s(k) = sum_h w_h [q_h^T k]_+, index key shared across heads, weights of
    either sign, no softmax).
  * same page, section 1 and the note after section 2 (the final choice is the
    top-K by the original scorer; equal ids across runs need one consistent
    total order).  The order used is score descending, then key id ascending.
"""
from __future__ import annotations

import numpy as np

NEG_INF = float("-inf")


def relu(x: np.ndarray) -> np.ndarray:
    """[x]_+ = max(x, 0) (section 3)."""
    return np.maximum(x, 0.0)


def head_activations(q_m: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """All q_h^T k for one query: keys [L, D], q_m [H, D] -> [L, H] (fp64)."""
    return np.asarray(keys, dtype=np.float64) @ np.asarray(q_m, dtype=np.float64).T


def indexer_score(q_m: np.ndarray, w_m: np.ndarray, keys: np.ndarray):
    """s(k) = sum_h w_h [q_h^T k]_+ for every key row (section 3).

    Returns (s, a) where a(k) = sum_h |w_h| [q_h^T k]_+ is the magnitude the
    score is built from; the parity tolerance is relative to it so that
    cancellation between heads of opposite sign cannot blow it up.
    """
    act = relu(head_activations(q_m, keys))
    w = np.asarray(w_m, dtype=np.float64)
    return act @ w, act @ np.abs(w)


def dequantised_keys(problem, m: int) -> np.ndarray:
    """The visible keys of row m as fp64 values (FP8 keys times their scale)."""
    off = problem.row_offset(m)
    n = int(problem.key_len[m])
    k = problem.keys_f32(off, off + n).astype(np.float64)
    if problem.key_scale is not None:
        k = k * problem.key_scale[off:off + n].astype(np.float64)[:, None]
    return k


def row_scores(problem, m: int):
    """Scores of every visible key of row m (ids 0..key_len-1)."""
    q = problem.q_f32()[m]
    return indexer_score(q, problem.w[m], dequantised_keys(problem, m))


def topk_order(scores: np.ndarray, ids: np.ndarray | None = None) -> np.ndarray:
    """Indices of `scores` sorted by the total order (score desc, id asc).

    -0.0 and +0.0 compare equal, as they do under IEEE comparison.
    """
    s = np.asarray(scores, dtype=np.float64)
    if ids is None:
        ids = np.arange(s.shape[0], dtype=np.int64)
    return np.lexsort((np.asarray(ids, dtype=np.int64), -s))


def topk(scores: np.ndarray, K: int, ids: np.ndarray | None = None):
    """The K best (id, score) under (score desc, id asc), sorted in that order.

    Rows with fewer than K entries are padded with id -1 and score -inf.
    """
    s = np.asarray(scores, dtype=np.float64)
    if ids is None:
        ids = np.arange(s.shape[0], dtype=np.int64)
    ids = np.asarray(ids, dtype=np.int64)
    order = topk_order(s, ids)[:K]
    out_ids = np.full(K, -1, dtype=np.int64)
    out_s = np.full(K, NEG_INF, dtype=np.float64)
    out_ids[:order.shape[0]] = ids[order]
    out_s[:order.shape[0]] = s[order]
    return out_ids, out_s


def row_topk(problem, m: int, K: int | None = None):
    """Exact top-K of row m of an indexer problem: (ids, scores, s_all, a_all)."""
    K = problem.K if K is None else K
    s, a = row_scores(problem, m)
    ids, sc = topk(s, K)
    return ids, sc, s, a
