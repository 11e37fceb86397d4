"""Pins of the DoSA oracle's planner readings and its cold seed rule.

The DoSA page (section 4, the `_cold_prior` and `_body` rows) names the steps
but not their rules; oracle.dosa states the readings it takes:
  * cold seeds: representatives m_i = floor(i (M-1) / 3), i = 0..3, scored over
    the common visible prefix; keys ranked by (number of representative top-K
    lists holding them desc, best representative score desc, id asc); the
    first n_seed;
  * retained heads: the R largest |w_h| ||q_h||, ties to the lower head;
  * anchor: the retained j minimising ||q_h - beta q_j||, beta = max(0,
    q_h.q_j / ||q_j||^2), ties to the lower j.
These tests hold the oracle to those readings by other means than the oracle's
own code: hand-built cases in which each plausible mistake (count ascending, no
best-score tie-break, id descending, the wrong representatives, keys beyond the
common prefix, |w| or ||q|| alone, signed w, the wrong residual) gives another
answer, and brute force on random integer inputs with many exact ties (pairwise
ranks instead of sorting, exact rational residuals instead of norms).
"""
from __future__ import annotations

import functools
from fractions import Fraction

import numpy as np
import pytest

from oracle import dosa
from sparse_attention_indexer_idx_gb300 import workloads as wl


# ------------------------------------------------------------ cold seed rule --

def _one_hot_problem(score_rows, key_len, K):
    """f32 problem with H = 1, w = 1 and one-hot keys, so that query m's score of
    key k is exactly max(score_rows[m][k], 0)."""
    S = np.asarray(score_rows, dtype=np.float32)
    M, n = S.shape
    q = S.reshape(M, 1, n).copy()
    keys = np.eye(n, dtype=np.float32)
    w = np.ones((M, 1), dtype=np.float32)
    return wl.IndexerProblem("one_hot", "f32", q, w, keys, np.asarray(key_len, dtype=np.int32), None, K)


# rows 0, 2, 4, 6 are the representatives of M = 7 (floor(i * 6 / 3)); rows
# 1, 3, 5 prefer keys 0 and 7; keys 8..13 lie beyond the common prefix (8) and
# score highest for every row.
_HI = 2.0
_COLD_ROWS = [
    # key: 0    1    2    3    4    5     6     7   | 8 .. 13
    [0.3, 0.9, 0.1, 0.8, 0.2, 0.1, 0.1, 0.1] + [_HI] * 6,    # rep: top-2 {1, 3}
    [1.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.99] + [_HI] * 6,   # not a rep
    [0.1, 0.9, 0.5, 0.1, 0.2, 0.85, 0.1, 0.1] + [_HI] * 6,   # rep: top-2 {1, 5}
    [1.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.99] + [_HI] * 6,   # not a rep
    [0.1, 0.1, 0.1, 0.7, 0.6, 0.1, 0.95, 0.5] + [_HI] * 6,   # rep: top-2 {6, 3}
    [1.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.99] + [_HI] * 6,   # not a rep
    [0.1, 0.9, 0.1, 0.1, 0.1, 0.1, 0.88, 0.1] + [_HI] * 6,   # rep: top-2 {1, 6}
]
# counts: key 1: 3, keys 3 and 6: 2, key 5: 1, the rest 0; best scores 0.3, 0.9,
# 0.5, 0.8, 0.6, 0.85, 0.95, 0.5 -> ranking 1, 6, 3, 5, 4, 2, 7, 0
_COLD_RANKING = [1, 6, 3, 5, 4, 2, 7, 0]


@pytest.mark.parametrize("n_seed", [1, 2, 3, 4, 5, 6, 7, 8, 50])
def test_cold_seeds_hand_built(n_seed):
    p = _one_hot_problem(_COLD_ROWS, key_len=[8, 9, 10, 11, 12, 13, 14], K=2)
    got = dosa.cold_seeds(p, n_seed, 2).tolist()
    want = sorted(_COLD_RANKING[:min(n_seed, 8)])
    assert got == want


def test_cold_seeds_hand_built_mistakes_would_show():
    """The hand-built case separates the reading from its plausible variants."""
    full = sorted(_COLD_RANKING[:2])                 # n_seed = 2: {1, 6}
    assert full != sorted([1, 3])                    # count tie broken by id instead of best score
    six = sorted(_COLD_RANKING[:6])                  # {1, 2, 3, 4, 5, 6}
    assert six != sorted([1, 6, 3, 5, 0, 2])         # no best-score tie-break among count 0
    assert six != sorted([1, 6, 3, 5, 4, 7])         # id descending among equal (count, best)
    p = _one_hot_problem(_COLD_ROWS, key_len=[8, 9, 10, 11, 12, 13, 14], K=2)
    assert dosa.cold_seeds(p, 6, 2).tolist() == six


def _brute_cold_seeds(S, common, n_seed, K):
    """Cold rule by pairwise ranks and a comparator sort over Python tuples."""
    M = len(S)
    reps = sorted(set((i * (M - 1)) // 3 for i in range(4)))
    count = [0] * common
    best = [None] * common
    for m in reps:
        row = S[m]
        for k in range(common):
            better = sum(1 for j in range(common) if row[j] > row[k] or (row[j] == row[k] and j < k))
            if better < K:
                count[k] += 1
            best[k] = row[k] if best[k] is None else max(best[k], row[k])

    def cmp(a, b):
        ka = (count[a], best[a])
        kb = (count[b], best[b])
        if ka != kb:
            return -1 if ka > kb else 1
        return -1 if a < b else (1 if a > b else 0)

    order = sorted(range(common), key=functools.cmp_to_key(cmp))
    return sorted(order[:min(n_seed, common)])


@pytest.mark.parametrize("trial", range(12))
def test_cold_seeds_brute_force_with_ties(trial):
    rng = np.random.default_rng(700 + trial)
    M = int(rng.integers(1, 10))
    n = int(rng.integers(4, 40))
    H, D = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    # small integers: every score is an exact integer, ties in counts and best scores abound
    q = rng.integers(-2, 3, (M, H, D)).astype(np.float32)
    w = rng.choice([-1.0, 1.0, 2.0], (M, H)).astype(np.float32)
    keys = rng.integers(-2, 3, (n, D)).astype(np.float32)
    key_len = np.sort(rng.integers(1, n + 1, M)).astype(np.int32)
    K = int(rng.integers(1, 6))
    n_seed = int(rng.integers(1, n + 3))
    p = wl.IndexerProblem("ties", "f32", q, w, keys, key_len, None, K)
    common = int(key_len.min())
    S = []
    for m in range(M):
        row = []
        for k in range(common):
            s = 0.0
            for h in range(H):
                dot = float(sum(float(q[m, h, d]) * float(keys[k, d]) for d in range(D)))
                s += float(w[m, h]) * max(dot, 0.0)
            row.append(s)
        S.append(row)
    assert dosa.cold_seeds(p, n_seed, K).tolist() == _brute_cold_seeds(S, common, n_seed, K)


# ------------------------------------------------------------ retained heads --

def test_retained_heads_hand_built():
    # |w| ||q||: 3, 5, 2, 4 -> R = 2 keeps heads 1 and 3; |w| alone would keep 0 and 3,
    # ||q|| alone 1 and 2, signed w 0 and 3
    q = np.array([[1.0, 0.0], [3.0, 4.0], [0.0, 4.0], [2.0, 0.0]])
    w = np.array([3.0, -1.0, 0.5, 2.0])
    assert dosa.choose_retained(q, w, 2).tolist() == [1, 3]
    assert dosa.choose_retained(q, w, 1).tolist() == [1]
    assert dosa.choose_retained(q, w, 3).tolist() == [0, 1, 3]
    assert dosa.choose_retained(q, w, 9).tolist() == [0, 1, 2, 3]


def test_retained_heads_ties_go_to_the_lower_head():
    # |w| ||q|| = 4, 4, 4, 1: R = 2 keeps heads 0 and 1, R = 1 keeps head 0
    q = np.array([[2.0, 0.0], [0.0, 1.0], [4.0, 0.0], [1.0, 0.0]])
    w = np.array([2.0, -4.0, 1.0, 1.0])
    assert dosa.choose_retained(q, w, 2).tolist() == [0, 1]
    assert dosa.choose_retained(q, w, 1).tolist() == [0]
    # the same magnitudes listed the other way round: still the lower heads
    assert dosa.choose_retained(q[[3, 2, 1, 0]], w[[3, 2, 1, 0]], 2).tolist() == [1, 2]


@pytest.mark.parametrize("trial", range(30))
def test_retained_heads_brute_force(trial):
    rng = np.random.default_rng(800 + trial)
    H, D = int(rng.integers(1, 12)), int(rng.integers(1, 5))
    q = rng.integers(-2, 3, (H, D)).astype(np.float64)
    w = rng.choice([-4.0, -2.0, -1.0, 0.0, 1.0, 2.0, 4.0], H)
    R = int(rng.integers(1, H + 2))
    # exact comparison of |w| ||q|| through w^2 (q.q), integers
    mag2 = [int(w[h] ** 2) * int(q[h] @ q[h]) for h in range(H)]
    want = [h for h in range(H)
            if sum(1 for g in range(H) if mag2[g] > mag2[h] or (mag2[g] == mag2[h] and g < h)) < R]
    assert dosa.choose_retained(q, w, R).tolist() == want


# ------------------------------------------------------------------- anchors --

def test_anchor_hand_built():
    q = np.array([
        [2.0, 1.0],    # 0: the omitted head
        [1.0, 0.0],    # 1: beta 2, residual (0, 1) -> 1
        [0.0, 1.0],    # 2: beta 1, residual (2, 0) -> 2
        [-1.0, 0.0],   # 3: negative dot -> beta 0, residual ||q_h|| = sqrt 5
        [1.0, 0.0],    # 4: same as head 1 (a tie: the lower head wins)
    ])
    j, beta, r = dosa.choose_anchor(q[0], q, [1, 2, 3, 4])
    assert (j, beta, r) == (1, 2.0, 1.0)
    j, beta, r = dosa.choose_anchor(q[0], q, [4, 2, 3, 1])
    assert j == 1 and beta == 2.0
    j, beta, r = dosa.choose_anchor(q[0], q, [2, 3])
    assert (j, beta, r) == (2, 1.0, 2.0)
    j, beta, r = dosa.choose_anchor(q[0], q, [3])
    assert j == 3 and beta == 0.0 and r == pytest.approx(np.sqrt(5.0), rel=1e-15)


def _brute_anchor(qh, q, retained):
    """argmin over j of ||q_h||^2 - max(0, q_h.q_j)^2 / ||q_j||^2 (the squared
    residual at the best beta >= 0), exact rationals, ties to the lower j."""
    qh = [int(x) for x in qh]
    n_h = sum(x * x for x in qh)
    best, best_j = None, None
    for j in sorted(int(t) for t in retained):
        qj = [int(x) for x in q[j]]
        nj = sum(x * x for x in qj)
        dot = sum(a * b for a, b in zip(qh, qj))
        r2 = Fraction(n_h) if (nj == 0 or dot <= 0) else Fraction(n_h) - Fraction(dot * dot, nj)
        if best is None or r2 < best:
            best, best_j = r2, j
    return best_j, best


@pytest.mark.parametrize("trial", range(40))
def test_anchor_brute_force(trial):
    rng = np.random.default_rng(900 + trial)
    H, D = int(rng.integers(2, 10)), int(rng.integers(1, 5))
    q = rng.integers(-3, 4, (H, D)).astype(np.float64)
    if trial % 3 == 0:
        q[rng.integers(0, H)] = q[rng.integers(0, H)]     # repeated vectors: exact ties
    h = int(rng.integers(0, H))
    retained = sorted(set(int(x) for x in rng.choice(H, int(rng.integers(1, H + 1)), replace=False)) - {h}) or \
        [(h + 1) % H]
    j, beta, r = dosa.choose_anchor(q[h], q, retained)
    bj, r2 = _brute_anchor(q[h], q, retained)
    # the oracle's pick has the smallest exact squared residual; among exact ties the lowest j
    _, r2_got = _brute_anchor(q[h], q, [j])
    assert r2_got == r2
    tied = [t for t in retained if _brute_anchor(q[h], q, [t])[1] == r2]
    assert j == min(tied) == bj
    assert r == pytest.approx(float(r2) ** 0.5, rel=1e-12, abs=1e-12)
    nj = float(q[j] @ q[j])
    want_beta = max(0.0, float(q[h] @ q[j]) / nj) if nj > 0 else 0.0
    assert beta == pytest.approx(want_beta, rel=1e-15)
