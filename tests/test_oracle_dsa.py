"""Pins of the indexer-score and top-K oracle: the DoSA page's section 3
worked example, closed forms and brute force on tiny inputs."""
import itertools
import json
import os

import numpy as np

from oracle import dsa
from sparse_attention_indexer_idx_gb300 import workloads as wl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "dosa_examples.json")))


def test_worked_example_score():
    g = GOLD["score"]
    # one key k = e0; head h's query is activation_h * e0, so q_h . k = activation_h
    k = np.array([[1.0, 0.0]])
    q = np.array([[a, 0.0] for a in g["activations"]])
    s, a = dsa.indexer_score(q, g["w"], k)
    assert s[0] == g["s"]
    assert a[0] == 2 * 4 + 1 * 3
    # a negative dot passes ReLU as 0 even under a negative weight
    q2 = np.array([[4.0, 0.0], [-3.0, 0.0]])
    s2, _ = dsa.indexer_score(q2, g["w"], k)
    assert s2[0] == 8.0


def _brute_score(q, w, k):
    H, D = q.shape
    out = []
    for key in k:
        tot = 0.0
        for h in range(H):
            dot = 0.0
            for d in range(D):
                dot += float(q[h, d]) * float(key[d])
            tot += float(w[h]) * (dot if dot > 0 else 0.0)
        out.append(tot)
    return np.array(out)


def test_score_bruteforce_nonsquare():
    rng = np.random.default_rng(31)
    for H, D, L in [(3, 5, 7), (1, 2, 9), (5, 3, 4)]:
        q = rng.standard_normal((H, D))
        w = rng.uniform(-1, 1, H)
        k = rng.standard_normal((L, D))
        s, a = dsa.indexer_score(q, w, k)
        np.testing.assert_allclose(s, _brute_score(q, w, k), rtol=0, atol=1e-12)
        np.testing.assert_allclose(a, _brute_score(q, np.abs(w), k), rtol=0, atol=1e-12)


def test_single_head_closed_form():
    rng = np.random.default_rng(32)
    q = rng.standard_normal((1, 6))
    k = rng.standard_normal((50, 6))
    s, _ = dsa.indexer_score(q, [1.0], k)
    np.testing.assert_allclose(s, np.maximum(k @ q[0], 0), atol=1e-12)


def _brute_topk(s, K):
    """Rank of each element = number of elements strictly better under
    (score desc, id asc); the top-K are those with rank < K, in rank order."""
    n = len(s)
    rank = [sum(1 for j in range(n) if (s[j] > s[i]) or (s[j] == s[i] and j < i)) for i in range(n)]
    ids = [i for i in sorted(range(n), key=lambda i: rank[i]) if rank[i] < K]
    return ids + [-1] * (K - len(ids))


def test_topk_bruteforce_with_ties_and_short_rows():
    rng = np.random.default_rng(33)
    for _ in range(200):
        n = int(rng.integers(0, 40))
        K = int(rng.integers(1, 20))
        s = rng.integers(-3, 4, n).astype(np.float64)     # many exact ties
        ids, sc = dsa.topk(s, K)
        assert ids.tolist() == _brute_topk(s.tolist(), K)
        assert all(np.isneginf(sc[ids < 0]))
    # -0.0 ties with +0.0 and falls back to the id order
    ids, _ = dsa.topk(np.array([0.0, -0.0, 0.0]), 3)
    assert ids.tolist() == [0, 1, 2]


def test_topk_with_explicit_ids():
    s = np.array([1.0, 3.0, 3.0, 2.0])
    ids, sc = dsa.topk(s, 3, np.array([40, 7, 5, 9]))
    assert ids.tolist() == [5, 7, 9] and sc.tolist() == [3.0, 3.0, 2.0]


def test_fp8_rows_scale_the_keys():
    p = wl.ragged_fp8(seed=1, M=2, H=4, D=8, L_min=5, L_max=9, K=3)
    for m in range(2):
        k = p.keys_f32()[p.key_off[m]:p.key_off[m] + p.key_len[m]].astype(np.float64)
        sc = p.key_scale[p.key_off[m]:p.key_off[m] + p.key_len[m]].astype(np.float64)
        s, _ = dsa.row_scores(p, m)
        ref = _brute_score(p.q_f32()[m], p.w[m], k * sc[:, None])
        np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
        # positive per-token scale factors out of the ReLU
        s_unscaled, _ = dsa.indexer_score(p.q_f32()[m], p.w[m], k)
        np.testing.assert_allclose(s, s_unscaled * sc, rtol=1e-12, atol=1e-12)


def test_a_planted_transpose_is_caught():
    """Using q^T k with the roles of heads and dims swapped changes the worked example."""
    q = np.array([[4.0, 0.0], [3.0, 0.0]])
    k = np.array([[1.0, 0.0]])
    s, _ = dsa.indexer_score(q, [2.0, -1.0], k)
    wrong = np.maximum(k @ q, 0) @ np.array([2.0, -1.0])
    assert s[0] == 5.0 and wrong[0] != 5.0
