"""Pins of the block-select oracle against the "ferrox_core/block_sparse.rs"
page: the module's unit tests with their printed outputs
(tests/golden/block_select_examples.json), brute force on small inputs and
the dot's sequential f32 order."""
import json
import os

import numpy as np

from oracle import block_select as B

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "block_select_examples.json")))


def _keys(case):
    n = case["n"]
    if "all" in case:
        return np.tile(np.array(case["all"], dtype=np.float32), (n, 1))
    if "set" in case:
        k = np.zeros((n, 2), dtype=np.float32)
        for p, v in case["set"].items():
            k[int(p)] = v
        return k
    k = np.tile(np.array([0.0, 0.01], dtype=np.float32), (n, 1))
    for p in case["hot"]:
        k[p] = [1.0, 0.0]
    return k


def _select(case, keys=None, pos=None):
    bs, top, init, local = case["cfg"]
    keys = _keys(case) if keys is None else keys
    q = np.array(case["q"], dtype=np.float32)
    return B.block_sparse_select(q, keys, case["pos"] if pos is None else pos, bs, top, init, local)


def test_printed_cases():
    for c in GOLD["cases"]:
        sel = _select(c)
        if "expected" in c:
            assert sel == c["expected"], c["name"]
        if "contains" in c:
            for h, need in enumerate(c["contains"]):
                assert set(need) <= set(sel[h]), c["name"]
        if "length" in c:
            assert len(sel[0]) == c["length"], c["name"]
        if "max_block" in c:
            assert all(b <= c["max_block"] for b in sel[0]), c["name"]
        if "covered" in c:
            assert B.positions_of_blocks(sel[0], c["pos"], c["n"], c["cfg"][0]) == c["covered"], c["name"]


def test_per_head_independence():
    c = GOLD["per_head"]
    sel = _select(c)
    assert len(sel) == 2
    for h, need in enumerate(c["contains"]):
        assert set(need) <= set(sel[h])
    assert sel[0] != sel[1]


def test_never_empty_and_causal():
    c = GOLD["never_empty"]
    for pos in c["positions"]:
        sel = _select(c, pos=pos)
        assert sel[0]
        cov = B.positions_of_blocks(sel[0], pos, c["n"], c["cfg"][0])
        assert cov and all(p <= pos for p in cov)


def test_order_only_under_positive_scaling():
    c = GOLD["cases"][0]
    k = _keys(c)
    assert _select(c, keys=k) == _select(c, keys=k * np.float32(1000.0))


def test_causal_blocks_and_defaults():
    c = GOLD["causal_blocks"]
    assert B.MINIMAX_BLOCK_SIZE == c["block_size"] == c["defaults"]["block_size"]
    assert [B.causal_blocks(c["block_size"], p) for p in c["pos"]] == c["blocks"]
    assert B.causal_blocks(0, 5) == 0
    assert B.block_sparse_select(np.ones((2, 2), np.float32), np.ones((8, 2), np.float32), 5, 0, 3, 1, 1) == [[], []]


def test_dot_is_sequential_f32():
    """The sum must be left to right in f32: (1e8 + 1) - 1e8 loses the 1 in f32
    but a pairwise or fp64 sum keeps it."""
    q = np.array([1.0, 1.0, 1.0], dtype=np.float32)
    k = np.array([[1e8, 1.0, -1e8]], dtype=np.float32)
    assert B.dot_f32(q, k)[0] == np.float32(0.0)
    k2 = np.array([[1e8, -1e8, 1.0]], dtype=np.float32)
    assert B.dot_f32(q, k2)[0] == np.float32(1.0)
    # products are rounded to f32 before the add (no fused multiply-add)
    a = np.float32(1.0 + 2.0 ** -12)
    q3 = np.array([a, np.float32(-1.0)], dtype=np.float32)
    k3 = np.array([[a, np.float32(np.float32(a) * np.float32(a))]], dtype=np.float32)
    assert B.dot_f32(q3, k3)[0] == np.float32(0.0)
    # -0.0 is returned as +0.0
    assert np.signbit(B.dot_f32(np.array([-1.0], np.float32), np.array([[0.0]], np.float32))[0]) == False


def _brute_select(q, keys, pos, bs, top, init, local):
    """Brute force: enumerate every subset of the non-forced blocks of the
    right size and keep the one whose sorted (score, -block) list is best."""
    import itertools
    L = keys.shape[0]
    n = min(pos // bs + 1, -(-L // bs))
    forced = set(range(min(init, n))) | set(range(max(n - local, 0), n))
    budget = max(top, len(forced))
    free = [b for b in range(n) if b not in forced]
    take = min(budget - len(forced), len(free))
    if take <= 0:
        return sorted(forced)
    sc = {}
    for b in free:
        vals = []
        for p in range(b * bs, min((b + 1) * bs, L, pos + 1)):
            acc = np.float32(0.0)
            for d in range(q.shape[0]):
                acc = np.float32(acc + np.float32(q[d] * keys[p, d]))
            vals.append(acc + np.float32(0.0))
        sc[b] = max(vals)
    best = None
    for sub in itertools.combinations(free, take):
        key = sorted(((-float(sc[b]), b) for b in sub))
        if best is None or key < best[0]:
            best = (key, sub)
    return sorted(forced | set(best[1]))


def test_bruteforce_small():
    rng = np.random.default_rng(21)
    for _ in range(60):
        bs = int(rng.integers(1, 5))
        L = int(rng.integers(1, 24))
        D = int(rng.integers(1, 5))
        keys = rng.standard_normal((L, D)).astype(np.float32)
        # a few exact ties
        if L > 3:
            keys[rng.integers(0, L)] = keys[0]
        q = rng.standard_normal((2, D)).astype(np.float32)
        pos = int(rng.integers(0, L + 5))
        top, init, local = int(rng.integers(0, 5)), int(rng.integers(0, 3)), int(rng.integers(0, 3))
        got = B.block_sparse_select(q, keys, pos, bs, top, init, local)
        for h in range(2):
            assert got[h] == _brute_select(q[h], keys, pos, bs, top, init, local)


def test_max_not_mean_separates():
    """A block with one strong position and weak neighbours must beat a block of
    uniformly mediocre positions (max 1.0 vs 0.1), although its mean is lower."""
    keys = np.array([[0, 0]] * 4 + [[1, 0], [-1, 0], [-1, 0], [-1, 0]] + [[0.1, 0]] * 4 + [[0, 0]] * 4,
                    dtype=np.float32)
    q = np.array([[1, 0]], dtype=np.float32)
    sel = B.block_sparse_select(q, keys, 15, 4, 3, 1, 1)
    assert sel[0] == [0, 1, 3]
