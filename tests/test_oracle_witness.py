"""Pins of the witness oracle against the "Segment Witnesses" page: its printed
examples (tests/golden/witness_examples.json), the invariants it derives and
brute-force checks on random rows."""
import json
import os

import numpy as np
import pytest

from oracle import witness as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "witness_examples.json")))


def test_printed_witness_table():
    for c in GOLD["witness_indices"]:
        got = W.topology_witness_indices(c["learned"], len(c["learned"]), [c["L"]], c["S"])
        assert got[0].tolist() == c["expected"], c["cite"]


def test_printed_merges():
    for c in GOLD["merge"]:
        got = W.apply_topology_witnesses(c["learned"], len(c["learned"]), [c["L"]], c["keep"],
                                         c["S"], c["max_replacements"])[0].tolist()
        if "expected" in c:
            assert got == c["expected"], c["cite"]
        else:
            assert set(x for x in got if x >= 0) == set(c["expected_set"]), c["cite"]


def test_coverage_counterexample_and_serving_form():
    for c in GOLD["serving"]:
        buf = np.array(c["learned"], dtype=np.int64)
        W.scatter_topology_witnesses(buf, len(buf), [c["L"]], c["S"])
        assert buf.tolist() == c["expected"], c["cite"]
        assert W.segment_coverage(buf, c["L"], c["S"]) == c["coverage"]


def test_segment_of_examples():
    for c in GOLD["segment_of"]:
        if "occupied_segment" in c:
            # an out-of-range entry marks min(floor(x S_eff / L), S - 1)
            wit = W.witness_row([c["x"]], c["L"], c["S"])
            s_eff = min(c["S"], c["L"])
            assert min((c["x"] * s_eff) // c["L"], c["S"] - 1) == c["occupied_segment"]
            # segment 7 is outside the partition, so every real segment still gets a witness
            assert wit[:s_eff] == [W.segment_edge(s, c["L"], s_eff) for s in range(s_eff)]
        else:
            assert W.segment_of(c["x"], c["L"], c["S"]) == c["segment"], c["cite"]
    # "rounding down does not round-trip": floor(1*10/4) = 2 lands in segment 0,
    # the ceiling e_1 = 3 lands in segment 1
    assert (1 * 10) // 4 == 2 and W.segment_of(2, 10, 4) == 0
    assert W.segment_edge(1, 10, 4) == 3 and W.segment_of(3, 10, 4) == 1


def test_coverage_examples():
    for c in GOLD["coverage"]:
        assert W.segment_coverage(c["candidates"], c["L"], c["S"]) == c["coverage"], c["cite"]
    assert W.segment_coverage([1, 2], 0, 4) == 1.0     # no segments -> 1
    assert W.segment_coverage([-1, 7, 7, 100], 8, 4) == 0.25  # padding / out of range count nothing


@pytest.mark.parametrize("L", list(range(1, 70)) + [100, 127, 128, 129, 1000, 4095, 65536, 131071])
def test_left_edge_lies_in_its_segment(L):
    for S in range(1, 65):
        s_eff = min(S, L)
        for s in range(s_eff):
            e = W.segment_edge(s, L, s_eff)
            assert 0 <= e < L
            assert W.segment_of(e, L, S) == s
            # brute force: e is the smallest x with sigma(x) == s
            assert e == 0 or W.segment_of(e - 1, L, S) == s - 1


def _brute_partition(L, S):
    s_eff = min(S, L)
    return [[x for x in range(L) if (x * s_eff) // L == s] for s in range(s_eff)]


def test_partition_is_consecutive_intervals_bruteforce():
    for L in range(1, 60):
        for S in range(1, 20):
            parts = _brute_partition(L, S)
            s_eff = min(S, L)
            for s, p in enumerate(parts):
                lo = W.segment_edge(s, L, s_eff)
                hi = W.segment_edge(s + 1, L, s_eff) if s + 1 < s_eff else L
                assert p == list(range(lo, hi))


def test_random_rows_disjoint_distinct_complete_and_run_bound():
    rng = np.random.default_rng(11)
    for _ in range(300):
        L = int(rng.integers(1, 400))
        S = int(rng.integers(1, 65))
        n = int(rng.integers(0, min(L, 40) + 1))
        K = rng.choice(L, size=n, replace=False).tolist()
        wit = [x for x in W.witness_row(K, L, S) if x >= 0]
        assert not (set(wit) & set(K))                      # (1) disjoint
        assert len(set(wit)) == len(wit)                    # (2) distinct
        s_eff = min(S, L)
        segs = {W.segment_of(x, L, S) for x in K + wit}
        assert segs == set(range(s_eff))                    # (3) complete
        assert wit == sorted(wit)                           # ascending segment order
        # longest run of unselected tokens
        sel = sorted(set(K + wit))
        gaps = [sel[0]] + [b - a - 1 for a, b in zip(sel, sel[1:])] + [L - 1 - sel[-1]]
        assert max(gaps) <= W.uncovered_run_bound(L, S)


def test_serving_rows_prefix_budget_and_single_run():
    rng = np.random.default_rng(12)
    for _ in range(200):
        L = int(rng.integers(1, 3000))
        S = int(rng.integers(1, 65))
        topk = int(rng.integers(1, 200))
        row = np.full(topk, -1, dtype=np.int64)
        n = min(topk, L)
        row[:n] = rng.choice(L, size=n, replace=False)
        row[rng.random(topk) < 0.2] = -1
        out = row.copy()
        W.scatter_topology_witnesses(out, topk, [L], S)
        keep = max(topk - S, 0)
        B = min(S, topk - keep)
        assert (out[:keep] == row[:keep]).all()
        changed = np.nonzero(out != row)[0]
        assert all(keep <= i < keep + B for i in changed)
        wit = [x for x in W.witness_row(row, L, S) if x >= 0][:B]
        assert out[keep:keep + len(wit)].tolist() == wit
        vals = [x for x in out if x >= 0]
        assert len(vals) == len(set(vals))


def test_padded_tail_gives_full_coverage():
    rng = np.random.default_rng(13)
    for _ in range(200):
        L = int(rng.integers(1, 3000))
        S = int(rng.integers(1, 65))
        topk = int(rng.integers(S, S + 200))
        keep = topk - S
        row = np.full(topk, -1, dtype=np.int64)
        n = min(keep, L)
        row[:n] = rng.choice(L, size=n, replace=False)
        W.scatter_topology_witnesses(row, topk, [L], S)
        assert W.segment_coverage(row, L, S) == 1.0


def test_witness_set_is_permutation_invariant():
    rng = np.random.default_rng(14)
    for _ in range(100):
        L = int(rng.integers(1, 500))
        S = int(rng.integers(1, 65))
        K = rng.choice(L, size=min(L, 20), replace=False)
        a = W.witness_row(K.tolist(), L, S)
        b = W.witness_row(rng.permutation(K).tolist(), L, S)
        assert a == b


def test_disabled_and_zero_budget_are_identity_and_short_rows():
    learned = [0, 5, 9, -1]
    assert W.apply_topology_witnesses(learned, 4, [16], 2, 0, 2)[0].tolist() == learned
    assert W.apply_topology_witnesses(learned, 4, [16], 4, 4, 2)[0].tolist() == learned  # B = 0
    assert W.apply_topology_witnesses(learned, 4, [16], 2, 4, 0)[0].tolist() == learned
    for L in (0, -3):
        assert W.apply_topology_witnesses([-1] * 4, 4, [L], 0, 4, 4)[0].tolist() == [-1] * 4
    # L < S: every token the row does not hold becomes a witness
    assert W.witness_row([1], 3, 8)[:3] == [0, -1, 2]


def test_refusals_leave_the_buffer_untouched():
    buf = np.array([0, 5, 9, -1], dtype=np.int64)
    for args, kind in [((4, [16], 65), "segments_out_of_range"),
                       ((4, [], 4), "rows_mismatch"),
                       ((3, [16, 16], 4), "rows_mismatch")]:
        with pytest.raises(W.WitnessError) as e:
            W.scatter_topology_witnesses(buf, *args)
        assert e.value.kind == kind
        assert buf.tolist() == [0, 5, 9, -1]
    with pytest.raises(W.WitnessError) as e:
        W.apply_topology_witnesses(buf, 4, [16], 5, 4, 4)
    assert e.value.kind == "keep_out_of_range"
    with pytest.raises(W.WitnessError) as e:
        W.topology_witness_indices(buf, 4, [16], 0)
    assert e.value.kind == "segments_out_of_range"


def test_a_planted_mistake_is_caught():
    """Floor instead of ceiling for e_s (the page's own warning) must break the
    left-edge invariant for L=10, S=4."""
    floor_edge = (1 * 10) // 4
    assert W.segment_of(floor_edge, 10, 4) != 1
    assert W.segment_of(W.segment_edge(1, 10, 4), 10, 4) == 1
