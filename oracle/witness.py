"""Oracle for the segment-witness covering pass (integers, exact).

Test infrastructure only (see the package docstring).

Source: "Segment Witnesses" page -- sections "Object" (S_eff, e_s, sigma,
O(K), W(K)), "Invariant and consequences", "Implementation rule and contracts"
(slots, budget B, padding, fallback, out-of-range entries), "Refusals" and
"Rust API" (segment_of's zero-length rule, coverage returning 1 with no
segments).

Readings where the page leaves a step open:
  * any negative entry is padding (the page names -1);
  * budget slots that receive no witness keep their input value;
  * the S = 0 off switch is checked before the segment-range refusal at the
    merge; witness_indices (no off switch) refuses S = 0;
  * context lengths shorter than the row count are a rows mismatch.
"""
from __future__ import annotations

import numpy as np

MAX_TOPOLOGY_SEGMENTS = 64


class WitnessError(Exception):
    """Refusal; `kind` is one of rows_mismatch / segments_out_of_range /
    keep_out_of_range (the page's three WitnessError variants)."""

    def __init__(self, kind: str):
        super().__init__(kind)
        self.kind = kind


def segment_of(x: int, L: int, S: int) -> int:
    """sigma(x) = floor(x * S_eff / L), S_eff = min(S, L); a length of 0 reads as 1."""
    L = max(int(L), 1)
    s_eff = min(int(S), L)
    return (int(x) * s_eff) // L


def segment_edge(s: int, L: int, s_eff: int) -> int:
    """e_s = ceil(s * L / S_eff)."""
    return -((-int(s) * int(L)) // int(s_eff))


def _occupied(row, L: int, S: int) -> set:
    """O(K): segments hit by valid learned entries; an entry x >= L marks
    min(floor(x S_eff / L), S - 1) (out-of-range contract)."""
    s_eff = min(S, L)
    occ = set()
    for x in row:
        x = int(x)
        if x < 0:
            continue
        occ.add(min((x * s_eff) // L, S - 1))
    return occ


def witness_row(row, L: int, S: int) -> list:
    """W(K) in ascending segment order, as a list of length S with -1 where
    segment s is occupied or s >= S_eff.  Rows with L <= 0 get no witnesses."""
    out = [-1] * S
    if L <= 0 or S <= 0:
        return out
    s_eff = min(S, L)
    occ = _occupied(row, L, S)
    for s in range(s_eff):
        if s not in occ:
            out[s] = segment_edge(s, L, s_eff)
    return out


def _check_rows(learned, topk: int, context_lens):
    learned = np.asarray(learned, dtype=np.int64).reshape(-1)
    if topk <= 0:
        rows = 0
        if learned.size != 0:
            raise WitnessError("rows_mismatch")
    else:
        if learned.size % topk != 0:
            raise WitnessError("rows_mismatch")
        rows = learned.size // topk
    if len(context_lens) < rows:
        raise WitnessError("rows_mismatch")
    return learned, rows


def topology_witness_indices(learned, topk: int, context_lens, num_segments: int) -> np.ndarray:
    """Row-major [rows, S] witness table (the page's topology_witness_indices)."""
    if num_segments == 0 or num_segments > MAX_TOPOLOGY_SEGMENTS:
        raise WitnessError("segments_out_of_range")
    learned, rows = _check_rows(learned, topk, context_lens)
    out = np.full((rows, num_segments), -1, dtype=np.int64)
    for r in range(rows):
        out[r] = witness_row(learned[r * topk:(r + 1) * topk], int(context_lens[r]), num_segments)
    return out


def apply_topology_witnesses(learned, topk: int, context_lens, keep: int, num_segments: int,
                             max_replacements: int) -> np.ndarray:
    """Merge rule: slots [0, keep) verbatim; witnesses in ascending segment order
    overwrite slots keep, keep+1, ... up to B = min(max_replacements, topk - keep);
    witnesses beyond B are dropped.  Returns a new [rows, topk] array."""
    learned = np.asarray(learned, dtype=np.int64).reshape(-1)
    if num_segments == 0:
        return learned.reshape(-1, max(topk, 1)).copy() if topk > 0 else learned.copy()
    if num_segments > MAX_TOPOLOGY_SEGMENTS:
        raise WitnessError("segments_out_of_range")
    if keep > topk:
        raise WitnessError("keep_out_of_range")
    learned, rows = _check_rows(learned, topk, context_lens)
    out = learned.reshape(rows, topk).copy() if topk > 0 else learned.copy()
    B = min(max_replacements, topk - keep)
    if B <= 0 or rows == 0:
        return out
    for r in range(rows):
        wit = [x for x in witness_row(out[r], int(context_lens[r]), num_segments) if x >= 0]
        for i, x in enumerate(wit[:B]):
            out[r, keep + i] = x
    return out


def scatter_topology_witnesses(topk_indices: np.ndarray, topk: int, context_lens,
                               num_segments: int) -> None:
    """Serving entry point, in place: keep = topk - S (saturating), B = S.
    A refused call leaves the buffer untouched."""
    keep = max(topk - num_segments, 0)
    res = apply_topology_witnesses(topk_indices, topk, context_lens, keep, num_segments,
                                   num_segments)
    topk_indices.reshape(-1)[:] = res.reshape(-1)


def segment_coverage(candidates, L: int, S: int) -> float:
    """|{sigma(x) : x in C, 0 <= x < L}| / S_eff; 1 when there are no segments."""
    s_eff = min(S, max(L, 0))
    if s_eff <= 0:
        return 1.0
    segs = {segment_of(x, L, S) for x in candidates if 0 <= int(x) < L}
    return len(segs) / s_eff


def uncovered_run_bound(L: int, S: int) -> int:
    """2 * ceil(L / S_eff) - 2, the longest run of unselected tokens once every
    segment holds a selected token ("Invariant and consequences")."""
    s_eff = min(S, L)
    return 2 * (-(-L // s_eff)) - 2
