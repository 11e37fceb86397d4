"""Oracle for MiniMax-M3 block-sparse selection (fp32, the page's dot order).

Test infrastructure only (see the package docstring).

Source: "ferrox_core/block_sparse.rs" page -- module docs (block score is the
MAX over the block's positions, raw dot with no softmax scale, selection per KV
head, forced init/local blocks), BlockSparseConfig and its defaults,
causal_blocks, block_sparse_select (n_blocks clipped to the keys that exist),
select_for_head (forced blocks, budget = max(top, #forced), early return,
(score desc, block asc) order, ascending output), dot (products summed in
sequence in f32) and positions_of_blocks.

Readings where the page leaves a step open:
  * -0.0 is replaced by +0.0 in every dot result, so the total order that puts
    -0.0 below +0.0 never has to decide between them (Rust leaves the sign of
    max(-0.0, +0.0) unspecified);
  * inputs are finite.
"""
from __future__ import annotations

import numpy as np

MINIMAX_BLOCK_SIZE = 128


def causal_blocks(block_size: int, query_pos: int) -> int:
    """Blocks covering 0..=query_pos; 0 when the block size is 0."""
    if block_size == 0:
        return 0
    return query_pos // block_size + 1


def dot_f32(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """Sequential f32 dot of q [D] with each row of k [P, D]: acc starts at 0,
    then acc = acc + q[d]*k[d] for d = 0..D-1, every product and sum rounded to
    f32 on its own (no fused multiply-add)."""
    q = np.asarray(q, dtype=np.float32)
    k = np.asarray(k, dtype=np.float32)
    acc = np.zeros(k.shape[0], dtype=np.float32)
    for d in range(q.shape[0]):
        prod = np.multiply(k[:, d], q[d], dtype=np.float32)
        acc = np.add(acc, prod, dtype=np.float32)
    return acc + np.float32(0.0)   # -0.0 -> +0.0


def _total_key(x: np.float32) -> int:
    """Rust's f32::total_cmp as an integer key (larger key = larger value)."""
    b = int(np.float32(x).view(np.uint32))
    if b & 0x80000000:
        return (~b) & 0xFFFFFFFF
    return b | 0x80000000


def n_blocks_visible(L: int, block_size: int, query_pos: int) -> int:
    if block_size == 0:
        return 0
    return min(causal_blocks(block_size, query_pos), -(-L // block_size))


def select_for_head(q, index_k, query_pos: int, n_blocks: int, block_size: int,
                    top_blocks: int, init_blocks: int, local_blocks: int):
    forced = [False] * n_blocks
    for b in range(min(init_blocks, n_blocks)):
        forced[b] = True
    for b in range(max(n_blocks - local_blocks, 0), n_blocks):
        forced[b] = True
    n_forced = sum(forced)
    budget = max(top_blocks, n_forced)
    chosen = [b for b in range(n_blocks) if forced[b]]
    if len(chosen) >= budget or len(chosen) == n_blocks:
        return sorted(chosen)
    L = index_k.shape[0]
    scored = []
    for b in range(n_blocks):
        if forced[b]:
            continue
        start = b * block_size
        end = min((b + 1) * block_size, L, query_pos + 1)
        best = np.float32(-np.inf)
        if end > start:
            best = np.max(dot_f32(q, index_k[start:end]))
        scored.append((b, np.float32(best)))
    scored.sort(key=lambda t: (-_total_key(t[1]), t[0]))
    for b, _ in scored[:budget - len(chosen)]:
        chosen.append(b)
    return sorted(chosen)


def block_sparse_select(index_q, index_k, query_pos: int, block_size: int, top_blocks: int,
                        init_blocks: int, local_blocks: int):
    """One ascending block list per KV head for one query position."""
    index_k = np.asarray(index_k, dtype=np.float32)
    n_blocks = n_blocks_visible(index_k.shape[0], block_size, query_pos)
    if n_blocks == 0:
        return [[] for _ in range(len(index_q))]
    return [select_for_head(q, index_k, query_pos, n_blocks, block_size, top_blocks,
                            init_blocks, local_blocks) for q in index_q]


def block_scores(q, index_k, query_pos: int, block_size: int):
    """Block score (max of the raw dot over causally visible positions) of every
    visible block, as f32; used by tests to find near-ties."""
    index_k = np.asarray(index_k, dtype=np.float32)
    n_blocks = n_blocks_visible(index_k.shape[0], block_size, query_pos)
    L = index_k.shape[0]
    end_all = min(L, query_pos + 1)
    d = dot_f32(q, index_k[:end_all])
    out = np.full(n_blocks, -np.inf, dtype=np.float32)
    for b in range(n_blocks):
        s, e = b * block_size, min((b + 1) * block_size, end_all)
        if e > s:
            out[b] = d[s:e].max()
    return out


def select_problem(problem, queries=None):
    """Selections for (a subset of) the queries of a BlockSelectProblem:
    dict query -> list over heads of ascending block lists."""
    queries = range(problem.index_q.shape[0]) if queries is None else queries
    res = {}
    for i in queries:
        res[int(i)] = block_sparse_select(problem.index_q[i], problem.index_k,
                                          int(problem.query_pos[i]), problem.block_size,
                                          problem.top_blocks, problem.init_blocks,
                                          problem.local_blocks)
    return res


def positions_of_blocks(blocks, query_pos: int, n_positions: int, block_size: int):
    """Blocks -> covered positions, ascending, deduplicated, causally clipped."""
    out = set()
    for b in blocks:
        start = b * block_size
        end = min((b + 1) * block_size, n_positions, query_pos + 1)
        out.update(range(start, end))
    return sorted(out)
