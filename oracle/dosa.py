"""Oracle for DoSA safe-upper-bound pruning (fp64), step by step.

Test infrastructure only (see the package docstring).

Source: "DoSA：用安全上界减少 Indexer 的完整打分".
  section 2 step 1   seed threshold tau = K-th best fully scored seed; the seed
                     top-K is kept; tau is fixed for the pass; the worked
                     example K=2, seeds 9, 6, 2 -> tau 6 (U=5 dropped, U=6 kept)
  section 2 step 2   U = computed retained contribution + upper bound of the
                     omitted positive-weight part - lower bound of the omitted
                     negative-weight deduction; drop only if U < tau
  section 2 step 3   survivors are scored with every head, those below tau are
                     dropped, the rest merged with the seed top-K and the final
                     K chosen by the full score
  section 3.1        q_h = beta_h q_j + d_h, beta_h >= 0, and
                     [q_h.k]_+ <= beta_h [q_j.k]_+ + ||d_h|| ||k||
  section 3.2        a_A = sum_{h in A} |w_h| q_h,
                     [a_A.k]_+ <= sum_{h in N} |w_h| [q_h.k]_+ ; A = omitted
                     negative heads active on at least half of the seed samples
  section 4          the cold seed rule (four evenly spaced representative
                     queries, occurrence counts of their top-2048, 12,288
                     seeds), 128 sampled seed positions for the statistics
  section 5          the teaching estimate 100 x 32 = 3,200 versus
                     100 x 16 + 5 x 32 = 1,760 dot products

Readings where the page leaves a step open (parity unpinned against the
paper's own planner, whose rules are not on the page):
  * retained heads: the R heads with the largest |w_h| * ||q_h||, ties to the
    lower head index;
  * anchor of an omitted positive head: the retained head j minimising
    ||q_h - beta q_j|| with beta = max(0, q_h.q_j / ||q_j||^2), ties to the
    lower j (reproduces the section 3.1 example beta = 2, d = (0, 1));
  * "active" means q_h.k > 0; A holds the omitted negative heads active on at
    least half of the samples; the samples are seed[floor(i n_seed / 128)];
  * omitted heads with w_h = 0 contribute nothing and are ignored;
  * cold seed rule: representatives m_i = floor(i (M-1) / 3), i = 0..3, scored
    over the common visible prefix; a key ranks by (number of representative
    top-K lists holding it desc, best representative score desc, id asc); the
    first n_seed keys are the seeds;
  * decode seed rule (no rule on the page): floor(i L / n_seed), i < n_seed.
The output of the whole pass equals the exact top-K of oracle.dsa; that
equality, the bound's validity and the worked examples are what is pinned.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import dsa


# ---------------------------------------------------------------- section 2 --

def seed_threshold(seed_scores, K: int, seed_ids=None) -> float:
    """tau = the K-th best seed score under (score desc, id asc)."""
    ids, sc = dsa.topk(np.asarray(seed_scores, dtype=np.float64), K, seed_ids)
    if ids[K - 1] < 0:
        raise ValueError("fewer than K seeds")
    return float(sc[K - 1])


def keep_key(U: float, tau: float) -> bool:
    """Drop only when U < tau; U == tau is kept."""
    return not (U < tau)


def total_upper_bound(retained: float, positive_upper: float, negative_lower: float) -> float:
    """U = retained contribution + positive-part upper bound - negative lower bound."""
    return retained + positive_upper - negative_lower


# -------------------------------------------------------------- section 3.1 --

def anchor_coefficient(q_h, q_j) -> float:
    """beta = max(0, q_h.q_j / ||q_j||^2) (0 for a zero anchor)."""
    q_h = np.asarray(q_h, dtype=np.float64)
    q_j = np.asarray(q_j, dtype=np.float64)
    nn = float(q_j @ q_j)
    if nn == 0.0:
        return 0.0
    return max(0.0, float(q_h @ q_j) / nn)


def anchor_bound(q_h, q_j, k, beta=None) -> float:
    """beta [q_j.k]_+ + ||d|| ||k|| with d = q_h - beta q_j: upper bound of [q_h.k]_+."""
    q_h = np.asarray(q_h, dtype=np.float64)
    q_j = np.asarray(q_j, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    beta = anchor_coefficient(q_h, q_j) if beta is None else beta
    d = q_h - beta * q_j
    return beta * max(float(q_j @ k), 0.0) + float(np.linalg.norm(d)) * float(np.linalg.norm(k))


# -------------------------------------------------------------- section 3.2 --

def aggregate_query(q_heads, w_heads) -> np.ndarray:
    """a_A = sum_{h in A} |w_h| q_h."""
    q = np.asarray(q_heads, dtype=np.float64)
    w = np.abs(np.asarray(w_heads, dtype=np.float64))
    if q.shape[0] == 0:
        return np.zeros(q.shape[1] if q.ndim == 2 else 0)
    return (w[:, None] * q).sum(axis=0)


def aggregate_deduction(a_A, k) -> float:
    """L_N(k) = [a_A.k]_+."""
    return max(float(np.asarray(a_A, dtype=np.float64) @ np.asarray(k, dtype=np.float64)), 0.0)


def true_deduction(q_heads, w_heads, k) -> float:
    """sum_h |w_h| [q_h.k]_+ over the given negative heads."""
    q = np.asarray(q_heads, dtype=np.float64)
    w = np.abs(np.asarray(w_heads, dtype=np.float64))
    return float((w * np.maximum(q @ np.asarray(k, dtype=np.float64), 0.0)).sum())


# ------------------------------------------------------------------ planning --

@dataclass
class Plan:
    w: np.ndarray             # [H] the query's head weights
    retained: np.ndarray      # [R] head ids, ascending
    pos_heads: np.ndarray     # omitted heads with w > 0
    anchors: np.ndarray       # anchor head id per pos_head
    beta: np.ndarray          # per pos_head
    d_norm: np.ndarray        # ||q_h - beta q_anchor|| per pos_head
    agg_heads: np.ndarray     # A
    a_A: np.ndarray           # [D]
    w_fold: np.ndarray        # [R] folded retained weights
    c: float                  # sum_{h in P} w_h ||d_h||


def choose_retained(q_m, w_m, R: int) -> np.ndarray:
    q = np.asarray(q_m, dtype=np.float64)
    w = np.asarray(w_m, dtype=np.float64)
    H = q.shape[0]
    R = min(R, H)
    mag = np.abs(w) * np.linalg.norm(q, axis=1)
    order = np.lexsort((np.arange(H), -mag))
    return np.sort(order[:R])


def choose_anchor(q_h, q_m, retained):
    """(j, beta, ||q_h - beta q_j||) for the retained j with the smallest residual;
    among equal residuals the lowest j (the heads are visited in ascending order)."""
    best, best_j, best_beta = None, -1, 0.0
    for j in sorted(int(x) for x in retained):
        beta = anchor_coefficient(q_h, q_m[j])
        r = float(np.linalg.norm(np.asarray(q_h, np.float64) - beta * np.asarray(q_m[j], np.float64)))
        if best is None or r < best:
            best, best_j, best_beta = r, int(j), beta
    return best_j, best_beta, best


def sample_seeds(seed_ids, n_sample: int = 128):
    """seed[floor(i n / n_sample)], i < n_sample (all seeds when n <= n_sample)."""
    n = len(seed_ids)
    if n <= n_sample:
        return np.asarray(seed_ids)
    return np.asarray([seed_ids[(i * n) // n_sample] for i in range(n_sample)])


def plan_query(q_m, w_m, sample_keys, R: int, act_min: float = 0.5, retained=None) -> Plan:
    """Retained heads, anchors, folded weights, c and the negative aggregate."""
    q = np.asarray(q_m, dtype=np.float64)
    w = np.asarray(w_m, dtype=np.float64)
    H = q.shape[0]
    retained = choose_retained(q, w, R) if retained is None else np.sort(np.asarray(retained))
    rset = set(int(j) for j in retained)
    omitted = [h for h in range(H) if h not in rset]
    pos = [h for h in omitted if w[h] > 0]
    neg = [h for h in omitted if w[h] < 0]
    anchors, betas, dn = [], [], []
    for h in pos:
        j, beta, r = choose_anchor(q[h], q, retained)
        anchors.append(j)
        betas.append(beta)
        dn.append(r)
    sk = np.asarray(sample_keys, dtype=np.float64)
    agg = []
    if sk.shape[0] > 0:
        for h in neg:
            active = int((sk @ q[h] > 0).sum())
            if active >= act_min * sk.shape[0]:
                agg.append(h)
    a_A = aggregate_query(q[agg], w[agg]) if agg else np.zeros(q.shape[1])
    w_fold = np.array([w[j] for j in retained], dtype=np.float64)
    pos_of = {int(j): i for i, j in enumerate(retained)}
    for h, j, beta in zip(pos, anchors, betas):
        w_fold[pos_of[j]] += w[h] * beta
    c = float(sum(w[h] * r for h, r in zip(pos, dn)))
    return Plan(w, np.asarray(retained), np.asarray(pos, dtype=np.int64),
                np.asarray(anchors, dtype=np.int64), np.asarray(betas),
                np.asarray(dn), np.asarray(agg, dtype=np.int64), a_A, w_fold, c)


def upper_bound(plan: Plan, q_m, keys) -> np.ndarray:
    """U(k) for every key row, term by term as on the page: the retained heads'
    real contribution + sum_{h in P} w_h (beta_h [q_a(h).k]_+ + ||d_h|| ||k||)
    - [a_A.k]_+ ."""
    q = np.asarray(q_m, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    act = np.maximum(keys @ q[plan.retained].T, 0.0)             # [n, R]
    knorm = np.linalg.norm(keys, axis=1)
    col = {int(j): i for i, j in enumerate(plan.retained)}
    U = act @ plan.w[plan.retained]
    for h, j, beta, r in zip(plan.pos_heads, plan.anchors, plan.beta, plan.d_norm):
        U = U + plan.w[int(h)] * (beta * act[:, col[int(j)]] + r * knorm)
    return U - np.maximum(keys @ plan.a_A, 0.0)


def upper_bound_folded(plan: Plan, q_m, keys) -> np.ndarray:
    """The same bound with the anchors folded into the retained weights:
    sum_j w'_j [q_j.k]_+ + c ||k|| - [a_A.k]_+ (equal to upper_bound in exact
    arithmetic; this is the form a kernel evaluates)."""
    q = np.asarray(q_m, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    act = np.maximum(keys @ q[plan.retained].T, 0.0)
    return act @ plan.w_fold + plan.c * np.linalg.norm(keys, axis=1) - np.maximum(keys @ plan.a_A, 0.0)


# --------------------------------------------------------------------- seeds --

def cold_seeds(problem, n_seed: int, K: int) -> np.ndarray:
    """Section 4 cold rule for a shared key sequence (prefill)."""
    M = problem.M
    reps = sorted(set((i * (M - 1)) // 3 for i in range(4)))
    common = int(np.min(problem.key_len))
    keys = dsa.dequantised_keys(problem, 0)[:common]
    count = np.zeros(common, dtype=np.int64)
    best = np.full(common, -np.inf)
    for m in reps:
        s, _ = dsa.indexer_score(problem.q_f32()[m], problem.w[m], keys)
        ids, _ = dsa.topk(s, K)
        count[ids[ids >= 0]] += 1
        best = np.maximum(best, s)
    order = np.lexsort((np.arange(common), -best, -count))
    return np.sort(order[:min(n_seed, common)])


def strided_seeds(L: int, n_seed: int) -> np.ndarray:
    """Decode rule: floor(i L / n), i < n = min(L, n_seed)."""
    n = min(L, n_seed)
    return np.asarray([(i * L) // n for i in range(n)], dtype=np.int64)


# ------------------------------------------------------------------ the pass --

@dataclass
class DosaRowResult:
    ids: np.ndarray
    scores: np.ndarray
    tau: float
    n_candidates: int
    n_survivors: int
    fell_back: bool


def dosa_topk_row(q_m, w_m, keys, seed_ids, K: int, R: int, n_sample: int = 128,
                  act_min: float = 0.5, retained=None) -> DosaRowResult:
    """One query, keys [L, D] fp64 with ids 0..L-1, in the page's order:
    seeds -> tau and seed top-K -> plan -> bound scan (drop iff U < tau) ->
    exact rescoring (drop s < tau) -> merge with the seed top-K -> top-K."""
    keys = np.asarray(keys, dtype=np.float64)
    L = keys.shape[0]
    seed_ids = np.unique(np.asarray(seed_ids, dtype=np.int64))
    seed_ids = seed_ids[(seed_ids >= 0) & (seed_ids < L)]
    if seed_ids.shape[0] < K:
        s, _ = dsa.indexer_score(q_m, w_m, keys)
        ids, sc = dsa.topk(s, K)
        return DosaRowResult(ids, sc, float("nan"), L, L, True)
    # The exact score of a key is a function of (q, w, k) alone; it is evaluated
    # once per key so that a seed, a survivor and the plain top-K all see the
    # same fp64 value whatever subset a matrix product was blocked over.
    s_all, _ = dsa.indexer_score(q_m, w_m, keys)
    s_seed = s_all[seed_ids]
    seed_top_ids, seed_top_s = dsa.topk(s_seed, K, seed_ids)
    tau = float(seed_top_s[K - 1])
    plan = plan_query(q_m, w_m, keys[sample_seeds(seed_ids, n_sample)], R, act_min, retained)
    is_seed = np.zeros(L, dtype=bool)
    is_seed[seed_ids] = True
    rest = np.nonzero(~is_seed)[0]
    U = upper_bound(plan, q_m, keys[rest])
    cand = rest[np.array([keep_key(u, tau) for u in U], dtype=bool)] if rest.size else rest
    s_c = s_all[cand]
    surv = s_c >= tau
    ids = np.concatenate([seed_top_ids, cand[surv]])
    sc = np.concatenate([seed_top_s, s_c[surv]])
    out_ids, out_s = dsa.topk(sc, K, ids)
    return DosaRowResult(out_ids, out_s, tau, int(cand.size), int(surv.sum()), False)


def teaching_dot_count(n_keys: int, H: int, scan_dots: int, survivors: int):
    """Section 5 estimate: (full count, pruned count) of dot products."""
    return n_keys * H, n_keys * scan_dots + survivors * H
