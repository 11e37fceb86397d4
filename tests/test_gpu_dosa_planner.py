"""The GPU's DoSA planner and cold seed rule held to the oracle's readings.

dosa_topk leaves its intermediate results in the workspace
(dosa_workspace_layout): the cold rule's per-key representative counts and
scores and the seed list, and per (row, head) the planner's decisions.  These
tests compare them with oracle.dosa ("DoSA：用安全上界减少 Indexer 的完整打分",
section 3.1 anchors and residual norms, section 3.2 the aggregate set A,
section 4 the cold rule and the planner step):

  * cold rule: the GPU's representative scores within the score tolerance of
    the oracle's; each key's count within the interval the tolerance allows
    (a key within tolerance of a representative's K-th score may go either
    way); the seed list exactly the first n_seed keys under (count desc, best
    score desc, id asc) of the GPU's own counts and scores; and every key the
    oracle's cold_seeds certainly keeps (or certainly drops) kept (dropped);
  * planner: the retained set equals oracle.dosa.choose_retained except at
    near-ties of |w| ||q||; with the GPU's retained set, each omitted positive
    head's anchor equals oracle.dosa.choose_anchor's except at near-ties of
    the residual, beta and ||d_h|| within fp32 rounding of the exact values for
    that anchor, A equals the oracle's set except for heads whose activation
    count is within rounding of the threshold, and the folded weights, the
    aggregate (bf16) and c + margin agree with values computed in fp64 from
    the GPU's decisions.
"""
import numpy as np
import pytest
import torch

from helpers import EPS
from oracle import dosa as odosa
from oracle import dsa as odsa
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GAMMA = 2.0 ** -10


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _run(B, wp, n_seed, R, cap=4096):
    p = B.problem_to_device(wp)
    dp = B.make_dosa_params(n_seed=n_seed, retained_heads=R, candidate_capacity=cap)
    K, M = wp.K, wp.M
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.zeros(B.dosa_topk_workspace_size(p, K, dp, 0), dtype=torch.uint8, device="cuda")
    B.dosa_topk(p, K, dp, ids, sc, ws)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    lay = B.dosa_workspace_layout(p, K, dp, 0)
    return ws.cpu().numpy(), lay


def _arr(wsh, off, dtype, count):
    n = np.dtype(dtype).itemsize * count
    return wsh[off:off + n].view(dtype)


def _keys_f64(wp, off, ids):
    """Keys (dequantised) of row-relative ids at key offset off."""
    rows = off + np.asarray(ids, dtype=np.int64)
    if wp.dtype == "bf16":
        return wl.bf16_bits_to_f32(wp.keys[rows]).astype(np.float64)
    if wp.dtype == "fp8":
        return wl.e4m3_bits_to_f32(wp.keys[rows]).astype(np.float64) * wp.key_scale[rows].astype(np.float64)[:, None]
    return wp.keys[rows].astype(np.float64)


# ----------------------------------------------------------------- cold rule --

def _check_cold_rule(wp, wsh, lay, n_seed):
    M, K = wp.M, wp.K
    eps = EPS[wp.dtype]
    reps = sorted(set((i * (M - 1)) // 3 for i in range(4)))
    common = int(np.min(wp.key_len))
    rep_ld = lay["rep_ld"]
    g_rsc = _arr(wsh, lay["rep_scores"], np.float32, len(reps) * rep_ld).reshape(len(reps), rep_ld)[:, :common]
    g_cnt = _arr(wsh, lay["rep_count"], np.uint32, rep_ld)[:common].astype(np.int64)
    n_list = int(_arr(wsh, lay["seed_count"], np.int32, 1)[0])
    g_list = _arr(wsh, lay["seed_list"], np.int32, lay["seed_ld"])[:n_list].astype(np.int64)
    keys = odsa.dequantised_keys(wp, 0)[:common]
    cnt_lo = np.zeros(common, np.int64)
    cnt_hi = np.zeros(common, np.int64)
    best = np.full(common, -np.inf)
    best_tol = np.zeros(common)
    for i, m in enumerate(reps):
        s, a = odsa.indexer_score(wp.q_f32()[m], wp.w[m], keys)
        err = np.abs(g_rsc[i].astype(np.float64) - s)
        assert (err <= eps * (a + 1e-30)).all(), f"representative {m}: score out of tolerance"
        if common <= K:
            cnt_lo += 1
            cnt_hi += 1
        else:
            kth = odsa.topk_order(s)[K - 1]
            tol = eps * (a + a[kth])
            cnt_lo += s > s[kth] + tol
            cnt_hi += s >= s[kth] - tol
        upd = s > best
        best = np.where(upd, s, best)
        best_tol = np.maximum(best_tol, eps * a)
    bad = np.nonzero((g_cnt < cnt_lo) | (g_cnt > cnt_hi))[0]
    assert bad.size == 0, f"{bad.size} representative counts outside their interval, e.g. key {bad[:5]}"
    # the selection on the GPU's own counts and scores, exactly
    g_best = (g_rsc.max(axis=0) + np.float32(0.0)).astype(np.float64)
    order = np.lexsort((np.arange(common), -g_best, -g_cnt))
    want = np.sort(order[:min(n_seed, common)])
    assert n_list == want.size and np.array_equal(g_list, want)
    # against oracle.cold_seeds: keys it certainly keeps / drops under the tolerance
    o_seeds = set(odosa.cold_seeds(wp, n_seed, K).tolist())
    span = 4.0 * (np.max(np.abs(best)) + np.max(best_tol) + 1.0)
    lo = cnt_lo * span + (best - best_tol)      # the weakest rank key a key can have
    hi = cnt_hi * span + (best + best_tol)      # the strongest
    hs, ls = np.sort(hi), np.sort(lo)
    could_beat = common - np.searchsorted(hs, lo, side="left") - 1     # others with hi >= my lo
    surely_beat = common - np.searchsorted(ls, hi, side="right")       # others with lo > my hi
    g_set = set(g_list.tolist())
    n_in = min(n_seed, common)
    for x in range(common):
        if could_beat[x] < n_in:
            assert x in g_set and x in o_seeds, f"key {x} certainly a seed"
        if surely_beat[x] >= n_in:
            assert x not in g_set and x not in o_seeds, f"key {x} certainly not a seed"
    return g_list


# ------------------------------------------------------------------- planner --

def _check_planner(wp, wsh, lay, R, seed_lists, n_sample=128, act_min=0.5):
    M, H, D = wp.M, wp.H, wp.D
    q_all = wp.q_f32().astype(np.float64)
    status = _arr(wsh, lay["status"], np.int32, M)
    ph_all = _arr(wsh, lay["plan_head"], np.int32, M * H).reshape(M, H)
    pb_all = _arr(wsh, lay["plan_beta"], np.float32, M * H).reshape(M, H).astype(np.float64)
    pd_all = _arr(wsh, lay["plan_dnorm"], np.float32, M * H).reshape(M, H).astype(np.float64)
    wf_all = _arr(wsh, lay["wfold"], np.float32, M * 32).reshape(M, 32).astype(np.float64)
    coef = _arr(wsh, lay["coef"], np.float32, M).astype(np.float64)
    qprep = _arr(wsh, lay["qprep"], np.uint16, (((M + 7) // 8) * 144 if lay["group_layout"] else M * 32) * D)
    qprep = qprep.reshape(-1, D)
    checked = {"rows": 0, "anchored": 0, "agg": 0}
    for m in range(M):
        if status[m] & 1:
            continue
        q = q_all[m]
        w = wp.w[m].astype(np.float64)
        ph, pb, pd = ph_all[m], pb_all[m], pd_all[m]
        # retained heads
        is_ret = (ph >= 0) & (ph < 1024)
        pos = ph[is_ret]
        rlist = np.argsort(np.where(is_ret, ph, 1 << 20), kind="stable")[:pos.size]
        assert sorted(pos.tolist()) == list(range(min(R, H))), f"row {m}: retained positions"
        assert np.all(np.diff(rlist) > 0), f"row {m}: retained heads not ascending"
        mag = np.abs(w) * np.linalg.norm(q, axis=1)
        o_ret = set(odosa.choose_retained(q, w, R).tolist())
        cut = np.sort(mag)[::-1][min(R, H) - 1]
        for h in o_ret ^ set(rlist.tolist()):
            assert abs(mag[h] - cut) <= 1e-5 * cut, f"row {m}: head {h} retained differently, not a near-tie"
        # the plan for the GPU's retained set and samples
        sl = seed_lists[0] if len(seed_lists) == 1 else seed_lists[m]
        samp = odosa.sample_seeds(sl, n_sample)
        off = wp.row_offset(m)
        sk = _keys_f64(wp, off, samp)
        plan = odosa.plan_query(q, w, sk, R, act_min, retained=rlist)
        anch = {int(h): int(j) for h, j in zip(plan.pos_heads, plan.anchors)}
        rset = set(rlist.tolist())
        for h in range(H):
            if h in rset:
                continue
            if w[h] > 0:
                assert ph[h] >= 1024, f"row {m}: positive head {h} not anchored"
                jg = int(ph[h]) - 1024
                assert jg in rset
                if jg != anch[h]:
                    rg = odosa.choose_anchor(q[h], q, [jg])[2]
                    ro = odosa.choose_anchor(q[h], q, [anch[h]])[2]
                    assert rg <= ro * (1 + 1e-4) + 1e-6 * np.linalg.norm(q[h]), f"row {m} head {h}: anchor"
                b_ex = odosa.anchor_coefficient(q[h], q[jg])
                assert abs(pb[h] - b_ex) <= 1e-5 * b_ex + 1e-7 * np.linalg.norm(q[h]) / max(np.linalg.norm(q[jg]), 1e-30)
                r_ex = float(np.linalg.norm(q[h] - pb[h] * q[jg]))
                nh = float(np.linalg.norm(q[h]))
                assert pd[h] >= r_ex - 1e-6 * nh and pd[h] <= r_ex * (1 + 1e-5) + 1e-6 * nh, \
                    f"row {m} head {h}: ||d|| {pd[h]} vs {r_ex}"
                checked["anchored"] += 1
            elif w[h] < 0:
                dots = sk @ q[h]
                tol = 1e-5 * np.linalg.norm(q[h]) * np.linalg.norm(sk, axis=1)
                need = act_min * len(samp)
                lo, hi = int((dots > tol).sum()), int((dots > -tol).sum())
                in_g = ph[h] == -2
                if lo >= need:
                    assert in_g, f"row {m}: head {h} belongs to A"
                if hi < need:
                    assert not in_g, f"row {m}: head {h} does not belong to A"
                checked["agg"] += int(in_g)
            else:
                assert ph[h] == -1
        # folded weights from the GPU's decisions
        wf = np.zeros(32)
        mag_wf = np.zeros(32)
        for r, j in enumerate(rlist):
            wf[r] = w[j]
            mag_wf[r] = abs(w[j])
        for h in range(H):
            if ph[h] >= 1024:
                r = int(np.nonzero(rlist == ph[h] - 1024)[0][0])
                wf[r] += w[h] * pb[h]
                mag_wf[r] += abs(w[h] * pb[h])
        assert np.all(np.abs(wf_all[m] - wf) <= 1e-5 * mag_wf + 1e-7), f"row {m}: folded weights"
        # aggregate (bf16 row) and prepared retained rows
        agg = [h for h in range(H) if ph[h] == -2]
        a = (np.abs(w[agg])[:, None] * q[agg]).sum(axis=0) if agg else np.zeros(D)
        if lay["group_layout"]:
            g, qi = m // 8, m % 8
            vec_row = lambda r: g * 144 + qi * 16 + r
            agg_row = g * 144 + 128 + qi
        else:
            vec_row = lambda r: m * 32 + r
            agg_row = m * 32 + 31
        a_g = wl.bf16_bits_to_f32(qprep[agg_row]).astype(np.float64)
        amag = (np.abs(w[agg])[:, None] * np.abs(q[agg])).sum(axis=0) if agg else np.zeros(D)
        assert np.all(np.abs(a_g - a) <= 2.0 ** -8 * np.abs(a) + 1e-6 * amag + 1e-30), f"row {m}: aggregate"
        for r, j in enumerate(rlist):
            assert np.array_equal(qprep[vec_row(r)], wp.q[m, j]), f"row {m}: prepared row {r}"
        # c + margin
        c = float(sum(w[h] * pd[h] for h in range(H) if ph[h] >= 1024))
        Wm = float(np.sum(np.abs(w) * np.linalg.norm(q, axis=1)))
        an = float(np.linalg.norm(a))
        lo_c = c + GAMMA * (Wm + an)
        assert coef[m] >= lo_c * (1 - 1e-4) - 1e-6, f"row {m}: coef {coef[m]} below c + gamma terms {lo_c}"
        if wp.dtype == "bf16":
            e = float(np.linalg.norm(a_g - a))
            hi_c = c + e * 1.01 + GAMMA * (Wm + 1.02 * an)
            assert coef[m] <= hi_c * (1 + 1e-4) + 1e-6, f"row {m}: coef {coef[m]} above {hi_c}"
        checked["rows"] += 1
    return checked


@pytest.mark.parametrize("q_noise,R", [(0.1, 16), (None, 20)])
def test_prefill_cold_rule_and_planner(B, q_noise, R):
    wp = wl.prefill_bf16(seed=21, n_queries=48, H=64, D=128, L=6000, K=256, n_seed=1024, R=R, q_noise=q_noise)
    wsh, lay = _run(B, wp, n_seed=1024, R=R)
    g_list = _check_cold_rule(wp, wsh, lay, 1024)
    checked = _check_planner(wp, wsh, lay, R, [g_list])
    assert checked["rows"] == wp.M and checked["anchored"] > 0
    print("planner rows", checked)


def test_prefill_small_seed_count(B):
    # n_seed below the common prefix by little: the cut falls among many count levels
    wp = wl.prefill_bf16(seed=22, n_queries=13, H=32, D=128, L=3000, K=128, n_seed=400, R=12, q_noise=0.2)
    wsh, lay = _run(B, wp, n_seed=400, R=12)
    g_list = _check_cold_rule(wp, wsh, lay, 400)
    _check_planner(wp, wsh, lay, 12, [g_list])


def test_ragged_fp8_planner(B):
    wp = wl.ragged_fp8(seed=23, M=6, L_min=3000, L_max=9000, K=256, R=20)
    wsh, lay = _run(B, wp, n_seed=2048, R=20)
    nld = lay["seed_ld"]
    cnt = _arr(wsh, lay["seed_count"], np.int32, wp.M)
    lists = _arr(wsh, lay["seed_list"], np.int32, wp.M * nld).reshape(wp.M, nld)
    seed_lists = []
    for m in range(wp.M):
        want = odosa.strided_seeds(int(wp.key_len[m]), 2048)
        assert np.array_equal(lists[m, :cnt[m]], want), f"row {m}: strided seeds"
        seed_lists.append(want)
    checked = _check_planner(wp, wsh, lay, 20, seed_lists)
    assert checked["rows"] == wp.M
