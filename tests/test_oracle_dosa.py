"""Pins of the DoSA oracle: the DoSA page's worked examples (sections 2, 3.1,
3.2, 5; tests/golden/dosa_examples.json), the bound's validity on random
inputs and exactness of the pruned pass against the plain top-K."""
import json
import os

import numpy as np
import pytest

from oracle import dosa, dsa

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "dosa_examples.json")))


def test_anchor_example():
    g = GOLD["anchor"]
    assert dosa.anchor_coefficient(g["q_h"], g["q_j"]) == g["beta"]
    d = np.array(g["q_h"], float) - g["beta"] * np.array(g["q_j"], float)
    assert d.tolist() == g["d"]
    assert dosa.anchor_bound(g["q_h"], g["q_j"], g["k"]) == g["bound"]
    true = max(float(np.dot(g["q_h"], g["k"])), 0.0)
    assert true == g["true"]
    assert g["w"] * dosa.anchor_bound(g["q_h"], g["q_j"], g["k"]) == g["weighted_bound"]
    assert g["w"] * true == g["weighted_true"]


def test_aggregate_example():
    g = GOLD["aggregate"]
    a = dosa.aggregate_query(g["q"], g["w"])
    assert a.tolist() == g["a_A"]
    assert dosa.aggregate_deduction(a, g["k1"]) == g["agg1"]
    assert dosa.true_deduction(g["q"], g["w"], g["k1"]) == g["true1"]
    assert dosa.total_upper_bound(g["upper_before"], 0.0, g["agg1"]) == g["upper_after"]
    assert not dosa.keep_key(g["upper_after"], g["tau"])
    assert dosa.aggregate_deduction(a, g["k2"]) == g["agg2"]
    assert dosa.true_deduction(g["q"], g["w"], g["k2"]) == g["true2"]


def test_threshold_example():
    g = GOLD["threshold"]
    assert dosa.seed_threshold(g["seed_scores"], g["K"]) == g["tau"]
    assert not dosa.keep_key(g["dropped_U"], g["tau"])
    assert dosa.keep_key(g["kept_U"], g["tau"])
    with pytest.raises(ValueError):
        dosa.seed_threshold([1.0], 2)


def test_teaching_count():
    g = GOLD["teaching"]
    assert dosa.teaching_dot_count(g["n_keys"], g["H"], g["scan"], g["survivors"]) == (g["full"], g["pruned"])


def test_plan_reproduces_the_anchor_example():
    # heads: 0 retained q=(1,0); 1 omitted positive q=(2,1); 2,3 omitted negative
    q = np.array([[1.0, 0.0], [2.0, 1.0], [1.0, 0.0], [0.0, 1.0]])
    w = np.array([1.0, 2.0, -1.0, -1.0])
    samples = np.array([[1.0, 1.0]] * 4)       # both negative heads active on every sample
    plan = dosa.plan_query(q, w, samples, R=1, retained=[0])
    assert plan.pos_heads.tolist() == [1] and plan.anchors.tolist() == [0]
    assert plan.beta.tolist() == [2.0] and plan.d_norm.tolist() == [1.0]
    assert plan.agg_heads.tolist() == [2, 3] and plan.a_A.tolist() == [1.0, 1.0]
    k = np.array([[3.0, 4.0]])
    # U = 1*3 + 2*(2*3 + 1*5) - 7 = 18; true s = 3 + 20 - 3 - 4 = 16
    U = dosa.upper_bound(plan, q, k)[0]
    s, _ = dsa.indexer_score(q, w, k)
    assert U == 18.0 and s[0] == 16.0
    assert dosa.upper_bound_folded(plan, q, k)[0] == pytest.approx(18.0)


def test_activation_frequency_rule():
    q = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, -1.0]])
    w = np.array([1.0, -1.0, -1.0])
    samples = np.array([[1.0, 1.0], [1.0, 1.0], [1.0, -1.0], [1.0, -1.0]])  # each neg head active on half
    plan = dosa.plan_query(q, w, samples, R=1, retained=[0])
    assert plan.agg_heads.tolist() == [1, 2]
    samples3 = np.array([[1.0, 1.0], [1.0, -1.0], [1.0, -1.0]])  # head 1 active on 1 of 3
    plan = dosa.plan_query(q, w, samples3, R=1, retained=[0])
    assert plan.agg_heads.tolist() == [2]


def _random_problem(rng, H, D, L, structured):
    if structured:
        base = rng.standard_normal(D)
        q = base[None, :] * rng.uniform(0.5, 1.5, (H, 1)) + 0.3 * rng.standard_normal((H, D))
    else:
        q = rng.standard_normal((H, D))
    w = rng.standard_normal(H) / np.sqrt(H)
    k = rng.standard_normal((L, D))
    return q, w, k


@pytest.mark.parametrize("structured", [False, True])
def test_bound_is_an_upper_bound(structured):
    rng = np.random.default_rng(41 + structured)
    for _ in range(40):
        H, D, L = int(rng.integers(2, 12)), int(rng.integers(2, 10)), 200
        q, w, k = _random_problem(rng, H, D, L, structured)
        R = int(rng.integers(1, H + 1))
        plan = dosa.plan_query(q, w, k[:64], R)
        U = dosa.upper_bound(plan, q, k)
        Uf = dosa.upper_bound_folded(plan, q, k)
        s, _ = dsa.indexer_score(q, w, k)
        assert (U >= s - 1e-9).all()
        np.testing.assert_allclose(U, Uf, rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("structured", [False, True])
def test_pruned_pass_equals_plain_topk(structured):
    rng = np.random.default_rng(51 + structured)
    survived = []
    for trial in range(40):
        H, D, L = 8, 6, int(rng.integers(20, 300))
        K = int(rng.integers(1, 16))
        q, w, k = _random_problem(rng, H, D, L, structured)
        if trial % 4 == 0:
            # adversarial ties: duplicate keys so some scores equal tau exactly
            k[rng.integers(0, L, L // 3)] = k[rng.integers(0, L, L // 3)]
        seeds = dosa.strided_seeds(L, max(K, L // 4))
        res = dosa.dosa_topk_row(q, w, k, seeds, K, R=3)
        s, _ = dsa.indexer_score(q, w, k)
        ids, sc = dsa.topk(s, K)
        assert res.ids.tolist() == ids.tolist()
        assert np.array_equal(res.scores, sc)
        survived.append(res.n_candidates / max(L, 1))
    if structured:
        assert np.mean(survived) < 0.9      # the bound prunes something on structured heads


def test_too_few_seeds_fall_back_to_full_scoring():
    rng = np.random.default_rng(61)
    q, w, k = _random_problem(rng, 4, 5, 30, False)
    res = dosa.dosa_topk_row(q, w, k, [0, 1], 5, R=2)
    s, _ = dsa.indexer_score(q, w, k)
    assert res.fell_back and res.ids.tolist() == dsa.topk(s, 5)[0].tolist()


def test_seed_rules():
    assert dosa.strided_seeds(10, 4).tolist() == [0, 2, 5, 7]
    assert dosa.strided_seeds(3, 8).tolist() == [0, 1, 2]
    assert dosa.sample_seeds(list(range(1000)), 128)[:3].tolist() == [0, 7, 15]


def test_a_planted_sign_error_in_the_aggregate_is_caught():
    """Adding the aggregate instead of subtracting it breaks the section 3.2 example."""
    g = GOLD["aggregate"]
    a = dosa.aggregate_query(g["q"], g["w"])
    assert dosa.total_upper_bound(g["upper_before"], 0.0, dosa.aggregate_deduction(a, g["k1"])) == 5
    assert g["upper_before"] + dosa.aggregate_deduction(a, g["k1"]) != 5
