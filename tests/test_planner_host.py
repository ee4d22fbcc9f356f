"""Host side of the anchor-guided planner and the cache-state restore (no GPU).

ditango_planner_select (C, host) against the oracle's select (numpy/Python): bit-exact masks
on seeded random weights, drifts, thresholds, group sizes, budgets and cache validity (set
through ditango_plan_set_cache_state, whose own argument checks are covered here too).
"""
import numpy as np
import pytest

import attention_state_reuse_gb300 as dt
from oracle import planner as oplan


def _random_state(rng, P, frac_valid):
    valid = (rng.random((P, P)) < frac_valid).astype(np.uint8)
    np.fill_diagonal(valid, 1)
    steps = 5
    sc = np.where(valid == 1, rng.integers(0, steps, size=(P, P)), -1).astype(np.int64)
    return valid, sc, steps


@pytest.mark.parametrize("P", [2, 3, 5, 8, 16, 64])
def test_select_bit_exact_against_oracle(P):
    rng = np.random.default_rng(1000 + P)
    plan = dt.Plan(P * 7, P)
    for trial in range(12):
        valid, sc, steps = _random_state(rng, P, 1.0 if trial % 3 else 0.8)
        plan.set_cache_state(valid, sc, steps)
        w = rng.dirichlet(np.ones(P) * 0.5, size=P)
        delta = rng.uniform(0.0, 0.3, size=P)
        if trial % 4 == 0:
            delta[rng.integers(0, P)] = 0.0
        g = int(rng.integers(1, max(2, P // 2) + 1))
        tau = float(rng.choice([0.0, 1e-3, 1e-2, 0.05]))
        budget = int(rng.choice([-1, P, P + P * P // 4, P * P]))
        got = dt.planner_select(plan, w, delta, tau, g, budget)
        want = oplan.select(w, delta, tau, g, budget, valid.astype(bool))
        assert np.array_equal(got, want), (trial, P, g, tau, budget)


def test_select_ties_and_duplicates_bit_exact():
    # equal weights make many errors equal: the tie order (lower i, then lower group) decides
    P = 8
    plan = dt.Plan(64, P)
    plan.set_cache_state(np.ones((P, P), np.uint8), np.zeros((P, P), np.int64), 1)
    w = np.full((P, P), 1.0 / P)
    for budget in (P, P + 3, P + 10, -1):
        for g in (1, 2, 3):
            delta = np.full(P, 0.1)
            got = dt.planner_select(plan, w, delta, 0.0, g, budget)
            want = oplan.select(w, delta, 0.0, g, budget, np.ones((P, P), bool))
            assert np.array_equal(got, want), (budget, g)


def test_select_argument_checks():
    P = 4
    plan = dt.Plan(16, P)
    w = np.full((P, P), 0.25)
    d = np.zeros(P)
    for bad in [dict(group=0), dict(tau=-1.0), dict(tau=float("nan"))]:
        kw = dict(tau=0.0, group=1, budget=-1)
        kw.update(bad)
        with pytest.raises(dt.DitangoError) as e:
            dt.planner_select(plan, w, d, kw["tau"], kw["group"], kw["budget"])
        assert e.value.name == "INVALID_ARG"
    w2 = w.copy()
    w2[1, 2] = np.inf
    with pytest.raises(dt.DitangoError):
        dt.planner_select(plan, w2, d, 0.0, 1, -1)


def test_set_cache_state_round_trip_and_checks():
    P = 5
    plan = dt.Plan(50, P)
    rng = np.random.default_rng(7)
    valid, sc, steps = _random_state(rng, P, 0.7)
    plan.set_cache_state(valid, sc, steps)
    v2, sc2, st2 = plan.cache_state()
    assert np.array_equal(v2, valid) and np.array_equal(sc2, sc) and st2 == steps
    # the restored validity drives the reuse checks
    m = np.where(valid == 1, 1, 0).astype(np.uint8)
    np.fill_diagonal(m, 0)
    plan.check_mask(m)
    bad_cases = []
    v = valid.copy(); v[0, 1] = 2; bad_cases.append((v, sc, steps))            # value not 0/1
    s = sc.copy(); s[valid == 1] = steps; bad_cases.append((valid, s, steps))   # step not run yet
    v = valid.copy(); v[2, 2] = 0; s = sc.copy(); s[2, 2] = -1
    bad_cases.append((v, s, steps))                                            # diagonal invalid
    v = valid.copy(); v[0, 1] = 0; s = sc.copy(); s[0, 1] = 3
    bad_cases.append((v, s, steps))                                            # invalid with a step
    for v, s, st in bad_cases:
        with pytest.raises(dt.DitangoError) as e:
            plan.set_cache_state(v, s, st)
        assert e.value.name == "INVALID_ARG"
    v3, sc3, st3 = plan.cache_state()  # unchanged by the refused calls
    assert np.array_equal(v3, valid) and np.array_equal(sc3, sc) and st3 == steps


def test_anchor_planner_predicts_the_reuse_mask(monkeypatch):
    # host logic of AnchorPlanner's ahead-of-time group build, with the device reductions
    # replaced by fakes: the mask chosen right after an anchor becomes the plan's default mask
    # before the next anchor, and only when build_ahead is on
    import torch

    P = 4
    chosen = [np.array(m, np.uint8) for m in ([[0, 1, 1, 1], [1, 0, 1, 1], [1, 1, 0, 1], [1, 1, 1, 0]],
                                              [[0, 0, 1, 1], [0, 0, 0, 1], [1, 0, 0, 0], [1, 1, 0, 0]])]
    calls = {"select": 0}

    def fake_select(plan, w, delta, tau, group, budget):
        calls["select"] += 1
        return chosen[(calls["select"] - 1) % 2]

    monkeypatch.setattr(dt, "planner_importance", lambda *a, **k: torch.zeros((P, P)))
    monkeypatch.setattr(dt, "planner_snapshot", lambda *a, **k: None)
    monkeypatch.setattr(dt, "planner_drift", lambda *a, **k: torch.zeros(P))
    monkeypatch.setattr(dt, "planner_select", fake_select)

    class FakePlan:
        def __init__(self):
            self.P, self.defaults = P, []

        def set_mask(self, m):
            self.defaults.append(np.array(m, np.uint8))

    cO = torch.empty((1, 1, P, 8, 4))
    cL = torch.empty((1, 1, P, 8))
    for ahead in (True, False):
        plan = FakePlan()
        calls["select"] = 0
        ap = dt.AnchorPlanner(plan, cO, cL, anchor_every=3, tau=1e-3, build_ahead=ahead)
        masks = []
        for _ in range(7):
            m = ap.mask()
            masks.append(m)
            ap.after_step(m)
        assert [bool(m.any()) for m in masks] == [False, True, True, False, True, True, False]
        if ahead:
            # anchors at steps 3 and 6 set the mask chosen right after the anchors at 0 and 3
            assert len(plan.defaults) == 2
            assert np.array_equal(plan.defaults[0], masks[1])
            assert np.array_equal(plan.defaults[1], masks[4])
            assert np.array_equal(ap.predicted, masks[4])
        else:
            assert plan.defaults == []
