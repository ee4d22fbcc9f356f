"""Pins of the planner oracle (oracle/planner.py) against facts that do not come from it.

Importance: a row's merge weights over all partitions sum to 1, so every row of w sums to 1;
equal lse values give w = 1/P; a worked two-partition example with weights 1/4 and 3/4 (lse
ln 1 and ln 3) averages to known values. Drift: zero for unchanged states, |eps| for states
scaled by (1 + eps), and the norm of a one-element perturbation. Selection: a worked example
by hand, the properties any best-first choice within tau and budget has, forced
recomputation of never-computed pairs, the diagonal, the extremes of tau.
"""
import math

import numpy as np
import pytest

from oracle import planner


def test_importance_rows_sum_to_one():
    rng = np.random.default_rng(3)
    lse = rng.normal(size=(2, 3, 5, 23)) * 4
    offs = np.array([0, 5, 10, 14, 19, 23])
    w = planner.importance(lse, offs)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert (w >= 0).all()


def test_importance_equal_lse_is_uniform():
    lse = np.full((1, 2, 4, 8), 0.7)
    w = planner.importance(lse, [0, 2, 4, 6, 8])
    assert np.allclose(w, 0.25, atol=1e-15)


def test_importance_worked_example():
    # P = 2, N = 4 (two rows per partition), B = H = 1.
    # rows 0, 1 (partition 0): lse = (ln 1, ln 3) -> weights (1/4, 3/4); (ln 3, ln 1) -> (3/4, 1/4)
    # rows 2, 3 (partition 1): lse = (0, 0) -> (1/2, 1/2); (ln 1, ln 3) -> (1/4, 3/4)
    lse = np.zeros((1, 1, 2, 4))
    lse[0, 0, :, 0] = [0.0, math.log(3)]
    lse[0, 0, :, 1] = [math.log(3), 0.0]
    lse[0, 0, :, 2] = [0.0, 0.0]
    lse[0, 0, :, 3] = [0.0, math.log(3)]
    w = planner.importance(lse, [0, 2, 4])
    assert np.allclose(w, [[0.5, 0.5], [0.375, 0.625]], atol=1e-15)


def test_drift_closed_forms():
    rng = np.random.default_rng(4)
    a = rng.normal(size=(2, 2, 12, 8))
    offs = [0, 4, 8, 12]
    assert np.all(planner.drift(a, a, offs) == 0.0)
    eps = np.array([0.1, -0.03, 0.5])
    b = a.copy()
    for i in range(3):
        b[:, :, offs[i]:offs[i + 1]] *= 1.0 + eps[i]
    assert np.allclose(planner.drift(b, a, offs), np.abs(eps), atol=1e-14)
    # a perturbation along one channel of one row: ||p|| / ||a_part||
    c = a.copy()
    c[1, 0, 5, 3] += 2.0
    d = planner.drift(c, a, offs)
    ref = 2.0 / math.sqrt((a[:, :, 4:8] ** 2).sum())
    assert d[0] == 0.0 and d[2] == 0.0 and abs(d[1] - ref) < 1e-14
    assert planner.drift(a, np.zeros_like(a), offs).tolist() == [0.0, 0.0, 0.0]


def _candidates(w, delta, g, P):
    out = []
    for i in range(P):
        for k, grp in enumerate(planner.groups(P, g)):
            mem = [j for j in grp if j != i]
            if mem:
                out.append((i, tuple(mem), sum(w[i, j] * delta[i] for j in mem)))
    return out


@pytest.mark.parametrize("P,g,budget,tau", [(3, 1, -1, 0.0), (4, 2, 9, 0.01), (4, 1, 7, 0.02),
                                            (5, 2, 12, 0.0), (4, 3, -1, 0.05), (8, 2, 30, 0.004)])
def test_select_properties(P, g, budget, tau):
    # what any correct best-first selection satisfies: (a) whole groups only, diagonal
    # computed; (b) only groups above tau; (c) within budget; (d) nothing above tau that is
    # left out would still fit; (e) no left-out group ranks above a chosen one of equal or
    # smaller size (it would have been taken first)
    rng = np.random.default_rng(P * 10 + g)
    for _ in range(6):
        w = rng.dirichlet(np.ones(P), size=P)
        delta = rng.uniform(0.0, 0.2, size=P)
        m = planner.select(w, delta, tau, g, budget, np.ones((P, P), bool))
        assert np.all(np.diag(m) == 0)
        used = int((m == 0).sum())
        chosen, left = [], []
        for i, mem, err in _candidates(w, delta, g, P):
            vals = {int(m[i, j]) for j in mem}
            assert len(vals) == 1
            (chosen if vals == {0} else left).append((i, mem, err))
        assert all(err > tau for _, _, err in chosen)
        if budget >= 0:
            assert used <= budget
        for i, mem, err in left:
            if err > tau:
                assert budget >= 0 and used + len(mem) > budget
                assert all(not (err > e2 and len(mem) <= len(m2)) for _, m2, e2 in chosen)


def test_select_worked_example():
    # P = 3, groups of one. errors e[i, j] = w[i, j] * delta[i]:
    #   row 0: (0,1) 0.03, (0,2) 0.02;  row 1: (1,0) 0.02, (1,2) 0.02;  row 2: (2,0) 0.1, (2,1) 0.1
    # tau = 0.025 keeps (2,0), (2,1), (0,1); budget 5 = 3 local pairs + 2: the two 0.1 groups
    # (tie broken by group index) fill it and (0,1) no longer fits.
    w = np.array([[0.5, 0.3, 0.2], [0.1, 0.8, 0.1], [0.25, 0.25, 0.5]])
    delta = np.array([0.1, 0.2, 0.4])
    m = planner.select(w, delta, 0.025, 1, 5, np.ones((3, 3), bool))
    assert m.tolist() == [[0, 1, 1], [1, 0, 1], [0, 0, 0]]
    m = planner.select(w, delta, 0.025, 1, -1, np.ones((3, 3), bool))
    assert m.tolist() == [[0, 0, 1], [1, 0, 1], [0, 0, 0]]


def test_select_forces_never_computed_groups_and_keeps_diagonal():
    P = 4
    w = np.full((P, P), 0.25)
    delta = np.zeros(P)  # no predicted error: everything valid would be reused
    valid = np.ones((P, P), bool)
    valid[2, 0] = False
    m = planner.select(w, delta, 0.0, 2, 0, valid)  # budget 0 cannot stop a forced group
    expect = np.ones((P, P), np.uint8)
    np.fill_diagonal(expect, 0)
    expect[2, 0] = expect[2, 1] = 0  # group {0, 1} of row 2
    assert np.array_equal(m, expect)


def test_select_extremes():
    P = 6
    w = np.full((P, P), 1.0 / P)
    delta = np.full(P, 0.5)
    valid = np.ones((P, P), bool)
    assert (planner.select(w, delta, 0.0, 1, -1, valid) == 0).all()      # recompute all
    m = planner.select(w, delta, 1.0, 1, -1, valid)                      # tau above every error
    assert (m == 1 - np.eye(P, dtype=np.uint8)).all()
