"""Pins for the oracle's reuse bookkeeping and multi-step driver.

DiTango (gist.science/paper/2607.15650), Methodology 1: each step a pair either computes fresh
or reuses the state of an earlier step; anchor steps compute everything; local states are
always computed. Methodology 2: what is cached is the composed state (output, lse).

Checks: masks the method cannot honour are refused; a reused pair contributes exactly the state
computed from the inputs of the step that last computed it (checked against dense attention on
the sub-block, by scipy); with unchanged inputs a reuse step equals the all-compute step up to
the cache's storage rounding.
"""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle


def distance_mask(P, D):
    i, j = np.indices((P, P))
    return (np.abs(i - j) >= D).astype(np.uint8)


def test_book_refuses_reuse_before_any_compute():
    book = oracle.ReuseBook(4)
    with pytest.raises(oracle.MaskError):
        book.advance(distance_mask(4, 2))


def test_book_refuses_diagonal_reuse_and_bad_values():
    book = oracle.ReuseBook(3)
    book.advance(np.zeros((3, 3), np.uint8))
    m = np.zeros((3, 3), np.uint8)
    m[1, 1] = 1
    with pytest.raises(oracle.MaskError):
        book.advance(m)
    m = np.zeros((3, 3), np.uint8)
    m[0, 2] = 2
    with pytest.raises(oracle.MaskError):
        book.advance(m)
    with pytest.raises(oracle.MaskError):
        book.advance(np.zeros((2, 2), np.uint8))


def test_book_records_step_computed():
    book = oracle.ReuseBook(4)
    book.advance(np.zeros((4, 4), np.uint8))
    m = distance_mask(4, 2)
    book.advance(m)
    book.advance(m)
    assert (book.step_computed[m == 1] == 0).all()
    assert (book.step_computed[m == 0] == 2).all()
    assert book.valid.all()


def test_reused_state_is_the_state_of_its_step():
    rng = np.random.default_rng(11)
    B, N, H, d, P, scale = 1, 48, 2, 8, 4, 0.4
    x0 = [rng.standard_normal((B, N, H, d)) for _ in range(3)]
    x1 = [x + 0.3 * rng.standard_normal(x.shape) for x in x0]
    run = oracle.OracleRun(B, N, H, d, P, scale, cache_round=oracle.ROUND_NONE,
                           input_round=oracle.ROUND_NONE, nthreads=2)
    run.step(*x0)
    mask = distance_mask(P, 2)
    res = run.step(*x1, mask)
    off = run.offsets
    for ri, (b, h, r) in enumerate(run.rows):
        i = np.searchsorted(off, r, side="right") - 1
        Os, ls = [], []
        for j in range(P):
            src = x0 if mask[i, j] else x1
            q, k, v = (a[b, :, h] for a in src)
            z = scale * k[off[j]:off[j + 1]] @ q[r]
            Os.append(softmax(z) @ v[off[j]:off[j + 1]])
            ls.append(logsumexp(z))
        L = logsumexp(ls)
        O = sum(np.exp(l - L) * o for o, l in zip(Os, ls))
        np.testing.assert_allclose(res["out"][ri], O, atol=1e-12)
        assert abs(res["out_lse"][ri] - L) < 1e-12


def test_reuse_step_with_unchanged_inputs_equals_anchor():
    rng = np.random.default_rng(12)
    B, N, H, d, P, scale = 1, 40, 2, 8, 5, 0.35
    x = [rng.standard_normal((B, N, H, d)) for _ in range(3)]
    run = oracle.OracleRun(B, N, H, d, P, scale, cache_round=oracle.ROUND_BF16,
                           input_round=oracle.ROUND_NONE, nthreads=2)
    a = run.step(*x)
    r = run.step(*x, distance_mask(P, 2))
    # identical up to the cache's storage rounding (same states, same rounding): exactly equal
    np.testing.assert_array_equal(r["out"], a["out"])
    np.testing.assert_array_equal(r["out_lse"], a["out_lse"])


def test_cache_rounding_is_bf16_of_fresh_state():
    rng = np.random.default_rng(13)
    B, N, H, d, P = 1, 32, 1, 8, 4
    x = [rng.standard_normal((B, N, H, d)) for _ in range(3)]
    run = oracle.OracleRun(B, N, H, d, P, 0.3, cache_round=oracle.ROUND_BF16,
                           input_round=oracle.ROUND_NONE, nthreads=1)
    res = run.step(*x)
    np.testing.assert_array_equal(run.cache_O, oracle.round_bf16(res["fresh_O"]))
    np.testing.assert_array_equal(run.cache_lse, res["fresh_lse"].astype(np.float32))


def test_fresh_states_nan_where_reused():
    rng = np.random.default_rng(14)
    B, N, H, d, P = 1, 32, 1, 4, 4
    x = [rng.standard_normal((B, N, H, d)) for _ in range(3)]
    run = oracle.OracleRun(B, N, H, d, P, 0.5, nthreads=1)
    run.step(*x)
    mask = distance_mask(P, 2)
    res = run.step(*x, mask)
    off = run.offsets
    for ri, (_, _, r) in enumerate(run.rows):
        i = np.searchsorted(off, r, side="right") - 1
        assert np.isnan(res["fresh_lse"][ri][mask[i] == 1]).all()
        assert np.isfinite(res["fresh_lse"][ri][mask[i] == 0]).all()


def test_rope_applies_to_q_and_k_only():
    rng = np.random.default_rng(15)
    Hl, Wl, T = 2, 3, 4
    B, N, H, d, P = 1, T * Hl * Wl, 2, 12, 3
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    rope = dict(Hl=Hl, Wl=Wl, start_frame=2, dt=4, dh=4, dw=4)
    run = oracle.OracleRun(B, N, H, d, P, 0.3, cache_round=oracle.ROUND_NONE,
                           input_round=oracle.ROUND_NONE, rope=rope, nthreads=1)
    res = run.step(q, k, v)
    qr = oracle.rope_apply(q, Hl, Wl, 2, 4, 4, 4)
    kr = oracle.rope_apply(k, Hl, Wl, 2, 4, 4, 4)
    out = res["out"].reshape(B, H, N, d)
    for h in range(H):
        z = 0.3 * qr[0, :, h] @ kr[0, :, h].T
        np.testing.assert_allclose(out[0, h], softmax(z, axis=1) @ v[0, :, h], atol=1e-12)
        np.testing.assert_allclose(res["out_lse"].reshape(B, H, N)[0, h],
                                   logsumexp(z, axis=1), atol=1e-12)
