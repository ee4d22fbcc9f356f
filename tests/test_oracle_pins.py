"""Pins for the CPU oracle: each test ties it to something other than itself.

* hand-derived worked example (tests/golden/tiny_state.txt);
* the closed form: with every pair computed, merged states equal dense softmax attention,
  evaluated by scipy's logsumexp / softmax (DiTango, Methodology 2, State Composition:
  composing all partition states yields the full attention state);
* algebraic invariants: merge order and grouping do not matter (states compose associatively
  and commutatively), a single partition is the identity, merge weights sum to one;
* bf16 rounding against torch's fp32 -> bf16 conversion;
* partition offsets against numpy.array_split sizes.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle


def dense_attention(q, k, v, scale):
    """Reference: softmax(scale q k^T) v and the row log-sum-exp, via scipy."""
    z = scale * q @ k.T
    return softmax(z, axis=1) @ v, logsumexp(z, axis=1)


# ---------------------------------------------------------------- golden worked example
def _golden_inputs(g):
    q = np.array(g["q"][0]).reshape(4, 2)
    k = np.array(g["k"][0]).reshape(4, 2)
    v0 = np.array(g["v0"][0]).reshape(4, 2)
    v1 = np.array(g["v1"][0]).reshape(4, 2)
    return q, k, v0, v1


@pytest.mark.parametrize("scale,key_state,key_merged", [(1.0, "s1_state", "s1_merged"),
                                                        (2.0, "s2_state", "s2_merged")])
def test_golden_states_and_merge(golden, scale, key_state, key_merged):
    g = golden("tiny_state.txt")
    q, k, v0, _ = _golden_inputs(g)
    off = oracle.partition_offsets(4, 2)
    for row, j, o0, o1, else_ in g[key_state]:
        O, lse = oracle.pair_state(q[int(row)], k[off[int(j)]:off[int(j) + 1]],
                                   v0[off[int(j)]:off[int(j) + 1]], scale)
        np.testing.assert_allclose(O, [o0, o1], atol=1e-12)
        assert abs(lse - np.log(else_)) < 1e-12
    for row, o0, o1, else_ in g[key_merged]:
        states = [oracle.pair_state(q[int(row)], k[off[j]:off[j + 1]], v0[off[j]:off[j + 1]],
                                    scale) for j in range(2)]
        O, lse = oracle.merge(np.stack([s[0] for s in states]), np.array([s[1] for s in states]))
        np.testing.assert_allclose(O, [o0, o1], atol=1e-12)
        assert abs(lse - np.log(else_)) < 1e-12


def test_golden_reuse_step(golden):
    g = golden("tiny_state.txt")
    q, k, v0, v1 = _golden_inputs(g)
    to4 = lambda x: x.reshape(1, 4, 1, 2)
    for key, mask in (("s1_reuse_merged", [[0, 1], [0, 0]]), ("s1_fresh_merged", [[0, 0], [0, 0]])):
        run = oracle.OracleRun(1, 4, 1, 2, 2, 1.0, cache_round=oracle.ROUND_NONE,
                               input_round=oracle.ROUND_NONE)
        run.step(to4(q), to4(k), to4(v0))
        res = run.step(to4(q), to4(k), to4(v1), np.array(mask, dtype=np.uint8))
        for row, o0, o1, else_ in g[key]:
            np.testing.assert_allclose(res["out"][int(row)], [o0, o1], atol=1e-12)
            assert abs(res["out_lse"][int(row)] - np.log(else_)) < 1e-12


# ---------------------------------------------------------------- closed form: dense attention
@pytest.mark.parametrize("N,P,d,scale", [(64, 4, 8, 0.35), (61, 5, 4, 1.0), (33, 1, 6, 0.5),
                                         (40, 8, 16, 0.25), (7, 7, 3, 2.0)])
def test_all_compute_equals_dense(N, P, d, scale):
    rng = np.random.default_rng(N * 100 + P)
    B, H = 2, 3
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    run = oracle.OracleRun(B, N, H, d, P, scale, cache_round=oracle.ROUND_NONE,
                           input_round=oracle.ROUND_NONE, nthreads=3)
    res = run.step(q, k, v)
    out = res["out"].reshape(B, H, N, d)
    lse = res["out_lse"].reshape(B, H, N)
    for b in range(B):
        for h in range(H):
            O_ref, L_ref = dense_attention(q[b, :, h], k[b, :, h], v[b, :, h], scale)
            np.testing.assert_allclose(out[b, h], O_ref, atol=1e-12, rtol=1e-12)
            np.testing.assert_allclose(lse[b, h], L_ref, atol=1e-12, rtol=1e-12)


def test_pair_state_equals_dense_on_block():
    rng = np.random.default_rng(7)
    q = rng.standard_normal(12)
    k = rng.standard_normal((37, 12)) * 2.0
    v = rng.standard_normal((37, 12))
    O, lse = oracle.pair_state(q, k, v, 0.3)
    O_ref, L_ref = dense_attention(q[None], k, v, 0.3)
    np.testing.assert_allclose(O, O_ref[0], atol=1e-13)
    assert abs(lse - L_ref[0]) < 1e-13


def test_pair_state_large_logits_stable():
    # the max-shift keeps exp() in range: logits near 1000 must not overflow
    q = np.array([100.0, 0.0])
    k = np.array([[10.0, 0.0], [9.99, 0.0], [0.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0], [5.0, 5.0]])
    O, lse = oracle.pair_state(q, k, v, 1.0)
    O_ref, L_ref = dense_attention(q[None], k, v, 1.0)
    assert np.isfinite(O).all() and np.isfinite(lse)
    np.testing.assert_allclose(O, O_ref[0], atol=1e-12)
    assert abs(lse - L_ref[0]) < 1e-9


# ---------------------------------------------------------------- merge invariants
def _random_states(rng, n, d):
    return rng.standard_normal((n, d)), rng.standard_normal(n) * 3.0


def test_merge_permutation_invariant():
    rng = np.random.default_rng(1)
    O_s, l_s = _random_states(rng, 9, 5)
    O, L = oracle.merge(O_s, l_s)
    for _ in range(5):
        p = rng.permutation(9)
        O2, L2 = oracle.merge(O_s[p], l_s[p])
        np.testing.assert_allclose(O2, O, atol=1e-13)
        assert abs(L2 - L) < 1e-13


def test_merge_grouping_invariant():
    # Dynamic Group Compose: merging cached states into coarser groups first changes nothing
    rng = np.random.default_rng(2)
    O_s, l_s = _random_states(rng, 8, 6)
    O, L = oracle.merge(O_s, l_s)
    for groups in ([[0, 1], [2, 3], [4, 5], [6, 7]], [[0, 5, 7], [1], [2, 3, 4, 6]]):
        parts = [oracle.merge(O_s[g], l_s[g]) for g in groups]
        O2, L2 = oracle.merge(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
        np.testing.assert_allclose(O2, O, atol=1e-13)
        assert abs(L2 - L) < 1e-13


def test_merge_single_state_is_identity():
    rng = np.random.default_rng(3)
    O_s, l_s = _random_states(rng, 1, 7)
    O, L = oracle.merge(O_s, l_s)
    np.testing.assert_array_equal(O, O_s[0])
    assert L == l_s[0]


def test_merge_weights_sum_to_one():
    rng = np.random.default_rng(4)
    _, l_s = _random_states(rng, 6, 3)
    # merging states whose outputs are all the same vector returns that vector
    O_s = np.tile(np.array([1.5, -2.0, 0.25]), (6, 1))
    O, L = oracle.merge(O_s, l_s)
    np.testing.assert_allclose(O, O_s[0], atol=1e-14)
    assert abs(np.exp(l_s - L).sum() - 1.0) < 1e-14
    assert abs(L - logsumexp(l_s)) < 1e-13


def test_one_partition_is_identity_of_dense():
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 20, 1, 4)) for _ in range(3))
    run = oracle.OracleRun(1, 20, 1, 4, 1, 0.5, cache_round=oracle.ROUND_NONE,
                           input_round=oracle.ROUND_NONE, nthreads=1)
    res = run.step(q, k, v)
    np.testing.assert_allclose(res["fresh_O"][:, 0, :], res["out"], atol=1e-15)
    np.testing.assert_allclose(res["fresh_lse"][:, 0], res["out_lse"], atol=1e-15)


# ---------------------------------------------------------------- partitioning
@pytest.mark.parametrize("N,P", [(1024, 4), (4096, 8), (32760, 8), (75600, 16), (32760, 16),
                                 (32760, 4), (10, 3), (5, 5)])
def test_partition_offsets_match_array_split(N, P):
    off = oracle.partition_offsets(N, P)
    sizes = [len(a) for a in np.array_split(np.arange(N), P)]
    np.testing.assert_array_equal(np.diff(off), sizes)
    assert off[0] == 0 and off[-1] == N


def test_partition_offsets_sweep_p16():
    off = oracle.partition_offsets(32760, 16)
    assert list(np.diff(off)) == [2048] * 8 + [2047] * 8


# ---------------------------------------------------------------- rounding
def test_round_bf16_matches_torch():
    rng = np.random.default_rng(6)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormal range
        (rng.standard_normal(2000) * 8e37).clip(-3.39e38, 3.39e38).astype(np.float32),
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 3.3961e38, 0.0, -0.0],
                 dtype=np.float32),                               # ties and overflow
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
