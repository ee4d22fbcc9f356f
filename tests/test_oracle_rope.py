"""Pins for the oracle's 3D rotary embedding.

Sources: "Accelerating Video Generation Inference with Sequential-Parallel 3D Positional
Encoding Using a Global Time Index" (gist.science/es/paper/2603.06664), section 2, Causal-RoPE
SP: each token's global time index is its local frame plus the start frame s, so no rank needs
the whole sequence to place its tokens; and "Kaleido" (gist.science/es/paper/2607.13770),
Methodology 1: RoPE splits the head channels into a temporal, a horizontal and a vertical group.

The pages give no formula, so these tests pin what any rotary embedding must satisfy and what
the pages do state:
* rotations preserve norms and are the identity at position 0;
* scores depend only on relative positions, per axis;
* each channel group moves only with its own axis (t / h / w split 44 / 42 / 42 at d = 128);
* pair k = 0 (the fastest-turning pair) of every axis turns by exactly `pos` radians,
  counter-clockwise (measured with atan2);
* global time index: a token of local frame t in a block starting at frame s is rotated
  exactly like frame t + s of a block starting at 0.
"""
import numpy as np
import pytest

import oracle

D, DT, DH, DW = 128, 44, 42, 42


def rot(x, t, h, w):
    return oracle.rope_rotate(x, t, h, w, DT, DH, DW)


def test_identity_at_origin():
    x = np.random.default_rng(0).standard_normal(D)
    np.testing.assert_array_equal(rot(x, 0, 0, 0), x)


@pytest.mark.parametrize("pos", [(1, 0, 0), (0, 7, 0), (0, 0, 51), (20, 29, 51), (1000, 3, 9)])
def test_norm_preserved(pos):
    x = np.random.default_rng(1).standard_normal(D)
    y = rot(x, *pos)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
    # pairwise norms too: each channel pair is an independent rotation
    np.testing.assert_allclose(np.hypot(y[0::2], y[1::2]), np.hypot(x[0::2], x[1::2]),
                               atol=1e-12)


def test_relative_position_property():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    p1, p2 = np.array([5, 11, 40]), np.array([2, 20, 3])
    base = rot(q, *p1) @ rot(k, *p2)
    for shift in ([1, 0, 0], [0, 3, 0], [0, 0, 17], [9, 4, 2]):
        s = np.array(shift)
        assert abs(rot(q, *(p1 + s)) @ rot(k, *(p2 + s)) - base) < 1e-10


@pytest.mark.parametrize("axis,lo,hi", [(0, 0, DT), (1, DT, DT + DH), (2, DT + DH, D)])
def test_axis_channel_groups(axis, lo, hi):
    x = np.random.default_rng(3).standard_normal(D)
    pos = [3, 4, 5]
    a = rot(x, *pos)
    pos[axis] += 6
    b = rot(x, *pos)
    changed = np.nonzero(np.abs(a - b) > 1e-12)[0]
    assert changed.min() >= lo and changed.max() < hi
    # every pair of the group moves (no frequency is zero)
    assert set(changed // 2) == set(range(lo // 2, hi // 2))


@pytest.mark.parametrize("axis,first_pair", [(0, 0), (1, DT // 2), (2, DT // 2 + DH // 2)])
def test_lowest_pair_turns_by_pos_radians(axis, first_pair):
    for pos_val in (1, 2, 5, 13):
        x = np.zeros(D)
        x[2 * first_pair] = 1.0
        pos = [0, 0, 0]
        pos[axis] = pos_val
        y = rot(x, *pos)
        ang = np.arctan2(y[2 * first_pair + 1], y[2 * first_pair])
        expect = np.angle(np.exp(1j * pos_val))  # pos mod 2 pi, counter-clockwise
        assert abs(ang - expect) < 1e-12


def test_frequencies_decrease_within_axis():
    # unit vectors on each pair, rotated by pos 1: turn angles fall monotonically inside a group
    angles = []
    for m in range(D // 2):
        x = np.zeros(D)
        x[2 * m] = 1.0
        axis = 0 if m < DT // 2 else (1 if m < DT // 2 + DH // 2 else 2)
        pos = [0, 0, 0]
        pos[axis] = 1
        y = rot(x, *pos)
        angles.append(np.arctan2(y[2 * m + 1], y[2 * m]))
    angles = np.array(angles)
    for lo, hi in ((0, DT // 2), (DT // 2, DT // 2 + DH // 2), (DT // 2 + DH // 2, D // 2)):
        seg = angles[lo:hi]
        assert abs(seg[0] - 1.0) < 1e-12
        assert np.all(np.diff(seg) < 0) and np.all(seg > 0)


def test_raster_order_and_global_time_index():
    Tl, Hl, Wl, s = 3, 4, 5, 7
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, Tl * Hl * Wl, 2, D))
    y_s = oracle.rope_apply(x, Hl, Wl, s, DT, DH, DW, nthreads=2)
    for t in range(Tl):
        for h in range(Hl):
            for w in range(Wl):
                n = (t * Hl + h) * Wl + w
                for hd in range(2):
                    np.testing.assert_allclose(y_s[0, n, hd], rot(x[0, n, hd], t + s, h, w),
                                               atol=1e-13)
    # a block that starts at frame s rotates like the same frames of a longer block from 0
    x_long = np.concatenate([rng.standard_normal((1, s * Hl * Wl, 2, D)), x], axis=1)
    y_long = oracle.rope_apply(x_long, Hl, Wl, 0, DT, DH, DW, nthreads=2)
    np.testing.assert_allclose(y_long[:, s * Hl * Wl:], y_s, atol=1e-13)


def test_rope_apply_rounds_to_bf16_when_asked():
    x = np.random.default_rng(5).standard_normal((1, 20, 1, D))
    y = oracle.rope_apply(x, 4, 5, 0, DT, DH, DW, round_mode=oracle.ROUND_BF16, nthreads=1)
    y64 = oracle.rope_apply(x, 4, 5, 0, DT, DH, DW, nthreads=1)
    np.testing.assert_array_equal(y, oracle.round_bf16(y64))
