"""Host-side checks of the C ABI (no GPU needed).

* the shared library loads and exports every entry point declared in include/ditango.h;
* the planner's partition offsets and computed-pair lists equal the oracle's, bit for bit;
* masks the method cannot honour are refused with the documented status codes, exactly where
  the oracle's bookkeeping refuses them (DiTango, Methodology 1: local states are always
  computed; a pair is reusable only after a state for it exists).
"""
import os
import re

import numpy as np
import pytest

import oracle
from attention_state_reuse_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ditango():
    import attention_state_reuse_gb300 as m

    m.build()
    m.load_library()
    return m


def header_symbols():
    text = open(os.path.join(ROOT, "include", "ditango.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ditango_[a-z_]+)\s*\(", text)))


def test_header_symbols_listed_in_binding(ditango):
    assert header_symbols() == sorted(ditango.SYMBOLS)


def test_library_exports_every_header_symbol(ditango):
    lib = ditango.load_library()
    for name in header_symbols():
        assert hasattr(lib, name), name


def test_version_and_status_strings(ditango):
    lib = ditango.load_library()
    header = open(os.path.join(ROOT, "include", "ditango.h")).read()
    want = int(re.search(r"#define DITANGO_ABI_VERSION (\d+)", header).group(1))
    assert lib.ditango_version() == want
    for code in range(11):
        assert lib.ditango_status_string(code)
    assert lib.ditango_status_string(99) == b"unknown status"


@pytest.mark.parametrize("N,P", [(1024, 4), (4096, 8), (32760, 8), (75600, 16), (32760, 16),
                                 (32760, 4), (1560, 8), (64, 64), (65, 64), (300, 1), (7, 3)])
def test_offsets_bit_exact(ditango, N, P):
    plan = ditango.Plan(N, P)
    np.testing.assert_array_equal(plan.offsets(), oracle.partition_offsets(N, P))


@pytest.mark.parametrize("P", [1, 4, 8, 16, 64])
def test_pairs_bit_exact(ditango, P):
    plan = ditango.Plan(max(P, 100), P)
    book = oracle.ReuseBook(P)
    masks = [np.zeros((P, P), np.uint8)] + [wl.distance_mask(P, D) for D in range(1, P + 1)]
    masks.append(wl.random_mask(P, 123))
    for m in masks:
        assert plan.pairs(m) == book.computed_pairs(m)
    assert plan.pairs() == [(i, j) for i in range(P) for j in range(P)]


def test_plan_rejects_bad_arguments(ditango):
    with pytest.raises(ditango.DitangoError) as e:
        ditango.Plan(3, 4)  # N < P
    assert e.value.name == "INVALID_ARG"
    with pytest.raises(ditango.DitangoError):
        ditango.Plan(100, 0)
    with pytest.raises(ditango.DitangoError):
        ditango.Plan(1000, 65)
    diag = np.zeros((4, 4), np.uint8)
    diag[2, 2] = 1
    with pytest.raises(ditango.DitangoError) as e:
        ditango.Plan(100, 4, diag)
    assert e.value.name == "INVALID_MASK"


def test_fault_injection_arguments(ditango):
    plan = ditango.Plan(100, 4)
    plan.inject_fault(1)
    plan.inject_fault(0)
    for kind in (2, -1):
        with pytest.raises(ditango.DitangoError) as e:
            plan.inject_fault(kind)
        assert e.value.name == "INVALID_ARG"


def test_mask_checks_match_oracle_book(ditango):
    P = 8
    plan = ditango.Plan(4096, P)
    book = oracle.ReuseBook(P)
    bad_val = np.zeros((P, P), np.uint8)
    bad_val[0, 3] = 2
    diag = np.zeros((P, P), np.uint8)
    diag[5, 5] = 1
    cases = [(np.zeros((P, P), np.uint8), 0), (wl.distance_mask(P, 2), 3), (bad_val, 2),
             (diag, 2), (wl.random_mask(P, 9), 3)]
    for m, status in cases:
        assert plan.check_mask(m) == status
        if status == 0:
            book.check(m)
        else:
            with pytest.raises(oracle.MaskError):
                book.check(m)
    # default mask (all computed) is always usable; nothing was run, so nothing is valid
    assert plan.check_mask(None) == 0
    valid, sc, steps = plan.cache_state()
    assert steps == 0 and not valid.any() and (sc == -1).all()


def _desc(ditango, shape, dtype):
    """A tensor descriptor with a NULL data pointer (never dereferenced by the checks below)."""
    t = ditango.Tensor()
    t.ptr = None
    t.dtype = dtype
    t.ndim = len(shape)
    stride = 1
    for a in reversed(range(len(shape))):
        t.shape[a] = shape[a]
        t.stride[a] = stride
        stride *= max(shape[a], 1)
    return t


@pytest.mark.parametrize("B,H", [(0, 2), (1, 0), (0, 0)])
def test_empty_batch_is_refused_before_any_pointer_is_read(ditango, B, H):
    import ctypes

    N, P, d = 256, 4, 64
    plan = ditango.Plan(N, P)
    lib = ditango.load_library()
    q = _desc(ditango, (B, N, H, d), ditango.BF16)
    cache = ditango.StateCache(_desc(ditango, (B, H, P, N, d), ditango.BF16),
                               _desc(ditango, (B, H, P, N), ditango.F32))
    out = _desc(ditango, (B, N, H, d), ditango.BF16)
    st = lib.ditango_attn_step(plan.handle, ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                               None, None, ctypes.byref(cache), ctypes.byref(out), None,
                               ctypes.c_float(0.125), None, ctypes.c_size_t(0), None)
    assert ditango.STATUS[st] == "SHAPE"
    assert plan.cache_state()[2] == 0


@pytest.mark.parametrize("shape", [(0, 3, 5, 64), (2, 0, 5, 64), (2, 3, 0, 64)])
def test_merge_without_rows_is_a_no_op(ditango, shape):
    import ctypes

    lib = ditango.load_library()
    sl = ditango.StateList()
    sl.n = 2
    sl.dtype = ditango.BF16
    nulls = (ctypes.c_void_p * 2)(None, None)
    sl.O = ctypes.cast(nulls, ctypes.POINTER(ctypes.c_void_p))
    sl.lse = ctypes.cast(nulls, ctypes.POINTER(ctypes.c_void_p))
    for a in range(4):
        sl.shape[a] = shape[a]
    out = _desc(ditango, shape, ditango.BF16)
    out_lse = _desc(ditango, shape[:3], ditango.F32)
    st = lib.ditango_merge(ctypes.byref(sl), ctypes.byref(out), ctypes.byref(out_lse), None)
    assert ditango.STATUS[st] == "OK"
    # the shape of out is still checked, and a d the vector width does not divide is refused
    bad = _desc(ditango, shape[:3] + (32,), ditango.BF16)
    assert ditango.STATUS[lib.ditango_merge(ctypes.byref(sl), ctypes.byref(bad), None, None)] == "SHAPE"
    sl.shape[3] = 60
    out60 = _desc(ditango, shape[:3] + (60,), ditango.BF16)
    assert ditango.STATUS[lib.ditango_merge(ctypes.byref(sl), ctypes.byref(out60), None, None)] == "SHAPE"


def test_workload_mask_fractions():
    # distance-threshold masks of the configurations (fractions of reused pairs)
    assert wl.reuse_fraction(wl.distance_mask(4, 2)) == 6 / 16
    assert wl.reuse_fraction(wl.distance_mask(8, 2)) == 42 / 64
    assert wl.reuse_fraction(wl.distance_mask(16, 3)) == 182 / 256
    assert wl.reuse_fraction(wl.distance_mask(8, 1)) == 56 / 64
    assert wl.reuse_fraction(wl.distance_mask(16, 2)) == 210 / 256
    m = wl.random_mask(16, 4023)
    assert (np.diag(m) == 0).all()
    np.testing.assert_array_equal(m, wl.random_mask(16, 4023))
    assert 0.3 < wl.reuse_fraction(m) < 0.6


@pytest.mark.parametrize("P,S", [(1, 1), (4, 4), (8, 3), (16, 5), (16, 1), (64, 7), (5, 2)])
def test_cache_slot_map_keeps_the_pairs_nearest_the_diagonal(ditango, P, S):
    # host storage of a state cache (DiTango, closing limitations paragraph: CPU offloading of
    # the state cache): each query partition keeps its S pairs nearest the diagonal on the
    # device, in ascending j, and the local pair always
    m = ditango.cache_slot_map(P, S)
    assert m.shape == (P, P) and m.dtype == np.int8
    for i in range(P):
        dev = [j for j in range(P) if m[i, j] >= 0]
        assert len(dev) == S and m[i, i] >= 0
        assert [int(m[i, j]) for j in dev] == list(range(S))  # slots in ascending j
        want = sorted(range(P), key=lambda j: (abs(i - j), j))[:S]
        assert sorted(want) == dev
        assert all(m[i, j] == -1 for j in range(P) if j not in dev)
    if S == P:
        np.testing.assert_array_equal(m, np.tile(np.arange(P, dtype=np.int8), (P, 1)))


def test_cache_slot_map_distance_band(ditango):
    # S = 2D - 1 holds every pair a |i - j| >= D mask computes
    for P, D in [(16, 3), (8, 2), (16, 2), (4, 1)]:
        m = ditango.cache_slot_map(P, 2 * D - 1)
        comp = wl.distance_mask(P, D) == 0
        assert (m[comp] >= 0).all()


@pytest.mark.parametrize("P,S", [(4, 0), (4, 5), (65, 3), (0, 1)])
def test_cache_slot_map_refuses_bad_sizes(ditango, P, S):
    import ctypes

    lib = ditango.load_library()
    buf = (ctypes.c_int8 * 64)()
    assert ditango.STATUS[lib.ditango_cache_slot_map(P, S, buf)] == "INVALID_ARG"
    assert ditango.STATUS[lib.ditango_cache_slot_map(4, 2, None)] == "INVALID_ARG"


@pytest.mark.parametrize("shape", [(-1, 256, 2, 64), (1, 256, 0, 64), (1, 255, 2, 64),
                                   (1 << 20, 256, 1 << 20, 64)])
def test_static_workspace_step_reports_bad_shapes_as_shape(ditango, shape):
    # the step without a workspace checks the shape before sizing its scratch from it
    import ctypes

    N, P = 256, 4
    plan = ditango.Plan(N, P)
    lib = ditango.load_library()
    q = _desc(ditango, (1, N, 2, 64), ditango.BF16)
    for a in range(4):
        q.shape[a] = shape[a]
    cache = ditango.StateCache(_desc(ditango, (1, 2, P, N, 64), ditango.BF16),
                               _desc(ditango, (1, 2, P, N), ditango.F32))
    out = _desc(ditango, (1, N, 2, 64), ditango.BF16)
    rope = ditango.Rope()
    st = lib.ditango_attn_step_static_workspace(plan.handle, ctypes.byref(q), ctypes.byref(q),
                                                ctypes.byref(q), ctypes.byref(rope), None,
                                                ctypes.byref(cache), ctypes.byref(out), None,
                                                ctypes.c_float(0.125), None)
    assert ditango.STATUS[st] == "SHAPE"
    assert plan.cache_state()[2] == 0
