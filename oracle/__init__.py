"""Plain CPU oracle for partitioned attention with attention-state reuse.

TEST INFRASTRUCTURE ONLY: the test suite, the package's smoke check and the CPU-baseline leg
of ``bench.py`` may import this package; the library (``attention_state_reuse_gb300``) never
does, and it shares no code with it.

The arithmetic lives in ``ditango_oracle.c`` (fp64, pthreads over rows); this module compiles
and loads it, and holds the reuse bookkeeping in plain Python.

Method (DiTango, gist.science/paper/2607.15650, Technical Summary / Methodology):
  * 1. Anchor-Guided Selection Planner: per step, each (query partition, KV partition) pair is
    either computed fresh or reuses its state from an earlier step; anchor steps compute all.
    "Online Prediction" states that local states are always computed, so the diagonal pair
    (i, i) is never reused (reading).
  * 2. State-Centric Parallel Runtime, State Composition: states are (output, log-sum-exp) and
    compose associatively and commutatively; Dynamic Group Compose merges cached states into
    coarser groups without recomputation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ditango_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

ROUND_NONE, ROUND_BF16, ROUND_F32 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle in place (gcc -O2, IEEE arithmetic without FMA contraction, no
    host-specific flags, so x86-64 and aarch64 builds give the same results)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o",
           tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.POINTER
        dp, i64p, u8p = P(ctypes.c_double), P(ctypes.c_int64), P(ctypes.c_uint8)
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        lib.oracle_partition_offsets.argtypes = [i64, i32, i64p]
        lib.oracle_round_bf16.argtypes = [dbl]
        lib.oracle_round_bf16.restype = dbl
        lib.oracle_round_array.argtypes = [dp, i64, i32]
        lib.oracle_rope_rotate.argtypes = [dp, dp, i32, i32, i32, i32, i64, i64, i64, dbl]
        lib.oracle_rope_apply.argtypes = [dp, dp, i64, i64, i64, i32, i32, i32, i32, i64, i64,
                                          i64, dbl, i32, i32]
        lib.oracle_pair_state.argtypes = [dp, dp, dp, i64, i64, i64, i32, dbl, dp, dp, dp]
        lib.oracle_merge.argtypes = [dp, dp, i32, i32, dp, dp]
        lib.oracle_rows_step.argtypes = [dp, dp, dp, i64, i64, i64, i32, i32, i64p, u8p, dbl,
                                         i64p, i64, dp, dp, i32, dp, dp, dp, dp, i32]
        _lib = lib
        return lib


def _dp(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i64p(a: np.ndarray):
    assert a.dtype == np.int64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _u8p(a: np.ndarray):
    assert a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------------------------------
# elementary functions
# ---------------------------------------------------------------------------------------
def partition_offsets(N: int, P: int) -> np.ndarray:
    """Contiguous partition offsets; the first N mod P partitions hold one extra row."""
    out = np.zeros(P + 1, dtype=np.int64)
    _load().oracle_partition_offsets(N, P, _i64p(out))
    return out


def round_array(x: np.ndarray, mode: int) -> np.ndarray:
    y = np.ascontiguousarray(x, dtype=np.float64).copy()
    _load().oracle_round_array(_dp(y), y.size, mode)
    return y


def round_bf16(x) -> np.ndarray:
    return round_array(np.asarray(x, dtype=np.float64), ROUND_BF16)


def rope_rotate(x: np.ndarray, t: int, h: int, w: int, dt: int, dh: int, dw: int,
                theta: float = 10000.0) -> np.ndarray:
    """Rotate one d-vector at 3D position (t, h, w)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_rope_rotate(_dp(x), _dp(y), x.size, dt, dh, dw, t, h, w, theta)
    return y


def rope_apply(x: np.ndarray, Hl: int, Wl: int, start_frame: int, dt: int, dh: int, dw: int,
               theta: float = 10000.0, round_mode: int = ROUND_NONE,
               nthreads: int | None = None) -> np.ndarray:
    """Rotate a [B, N, H, d] tensor by the 3D RoPE of each token's (t_global, h, w), in fp64.

    round_mode rounds the fp64 result once (nearest-even) to bf16 / fp32."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    B, N, H, d = x.shape
    y = np.empty_like(x)
    _load().oracle_rope_apply(_dp(x), _dp(y), B, N, H, d, dt, dh, dw, Hl, Wl, start_frame,
                              theta, round_mode, nthreads or default_threads())
    return y


def pair_state(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """State (O, lse) of one query vector q[d] against keys k[n, d] and values v[n, d]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    n, d = k.shape
    z = np.empty(max(n, 1))
    O = np.empty(d)
    lse = np.empty(1)
    _load().oracle_pair_state(_dp(q), _dp(k), _dp(v), d, 0, n, d, scale, _dp(z), _dp(O), _dp(lse))
    return O, float(lse[0])


def merge(O_s: np.ndarray, lse_s: np.ndarray):
    """Merge states O_s[n, d], lse_s[n] into one state (O[d], lse)."""
    O_s = np.ascontiguousarray(O_s, dtype=np.float64)
    lse_s = np.ascontiguousarray(lse_s, dtype=np.float64)
    n, d = O_s.shape
    O = np.empty(d)
    lse = np.empty(1)
    _load().oracle_merge(_dp(O_s), _dp(lse_s), n, d, _dp(O), _dp(lse))
    return O, float(lse[0])


# ---------------------------------------------------------------------------------------
# reuse bookkeeping (plain Python)
# ---------------------------------------------------------------------------------------
class MaskError(ValueError):
    """A reuse mask the method cannot honour."""


class ReuseBook:
    """Per-pair cache validity and the step at which each cached state was computed.

    A pair may be reused only if a state for it was computed at an earlier step; the local
    (diagonal) pair is always computed. Step 0 therefore computes every pair.
    """

    def __init__(self, P: int):
        self.P = P
        self.valid = np.zeros((P, P), dtype=bool)
        self.step_computed = np.full((P, P), -1, dtype=np.int64)
        self.step = 0

    def check(self, reuse: np.ndarray) -> np.ndarray:
        reuse = np.asarray(reuse)
        if reuse.shape != (self.P, self.P):
            raise MaskError("mask shape")
        if not np.isin(reuse, (0, 1)).all():
            raise MaskError("mask values must be 0 or 1")
        reuse = reuse.astype(np.uint8)
        if np.any(np.diag(reuse) != 0):
            raise MaskError("the local (diagonal) state is always computed")
        if np.any((reuse == 1) & ~self.valid):
            raise MaskError("reuse of a pair with no cached state")
        return reuse

    def advance(self, reuse: np.ndarray) -> np.ndarray:
        reuse = self.check(reuse)
        computed = reuse == 0
        self.valid |= computed
        self.step_computed[computed] = self.step
        self.step += 1
        return reuse

    def computed_pairs(self, reuse: np.ndarray):
        """Computed (i, j) pairs in row-major order."""
        reuse = np.asarray(reuse)
        return [(i, j) for i in range(self.P) for j in range(self.P) if reuse[i, j] == 0]


# ---------------------------------------------------------------------------------------
# multi-step driver over a set of query rows
# ---------------------------------------------------------------------------------------
class OracleRun:
    """Runs the method step by step for a chosen list of query rows (b, h, r).

    Each step: optional RoPE on q and k (rotated in fp64, then rounded once to the attention
    input dtype given by input_round: a bf16 pipeline hands the attention its rotated q and k
    as bf16 tensors; ROUND_NONE keeps them in fp64), fresh states
    for the computed pairs written into the per-row cache (O rounded to the cache dtype, lse
    kept in fp32), then the merge of all P cached states of each row.
    """

    def __init__(self, B, N, H, d, P, scale, rows=None, cache_round=ROUND_BF16,
                 input_round=ROUND_BF16, rope=None, nthreads=None):
        self.B, self.N, self.H, self.d, self.P = B, N, H, d, P
        self.scale = float(scale)
        self.offsets = partition_offsets(N, P)
        if rows is None:
            rows = [(b, h, r) for b in range(B) for h in range(H) for r in range(N)]
        self.rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = self.rows.shape[0]
        self.cache_O = np.full((n, P, d), np.nan)
        self.cache_lse = np.full((n, P), np.nan)
        self.cache_round = cache_round
        self.input_round = input_round
        self.rope = rope  # dict(Hl=, Wl=, start_frame=, dt=, dh=, dw=, theta=) or None
        self.book = ReuseBook(P)
        self.nthreads = nthreads or default_threads()

    def rotate(self, x: np.ndarray) -> np.ndarray:
        r = self.rope
        return rope_apply(x, r["Hl"], r["Wl"], r.get("start_frame", 0), r["dt"], r["dh"],
                          r["dw"], r.get("theta", 10000.0), self.input_round, self.nthreads)

    def step(self, q: np.ndarray, k: np.ndarray, v: np.ndarray, reuse=None):
        """q, k, v: float arrays [B, N, H, d] holding the config-dtype values."""
        P = self.P
        if reuse is None:
            reuse = np.zeros((P, P), dtype=np.uint8)
        reuse = np.ascontiguousarray(self.book.advance(reuse), dtype=np.uint8)
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        if self.rope is not None:
            q = self.rotate(q)
            k = self.rotate(k)
        n = self.rows.shape[0]
        fresh_O = np.empty((n, P, self.d))
        fresh_lse = np.empty((n, P))
        out = np.empty((n, self.d))
        out_lse = np.empty(n)
        _load().oracle_rows_step(
            _dp(q), _dp(k), _dp(v), self.B, self.N, self.H, self.d, P, _i64p(self.offsets),
            _u8p(reuse), self.scale, _i64p(self.rows), n, _dp(self.cache_O), _dp(self.cache_lse),
            self.cache_round, _dp(fresh_O), _dp(fresh_lse), _dp(out), _dp(out_lse),
            self.nthreads)
        return {"out": out, "out_lse": out_lse, "fresh_O": fresh_O, "fresh_lse": fresh_lse,
                "reuse": reuse}
