"""Seeded synthetic workloads: shapes, inputs, drift, reuse masks and step schedules.

This module holds no arithmetic of the method itself; it only draws inputs. Both the library
tests and the CPU oracle consume what it produces, so they see identical values.

Workloads (video-DiT attention layers; no model weights or data are involved):
  tiny_fp32     B=1, H=2,  d=64,  N=1024  (latent 4x16x16),  P=4,  fp32, 2 steps
  small_bf16    B=1, H=12, d=64,  N=4096  (latent 4x32x32),  P=8,  bf16, 10 steps
  wan14b_layer  B=1, H=40, d=128, N=32760 (latent 21x30x52), P=8,  bf16, 3D RoPE
  long_720p     B=1, H=40, d=128, N=75600 (latent 21x45x80), P=16, bf16, 3D RoPE, 8 steps
  sweep_P{4,8,16}  N=32760, H=40, d=128, bf16: distance masks from all-compute down to the
                   smallest distance with at most 87.5% of pairs reused, plus a random mask
The latent grids stand in for Wan2.1 video latents at 480p (21x30x52) and 720p (21x45x80).

Recipe: Q, K, V ~ N(0, 1) drawn with numpy's PCG64 generator in float32, one seed per tensor
(config index c -> seeds 1000c+1, +2, +3); step t adds drift sigma * N(0, 1) from seed
1000c+100+t (tensor x = 0, 1, 2 for Q, K, V). Each tensor is drawn in consecutive chunks of
2^22 values (flat row-major order), chunk m from its own generator seeded with [seed, m] (the
drift: [seed, x, m]), so the values do not depend on how many threads draw them. The fp32
master values are rounded to the config dtype for use. Per-(tensor, head) scales U(0.5, 2) for wan14b_layer come
from seed 1000c+50. small_bf16 divides Q (and its drift) by sqrt(d) and uses softmax scale 1.
Random masks: splitmix64 (Vigna's published generator) seeded with 1000c+7+P, one draw per
pair in row-major order; a pair is reused iff (x >> 11) * 2^-53 < 0.5; the diagonal is always
computed (its draw is still consumed).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1


@dataclass
class Workload:
    name: str
    index: int          # seed base index c
    B: int
    H: int
    d: int
    T: int
    Hl: int
    Wl: int
    P: int
    dtype: str          # "fp32" | "bf16"
    steps: int
    drift: float
    rope: bool = False
    start_frame: int = 0
    q_scale: float = 1.0         # multiplies Q and its drift
    softmax_scale: float | None = None
    head_scales: bool = False    # per-(tensor, head) U(0.5, 2) scales
    schedule: list = field(default_factory=list)  # per step: ("all",) | ("dist", D) | ("random",)

    @property
    def N(self) -> int:
        return self.T * self.Hl * self.Wl

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def rope_dims(self):
        dh = dw = 2 * (self.d // 6)
        return self.d - dh - dw, dh, dw


def _sched_alternate(steps, D):
    return [("all",) if t % 2 == 0 else ("dist", D) for t in range(steps)]


def get(name: str) -> Workload:
    if name == "tiny_fp32":
        return Workload(name, 0, 1, 2, 64, 4, 16, 16, 4, "fp32", 2, 0.05,
                        schedule=[("all",), ("dist", 2)])
    if name == "small_bf16":
        return Workload(name, 1, 1, 12, 64, 4, 32, 32, 8, "bf16", 10, 0.02,
                        q_scale=1.0 / math.sqrt(64), softmax_scale=1.0,
                        schedule=_sched_alternate(10, 2))
    if name == "wan14b_layer":
        return Workload(name, 2, 1, 40, 128, 21, 30, 52, 8, "bf16", 4, 0.02, rope=True,
                        head_scales=True, schedule=[("all",)] + [("dist", 2)] * 3)
    if name == "long_720p":
        return Workload(name, 3, 1, 40, 128, 21, 45, 80, 16, "bf16", 8, 0.02, rope=True,
                        schedule=[("all",) if t % 4 == 0 else ("dist", 3) for t in range(8)])
    if name.startswith("sweep_P"):
        P = int(name[len("sweep_P"):])
        dmin = {4: 1, 8: 1, 16: 2}[P]
        sched = [("all",)] + [("dist", D) for D in range(P - 1, dmin - 1, -1)] + [("random",)]
        return Workload(name, 4, 1, 40, 128, 21, 30, 52, P, "bf16", len(sched), 0.0,
                        schedule=sched)
    raise KeyError(name)


def scaled(w: Workload, name: str, H=None, T=None, Hl=None, Wl=None, P=None, start_frame=None,
           steps=None) -> Workload:
    """A smaller workload of the same kind (for tests the oracle finishes in seconds)."""
    import copy

    s = copy.deepcopy(w)
    s.name = name
    for k, v in dict(H=H, T=T, Hl=Hl, Wl=Wl, P=P, start_frame=start_frame).items():
        if v is not None:
            setattr(s, k, v)
    if steps is not None:
        s.steps = steps
        s.schedule = s.schedule[:steps]
    return s


# ---------------------------------------------------------------------------------- masks
def distance_mask(P: int, D: int) -> np.ndarray:
    """Reuse pair (i, j) iff |i - j| >= D (D >= P: every pair computed)."""
    i, j = np.indices((P, P))
    return (np.abs(i - j) >= D).astype(np.uint8)


def splitmix64_stream(seed: int):
    state = seed & MASK64
    while True:
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def random_mask(P: int, seed: int, p_reuse: float = 0.5) -> np.ndarray:
    g = splitmix64_stream(seed)
    m = np.zeros((P, P), dtype=np.uint8)
    for i in range(P):
        for j in range(P):
            u = (next(g) >> 11) * 2.0 ** -53
            m[i, j] = 1 if (i != j and u < p_reuse) else 0
    return m


def step_mask(w: Workload, t: int) -> np.ndarray:
    kind = w.schedule[t]
    if kind[0] == "all":
        return np.zeros((w.P, w.P), dtype=np.uint8)
    if kind[0] == "dist":
        return distance_mask(w.P, kind[1])
    return random_mask(w.P, 1000 * w.index + 7 + w.P)


def reuse_fraction(mask: np.ndarray) -> float:
    return float(np.asarray(mask).mean())


# ---------------------------------------------------------------------------------- inputs
CHUNK = 1 << 22


def normal(seed, shape) -> np.ndarray:
    """float32 N(0, 1) values of `shape`: chunk m of CHUNK consecutive values (flat order) from
    numpy's PCG64 generator seeded with [*seed, m]; chunks are drawn on several threads."""
    seed = list(seed) if isinstance(seed, (list, tuple)) else [seed]
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(m):
        lo, hi = m * CHUNK, min(n, (m + 1) * CHUNK)
        np.random.default_rng(seed + [m]).standard_normal(hi - lo, dtype=np.float32,
                                                          out=out[lo:hi])

    workers = max(1, min(16, os.cpu_count() or 1, nchunks))
    if workers == 1:
        for m in range(nchunks):
            fill(m)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


class InputStream:
    """Yields (q, k, v) as float32 numpy arrays [B, N, H, d] holding config-dtype values."""

    def __init__(self, w: Workload, heads=None):
        self.w = w
        self.heads = None if heads is None else np.asarray(heads)
        shape = (w.B, w.N, w.H, w.d)
        c = w.index
        self.master = []
        for x in range(3):
            a = normal(1000 * c + 1 + x, shape)
            if x == 0 and w.q_scale != 1.0:
                a *= np.float32(w.q_scale)
            self.master.append(a)
        if w.head_scales:
            hs = np.random.default_rng(1000 * c + 50).uniform(0.5, 2.0, size=(3, w.H))
            for x in range(3):
                self.master[x] *= hs[x].astype(np.float32)[None, None, :, None]
        self.t = 0

    def _drift(self, t):
        w = self.w
        for x in range(3):
            dz = normal([1000 * w.index + 100 + t, x], self.master[x].shape)
            dz *= np.float32(w.drift)
            if x == 0 and w.q_scale != 1.0:
                dz *= np.float32(w.q_scale)
            self.master[x] += dz

    def next(self):
        """Inputs of the next step, rounded to the config dtype (as float32 arrays)."""
        if self.t > 0 and self.w.drift != 0.0:
            self._drift(self.t)
        self.t += 1
        out = []
        for a in self.master:
            if self.heads is not None:
                a = a[:, :, self.heads, :]
            out.append(round_to_dtype(a, self.w.dtype))
        return tuple(out)


def round_to_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp32":
        return np.ascontiguousarray(a, dtype=np.float32)
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float32).numpy()


def torch_dtype(w: Workload):
    import torch

    return torch.bfloat16 if w.dtype == "bf16" else torch.float32
