"""Runs a workload through the library (C ABI) and through the CPU oracle side by side.

The GPU computes every row of every step; the oracle computes a chosen set of query rows
(all rows at small sizes, sampled rows at full sizes). After each step this compares, for the
oracle's rows:
  * merged output and log-sum-exp;
  * the fresh state of every computed pair (the cache slot the step wrote);
  * that cache slots of reused pairs are bit-identical to before the step (reuse moves nothing);
  * the plan's bookkeeping (valid, step computed, steps run) against the oracle's, bit-exact.

Tolerances: fp32 workloads 1e-4 max-abs for outputs, states and lse; bf16 workloads 2e-2
max-abs for outputs and 1e-3 for lse. The cached per-pair states are internal bf16 values with
no stated tolerance; they are held to 2e-2 relative to max(1, |value|), i.e. the output
tolerance below magnitude 1 and bf16's relative resolution above it. The library's bf16 values are compared
with the oracle's unrounded fp64 values, so the library's own final rounding (at most half a
bf16 ulp) is part of the error; rounding the oracle as well would double the rounding error.
The oracle's merge itself reads its cache rounded to the cache dtype, as the library does.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import attention_state_reuse_gb300 as dt
import oracle
from attention_state_reuse_gb300 import workloads as wl

TOL = {"fp32": dict(out=1e-4, lse=1e-4), "bf16": dict(out=2e-2, lse=1e-3)}


def sample_rows(w: wl.Workload, heads_local, per_partition_random=3, seed=0):
    """Rows (b, h_local, r): partition edges, tile edges and a few random rows per partition."""
    off = oracle.partition_offsets(w.N, w.P)
    rng = np.random.default_rng(seed)
    rows = set()
    for i in range(w.P):
        n = off[i + 1] - off[i]
        cand = {0, n - 1, 127, 128, 255, 256, n - 128, n - 129}
        cand |= set(rng.integers(0, n, size=per_partition_random).tolist())
        for c in cand:
            if 0 <= c < n:
                for b in range(w.B):
                    for hl in heads_local:
                        rows.add((b, hl, int(off[i] + c)))
    return sorted(rows)


class ParityRun:
    def __init__(self, w: wl.Workload, heads=None, rows=None, device="cuda", nthreads=None,
                 strided=False, group=False):
        self.w = w
        self.strided = strided  # inputs and output as views into buffers with 3 spare heads
        self.device = device
        self.dtype = wl.torch_dtype(w)
        self.heads = list(range(w.H)) if heads is None else list(heads)
        self.stream = wl.InputStream(w)
        N, P, B, H, d = w.N, w.P, w.B, w.H, w.d
        self.plan = dt.Plan(N, P)
        self.cO, self.cL = dt.new_state_cache(B, H, P, N, d, self.dtype, device)
        self.cO.zero_()
        self.cL.zero_()
        # optional group states (one composed state per row over its partition's reused pairs);
        # filled with NaN so that a group state the library failed to build shows up
        self.group = dt.new_group_state(B, H, N, d, device) if group else None
        if self.group is not None:
            self.group[0].fill_(float("nan"))
            self.group[1].fill_(float("nan"))
        self.out = self._alloc((B, N, H, d))
        self.out_lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
        self.rope = None
        rope_cfg = None
        if w.rope:
            dtt, dhh, dww = w.rope_dims
            self.rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                                      start_frame=w.start_frame, device=device)
            rope_cfg = dict(Hl=w.Hl, Wl=w.Wl, start_frame=w.start_frame, dt=dtt, dh=dhh, dw=dww)
        nbytes = dt.workspace_size(self.plan, B, H, d, self.dtype, w.rope)
        self.ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
        if rows is None:
            rows = [(b, hl, r) for b in range(B) for hl in range(len(self.heads)) for r in range(N)]
        self.rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
        rnd = oracle.ROUND_BF16 if w.dtype == "bf16" else oracle.ROUND_F32
        self.orc = oracle.OracleRun(B, N, len(self.heads), d, P, w.scale, rows=self.rows,
                                    cache_round=rnd, input_round=rnd, rope=rope_cfg,
                                    nthreads=nthreads)
        self.t = 0
        # index tensors of the oracle's rows inside the GPU tensors
        self.b_idx = torch.as_tensor(self.rows[:, 0], device=device)
        self.h_idx = torch.as_tensor(np.asarray(self.heads)[self.rows[:, 1]], device=device)
        self.r_idx = torch.as_tensor(self.rows[:, 2], device=device)
        self.part = np.searchsorted(self.orc.offsets, self.rows[:, 2], side="right") - 1

    def _alloc(self, shape):
        B, N, H, d = shape
        if not self.strided:
            return torch.empty(shape, dtype=self.dtype, device=self.device)
        return torch.empty((B, N, H + 3, d), dtype=self.dtype, device=self.device)[:, :, 1:H + 1]

    def _to_dev(self, a):
        x = self._alloc(a.shape)
        x.copy_(torch.from_numpy(a))
        return x

    def gather_cache(self):
        """Cache slots [rows, P, d] and [rows, P] of the oracle's rows."""
        pj = torch.arange(self.w.P, device=self.device)[None, :]
        b, h, r = self.b_idx[:, None], self.h_idx[:, None], self.r_idx[:, None]
        O = self.cO[b, h, pj, r]
        L = self.cL[b, h, pj, r]
        return O.float().cpu().numpy(), L.cpu().numpy()

    def step(self, mask=None, check=True):
        w = self.w
        if mask is None:
            mask = wl.step_mask(w, self.t)
        q, k, v = self.stream.next()
        before = self.gather_cache() if check else None
        dt.attn_step(self.plan, self._to_dev(q), self._to_dev(k), self._to_dev(v), self.cO,
                     self.cL, self.out, self.out_lse, reuse_mask=mask, rope=self.rope,
                     softmax_scale=w.scale, workspace=self.ws, group=self.group)
        torch.cuda.synchronize()
        st = dt.device_status()
        assert st == (0, 0), f"device status {st}"
        self.t += 1
        if not check:
            return None
        hs = self.heads
        res = self.orc.step(q[:, :, hs], k[:, :, hs], v[:, :, hs], mask)
        return self.compare(res, before, mask)

    def compare(self, res, before, mask):
        w = self.w
        tol = TOL[w.dtype]
        out = self.out[self.b_idx, self.r_idx, self.h_idx].float().cpu().numpy()
        lse = self.out_lse[self.b_idx, self.h_idx, self.r_idx].cpu().numpy()
        ref_out = res["out"]
        err = {"out": float(np.abs(out - ref_out).max()),
               "lse": float(np.abs(lse - res["out_lse"]).max())}
        O_after, L_after = self.gather_cache()
        comp = mask[self.part] == 0            # [rows, P] computed pairs of each row
        e_state = (np.abs(O_after - res["fresh_O"]) / np.maximum(1.0, np.abs(res["fresh_O"])))[comp]
        e_lse = np.abs(L_after - res["fresh_lse"])[comp]
        err["state_O"] = float(e_state.max()) if e_state.size else 0.0
        err["state_lse"] = float(e_lse.max()) if e_lse.size else 0.0
        reused = ~comp
        err["reused_changed"] = int((O_after[reused] != before[0][reused]).sum() +
                                    (L_after[reused] != before[1][reused]).sum())
        valid, sc, steps = self.plan.cache_state()
        book = self.orc.book
        err["book_equal"] = bool((valid.astype(bool) == book.valid).all() and
                                 (sc == book.step_computed).all() and steps == book.step)
        ok = (err["out"] <= tol["out"] and err["lse"] <= tol["lse"] and
              err["state_O"] <= tol["out"] and err["state_lse"] <= tol["lse"] and
              err["reused_changed"] == 0 and err["book_equal"])
        err["ok"] = ok
        err["step"] = self.t - 1
        err["workload"] = w.name
        log = os.environ.get("DITANGO_PARITY_LOG")
        if log:
            with open(log, "a") as f:
                f.write(json.dumps(err) + "\n")
        return err
