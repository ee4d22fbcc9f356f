#!/usr/bin/env python3
"""Benchmark: one attention-layer step of partitioned attention with attention-state reuse.

Workload (default): the long 720p-shaped layer - B=1, H=40, d=128, bf16, N=75600 tokens
(21x45x80 latent), P=16 contiguous partitions, 3D RoPE (t/h/w split 44/42/42) with a global
time index; the timed step reuses every pair with |i-j| >= 3 (182 of 256 pairs) after an
all-compute anchor step filled the state cache. A step is one call of ditango_attn_step: RoPE of
k (q is rotated inside the pair kernel), fresh states of the 74 computed pairs, merge of every
row's computed states with its group state (the composed state of its reused pairs). Inputs are
synthetic (seeded) and resident in HBM before timing; they are larger than L2 (774 MB per
tensor), so no L2 flush is needed between steps. `--workload wan14b_layer` times the
Wan2.1-14B-shaped layer (N=32760, P=8) instead.

Prints one JSON line: ms per step (lower is better) plus effective TFLOP/s counted over
computed pairs only, the pair kernel's roofline against the measured tensor-core peak, its SFU
rate, the merge's roofline against the measured copy bandwidth, the step's roofline time,
per-kernel times, the anchor and the first reuse step after it, a whole schedule cycle
(anchor + reuse steps) against computing every pair, the reuse-fraction sweep, the cycle with
the far states in host storage, an end-to-end number with host buffers, clocks, and the CPU
oracle baseline.

With --gpus N (under torchrun) the layer's heads are split across the ranks: rank r computes
heads [r*H/N, (r+1)*H/N) of the same layer (every (b, h) is independent, so no data crosses
ranks) and the line reports the whole layer's step time, the maximum over ranks.

`--impl reference` times the CPU oracle instead (a fixed sample of rows per step, extrapolated
to the full step) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms/attention-layer step and effective TFLOP/s vs reuse fraction (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def pair_flops(w, mask):
    """4 * B * H * n_i * n_j * d summed over computed pairs (QK^T and PV, 2 flops per MAC)."""
    import numpy as np

    off = np.array([(w.N // w.P) * p + min(p, w.N % w.P) for p in range(w.P + 1)])
    n = np.diff(off)
    comp = (np.asarray(mask) == 0)
    return float(4.0 * w.B * w.H * w.d * (n[:, None] * n[None, :] * comp).sum())


def merge_bytes(w, mask, group):
    """Algorithmic traffic of a step's merge: per query row of partition i, read its cache
    states (O in the cache dtype + fp32 lse): the computed ones, and the reused ones unless a
    group state (fp32 O + lse) stands for them; write out and out_lse. Group states are built
    only when the reused sets change, so the steady-state step does not count that build."""
    import numpy as np

    esz = 2 if w.dtype == "bf16" else 4
    st = w.d * esz + 4
    mask = np.asarray(mask)
    off = np.array([0] + list(np.cumsum([len(a) for a in np.array_split(np.arange(w.N), w.P)])))
    total = 0
    for i in range(w.P):
        reused = int(mask[i].sum())
        reads = (w.P - reused) * st + ((w.d * 4 + 4) if (group and reused) else reused * st)
        total += int(off[i + 1] - off[i]) * (reads + st)
    return float(w.B * w.H * total)


def src_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PAIR_SRC = ["attention_state_reuse_gb300/csrc/pair_tc.cu",
            "attention_state_reuse_gb300/csrc/ptx_sm103.cuh",
            "attention_state_reuse_gb300/csrc/rope_round.cuh"]


def profiled_traffic(workload, heads):
    """DRAM bytes per pair-kernel launch from a committed ncu summary, if it still applies:
    same kernel sources and workload; scaled from the captured head count to `heads` (every
    (b, h) reads its own q, k, v once and writes its own states)."""
    p = os.path.join(ROOT, "profiles", "pair_tc_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("src_sha") != src_hash(PAIR_SRC) or rec.get("workload") != workload:
        return None
    per_head = rec.get("traffic_bytes_per_head")
    return None if per_head is None else int(round(per_head * heads))


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 - 0.05 <= t <= t1 + 0.05] or \
               [s for (_, s) in self.samples]
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = max(smax, float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# dense bf16 tcgen05 rate of one SM: a 128x128x16 MMA (2^19 flops) every 64 cycles, measured
# with MMAs issued back to back on this GPU
DENSE_BF16_FLOP_PER_CLK_SM = 8192
# SFU exponentials of one SM per clock (ex2.approx, fp32 and bf16x2 alike), measured with a
# throughput loop on this GPU; the softmax takes one per score
SFU_EXP2_PER_CLK_SM = 32


def head_range(rank, world, H):
    """Heads [h0, h1) that rank `rank` computes when the layer's H heads are split over `world`
    ranks: contiguous ranges, the first H mod world ranks one head longer."""
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def mask_name(w):
    kind = w.schedule[1]
    return f"|i-j|>={kind[1]}" if kind[0] == "dist" else kind[0]


def config_of(w, world):
    """The `config` of the JSON line (the same for both arms)."""
    import numpy as np

    from attention_state_reuse_gb300 import workloads as wl

    esz = 2 if w.dtype == "bf16" else 4
    tensor_mb = w.B * w.N * w.H * w.d * esz / 1e6
    return {"workload": w.name, "B": w.B, "N": w.N, "H": w.H, "d": w.d, "P": w.P,
            "latent": [w.T, w.Hl, w.Wl], "rope": w.rope, "reuse_mask": mask_name(w),
            "reuse_fraction": round(float(np.asarray(wl.step_mask(w, 1)).mean()), 4),
            "parallelism": "1 GPU" if world == 1 else f"heads split over {world} GPUs",
            "l2": f"inputs larger than L2 ({tensor_mb:.0f} MB per tensor); no flush"}


# ------------------------------------------------------------------------------ our library
def run_ours(args, w, rank, world):
    import numpy as np
    import torch

    import attention_state_reuse_gb300 as dt
    from attention_state_reuse_gb300 import workloads as wl

    dt.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dtype = wl.torch_dtype(w)
    # this rank's heads of the layer (all of them on one GPU)
    h0, h1 = head_range(rank, world, w.H)
    B, N, H, d, P = w.B, w.N, h1 - h0, w.d, w.P
    stream = wl.InputStream(w)
    q_np, k_np, v_np = (np.ascontiguousarray(a[:, :, h0:h1]) for a in stream.next())
    to_dev = lambda a: torch.from_numpy(a).to(dev).to(dtype)
    q, k, v = to_dev(q_np), to_dev(k_np), to_dev(v_np)
    mask = wl.step_mask(w, 1)  # the steady-state reuse step of the workload's schedule
    # the plan's default mask is the steady reuse mask: the anchor's merge then builds the
    # group states that the reuse steps after it read
    plan = dt.Plan(N, P, mask=mask)
    cO, cL = dt.new_state_cache(B, H, P, N, d, dtype, dev)
    out = torch.empty((B, N, H, d), dtype=dtype, device=dev)
    out_lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    rope = None
    if w.rope:
        dtt, dhh, dww = w.rope_dims
        rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                             start_frame=w.start_frame, device=dev)
    ws = torch.empty(max(1, dt.workspace_size(plan, B, H, d, dtype, w.rope)), dtype=torch.uint8,
                     device=dev)
    group = dt.new_group_state(B, H, N, d, dev) if args.group else None
    anchor = np.zeros((P, P), np.uint8)
    step = lambda m: dt.attn_step(plan, q, k, v, cO, cL, out, out_lse, reuse_mask=m, rope=rope,
                                  softmax_scale=w.scale, workspace=ws, group=group)

    # anchor step (all pairs computed) fills the cache; time a few anchors for context
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    step(anchor)
    torch.cuda.synchronize()
    anchor_ms = []
    for _ in range(3):
        ev[0].record()
        step(anchor)
        ev[1].record()
        torch.cuda.synchronize()
        anchor_ms.append(ev[0].elapsed_time(ev[1]))
    # the first reuse step after an anchor, timed on its own: it finds the group states that
    # the anchor built current; its kernels are timed too
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(3)]
    for evs in fev:
        for e in evs:
            e.record()
    torch.cuda.synchronize()
    ev[0].record()
    plan.set_profile_events(fev[0])
    step(mask)
    plan.set_profile_events(None)
    ev[1].record()
    torch.cuda.synchronize()
    first_reuse_ms = ev[0].elapsed_time(ev[1])
    for _ in range(args.warmup):
        step(mask)
    torch.cuda.synchronize()
    st = dt.device_status()
    if st != (0, 0):
        raise RuntimeError(f"device status after warm-up: {st}")

    # timed region: exactly K steps, per-kernel events recorded by the library
    K = args.steps
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for evs in kev:  # torch creates the CUDA event at its first record
        for e in evs:
            e.record()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record()
    for s in range(K):
        plan.set_profile_events(kev[s])
        step(mask)
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    plan.set_profile_events(None)
    clocks.stop()
    st = dt.device_status()
    if st != (0, 0):
        raise RuntimeError(f"device status after timed steps: {st}")
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world)
    ms = total_ms / K
    rope_ms = statistics.mean(kev[s][0].elapsed_time(kev[s][1]) for s in range(K))
    pair_ms = statistics.mean(kev[s][1].elapsed_time(kev[s][2]) for s in range(K))
    merge_ms = statistics.mean(kev[s][2].elapsed_time(kev[s][3]) for s in range(K))

    # end to end through the public call with host buffers, pipelined the way a serving loop
    # runs it: every step copies its q, k, v from pinned host memory (one copy stream each) into
    # one of two device input sets while the step before computes, and reads its out and
    # out_lse back into pinned host memory (a fourth stream) while the step after computes. Every step still
    # moves its full inputs and outputs; the timed region runs from the first copy to the last
    # read-back.
    hq, hk, hv = (torch.from_numpy(a).to(dtype).pin_memory() for a in (q_np, k_np, v_np))
    ho = [torch.empty(out.shape, dtype=dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(out_lse.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    inbuf = [(q, k, v), tuple(torch.empty_like(x) for x in (q, k, v))]
    outbuf = [(out, out_lse), (torch.empty_like(out), torch.empty_like(out_lse))]
    comp = torch.cuda.current_stream(dev)
    h2d_s = [torch.cuda.Stream(dev) for _ in range(3)]  # q, k, v copied side by side
    d2h_s = torch.cuda.Stream(dev)
    e2e_steps = max(3, min(K, 20))

    def e2e_run(nsteps, start_event=None):
        done, read = [], []
        for st in range(nsteps):
            b = st % 2
            for dst, src, cs in zip(inbuf[b], (hq, hk, hv), h2d_s):
                copied = torch.cuda.Event()
                with torch.cuda.stream(cs):
                    if st == 0 and start_event is not None:
                        cs.wait_event(start_event)
                    if st >= 2:
                        cs.wait_event(done[st - 2])  # step st-2 has finished reading set b
                    dst.copy_(src, non_blocking=True)
                    copied.record(cs)
                comp.wait_event(copied)
            if st >= 2:
                comp.wait_event(read[st - 2])  # output set b has been read back
            qb, kb, vb = inbuf[b]
            dt.attn_step(plan, qb, kb, vb, cO, cL, outbuf[b][0], outbuf[b][1], reuse_mask=mask,
                         rope=rope, softmax_scale=w.scale, workspace=ws, group=group, stream=comp)
            ev = torch.cuda.Event()
            ev.record(comp)
            done.append(ev)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev)
                ho[b].copy_(outbuf[b][0], non_blocking=True)
                hl[b].copy_(outbuf[b][1], non_blocking=True)
                rv = torch.cuda.Event()
                rv.record(d2h_s)
            read.append(rv)
        return read[-1]

    comp.wait_event(e2e_run(3))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    last = e2e_run(e2e_steps, start_event=e0)
    comp.wait_event(last)
    e1.record(comp)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    # two more (anchor, first reuse step) cycles: first_reuse_step_ms is the median of three
    first_reuse = [first_reuse_ms]
    for c in range(2):
        step(anchor)
        ev[0].record()
        plan.set_profile_events(fev[c + 1])
        step(mask)
        plan.set_profile_events(None)
        ev[1].record()
        torch.cuda.synchronize()
        first_reuse.append(ev[0].elapsed_time(ev[1]))
    first_reuse_ms = statistics.median(first_reuse)
    first_kernel_ms = {name: round(statistics.median(fev[c][x].elapsed_time(fev[c][x + 1])
                                                     for c in range(3)), 4)
                       for x, name in enumerate(("rope", "pair", "merge"))}
    # two cycles of the workload's schedule (an anchor, then reuse steps until the next one),
    # each timed as a whole: the mean step over a cycle, against computing every pair each step
    sched = [wl.step_mask(w, t) for t in range(len(w.schedule))]
    period = next((t for t in range(1, len(sched)) if not sched[t].any()), len(sched))
    cycle_ms = []
    for _ in range(2):
        ev[0].record()
        for t in range(period):
            step(sched[t])
        ev[1].record()
        torch.cuda.synchronize()
        cycle_ms.append(ev[0].elapsed_time(ev[1]) / period)
    cycle = statistics.mean(cycle_ms)
    esz = 2 if dtype == torch.bfloat16 else 4
    # bytes of the whole job (every rank copies its own heads)
    h2d = 3 * B * N * w.H * d * esz
    d2h = B * N * w.H * d * esz + B * w.H * N * 4

    sweep = reuse_sweep(dev, use_group=args.group) if (args.sweep and world == 1) else None
    offload = offload_cycle(w, q, k, v, dev) if (args.offload and world == 1) else None
    planned = planner_cycle(w, q, k, v, dev) if (args.sweep and world == 1) else None

    flops = pair_flops(w, mask)            # the whole layer
    flops_rank = flops * H / w.H           # this rank's heads
    peaks, peak_src = load_peaks()
    tc_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tc_sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    achieved = flops_rank / (pair_ms * 1e-3) / 1e12
    mbytes = merge_bytes(w, mask, args.group) * H / w.H
    merge_gbs = mbytes / (merge_ms * 1e-3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    ck = clocks.summary(wall0, wall1)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = ck["sm_max_mhz"] or peaks.get("sm_max_mhz", 2070.0)
    med_mhz = ck["sm_mhz"] or max_mhz
    # the pair kernel's head-dim-64 build (SFU rate taken at the timed region's median clock)
    d64 = head_dim_64(dev, med_mhz) if (args.sweep and world == 1) else None
    dense = lambda mhz: n_sm * DENSE_BF16_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12
    exps_rank = flops_rank / (4 * d)  # one exponential per score
    sfu_rate = exps_rank / (pair_ms * 1e-3 * med_mhz * 1e6 * n_sm)
    rope_bytes = (2 * B * N * H * d * (2 if dtype == torch.bfloat16 else 4)) if w.rope else 0
    t_min_ms = (flops_rank / (tc_burst * 1e12) + (mbytes + rope_bytes) / (hbm * 1e9)) * 1e3
    timed_s = total_ms / 1e3
    line = {
        "metric": METRIC, "value": round(ms, 4), "unit": "ms", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": False,
        "scaling": "strong", "vs_baseline": None,
        "dtype": "bf16" if dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) inputs" + (", per-head scales U(0.5,2)" if w.head_scales
                                                     else "") + "; no weights)",
        "config": config_of(w, world),
        "effective_tflops": round(flops / (ms * 1e-3) / 1e12, 2),  # the whole layer
        "pair_flops_per_step": flops,
        "heads_per_rank": H,
        "kernel_ms": {"rope": round(rope_ms, 4), "pair": round(pair_ms, 4),
                      "merge": round(merge_ms, 4)},
        "anchor_ms": round(statistics.median(anchor_ms), 4),
        "first_reuse_step_ms": round(first_reuse_ms, 4),
        "first_reuse_kernel_ms": first_kernel_ms,
        "schedule_cycle": {"period": period, "ms_per_step": round(cycle, 4),
                           "dense_ms_per_step": round(statistics.median(anchor_ms), 4),
                           "speedup_vs_dense": round(statistics.median(anchor_ms) / cycle, 3)},
        "group_states": bool(args.group),
        "anchor_effective_tflops": round(pair_flops(w, anchor) / (statistics.median(anchor_ms) * 1e-3) / 1e12, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": tc_burst,
                     "unit": "TFLOP/s", "frac": round(achieved / tc_burst, 4),
                     "traffic": profiled_traffic(w.name, H),
                     "kernel": "pair_tc_kernel<128>",
                     "peak_source": (f"bf16_tflops (burst) of {peak_src}: the timed region lasts "
                                     f"{timed_s:.2f} s at a {med_mhz:.0f} MHz median SM clock"),
                     "frac_of_sustained": round(achieved / tc_sustained, 4),
                     "dense_peak_at_median_clock": round(dense(med_mhz), 1),
                     "frac_of_dense_at_median_clock": round(achieved / dense(med_mhz), 4),
                     "dense_peak_at_max_clock": round(dense(max_mhz), 1),
                     "frac_of_dense_at_max_clock": round(achieved / dense(max_mhz), 4),
                     "dense_rate": f"{n_sm} SMs x {DENSE_BF16_FLOP_PER_CLK_SM} bf16 flop/clk "
                                   "(a 128x128x16 tcgen05.mma every 64 cycles, measured)"},
        "sfu": {"exps_per_launch": exps_rank,
                "achieved_per_clk_per_sm": round(sfu_rate, 2),
                "peak_per_clk_per_sm": SFU_EXP2_PER_CLK_SM,
                "frac": round(sfu_rate / SFU_EXP2_PER_CLK_SM, 4),
                "clock": "sampled median SM clock of the timed region"},
        "step_roofline": {"t_min_ms": round(t_min_ms, 4), "frac": round(t_min_ms / ms, 4),
                          "sum_of": "pair flops at the measured bf16 burst rate + merge and "
                                    "RoPE (k read and written) bytes at the measured copy "
                                    "bandwidth"},
        "merge_roofline": {"bound": "hbm", "achieved": round(merge_gbs, 1), "peak": hbm,
                           "unit": "GB/s", "frac": round(merge_gbs / hbm, 4),
                           "frac_of_8tbs": round(merge_gbs / 8000.0, 4),
                           "bytes_per_launch": mbytes},
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": h2d,
                "pipelined": "each step's H2D and D2H overlap the neighbouring steps' compute",
                "d2h_bytes_per_step": d2h},
        "gpu_launches": world * K * (3 if w.rope else 2),  # all ranks
        "reuse_sweep": sweep,
        "head_dim_64": d64,
        "host_storage": offload,
        "planner": planned,
        "clocks": ck,
    }
    return line


def offload_cycle(w, q, k, v, dev, cycles=2):
    """The workload's step schedule with the far pairs' states in host memory.

    The device cache keeps S = 2D - 1 slots per row (D: the schedule's reuse distance), the
    pairs a steady step computes; the other states live in page-locked host memory and are
    written there by the anchor steps and read back by the group-state rebuilds. Times one
    schedule cycle (anchor, first reuse step, steady reuse steps) after a warm-up cycle, and
    reports the device bytes of the cache with and without host storage.
    """
    import numpy as np
    import torch

    import attention_state_reuse_gb300 as dt
    from attention_state_reuse_gb300 import workloads as wl

    kind = w.schedule[1]
    if kind[0] != "dist":
        return None
    D = kind[1]
    B, N, H, d, P = w.B, w.N, q.shape[2], w.d, w.P
    S = min(P, 2 * D - 1)
    dtype = q.dtype
    plan = dt.Plan(N, P)
    cO, cL = dt.new_state_cache(B, H, S, N, d, dtype, dev)
    host = dt.new_host_states(B, H, P, N, d, dtype)
    group = dt.new_group_state(B, H, N, d, dev)
    out = torch.empty_like(q)
    out_lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    rope = None
    if w.rope:
        dtt, dhh, dww = w.rope_dims
        rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                             start_frame=w.start_frame, device=dev)
    ws = torch.empty(max(1, dt.workspace_size(plan, B, H, d, dtype, w.rope)), dtype=torch.uint8,
                     device=dev)
    sched = [wl.step_mask(w, t) for t in range(len(w.schedule))]
    plan.set_mask(sched[1])  # the anchors build the reuse steps' group states
    period = next((t for t in range(1, len(sched)) if not sched[t].any()), len(sched))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(period + 1)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(period)]
    for evs in kev:  # torch creates the CUDA event at its first record
        for e in evs:
            e.record()
    times = []
    for c in range(cycles):
        ev[0].record()
        for t in range(period):
            plan.set_profile_events(kev[t])
            dt.attn_step(plan, q, k, v, cO, cL, out, out_lse, reuse_mask=sched[t], rope=rope,
                         softmax_scale=w.scale, workspace=ws, group=group, host=host)
            ev[t + 1].record()
        plan.set_profile_events(None)
        torch.cuda.synchronize()
        times = [ev[t].elapsed_time(ev[t + 1]) for t in range(period)]
    split = lambda t: {name: round(kev[t][x].elapsed_time(kev[t][x + 1]), 4)
                       for x, name in enumerate(("rope", "pair", "merge"))}
    st = dt.device_status()
    if st != (0, 0):
        raise RuntimeError(f"device status after the host-storage cycle: {st}")
    esz = 2 if dtype == torch.bfloat16 else 4
    per_slot = B * H * N * (d * esz + 4)
    return {"device_slots_per_row": S, "partitions": P,
            "cache_device_bytes_resident": P * per_slot,
            "cache_device_bytes_with_host_storage": S * per_slot,
            "device_bytes_saved": (P - S) * per_slot,
            "host_bytes": P * per_slot,
            "anchor_ms": round(times[0], 4), "anchor_kernel_ms": split(0),
            "first_reuse_step_ms": round(times[1], 4),
            "steady_step_ms": round(statistics.median(times[2:]), 4) if period > 2 else None,
            "ms_per_step_over_cycle": round(sum(times) / period, 4),
            "schedule": f"anchor every {period} steps, |i-j|>={D} reused"}


def head_dim_64(dev, med_mhz, steps=10):
    """The pair kernel at head dim 64 (its other build): N = 32760 (21x30x52), H = 40, d = 64,
    bf16, P = 8, no RoPE, |i - j| >= 2 reused, group states on; seeded N(0,1) inputs. At d = 64
    a tile's P V and Q K^T take half the tensor time of d = 128 while its softmax (one SFU
    exponential per score) stays the same, so the SFU rate is reported beside the tensor one."""
    import numpy as np
    import torch

    import attention_state_reuse_gb300 as dt
    from attention_state_reuse_gb300 import workloads as wl

    w = wl.Workload("d64_layer", 5, 1, 40, 64, 21, 30, 52, 8, "bf16", 2, 0.0,
                    schedule=[("all",), ("dist", 2)])
    q, k, v = (torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in wl.InputStream(w).next())
    out = torch.empty_like(q)
    out_lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    mask = wl.distance_mask(w.P, 2)
    plan = dt.Plan(w.N, w.P, mask=mask)
    cO, cL = dt.new_state_cache(w.B, w.H, w.P, w.N, w.d, torch.bfloat16, dev)
    grp = dt.new_group_state(w.B, w.H, w.N, w.d, dev)
    step = lambda m: dt.attn_step(plan, q, k, v, cO, cL, out, out_lse, reuse_mask=m,
                                  softmax_scale=w.scale, group=grp)
    step(np.zeros((w.P, w.P), np.uint8))
    step(mask)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for evs in kev:
        for e in evs:
            e.record()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for x in range(steps):
        plan.set_profile_events(kev[x])
        step(mask)
    t1.record()
    plan.set_profile_events(None)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    pair_ms = statistics.median(kev[x][1].elapsed_time(kev[x][2]) for x in range(steps))
    f = pair_flops(w, mask)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks, _ = load_peaks()
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tflops = f / (pair_ms * 1e-3) / 1e12
    sfu = f / (4 * w.d) / (pair_ms * 1e-3 * med_mhz * 1e6 * n_sm)
    return {"workload": "N=32760 (21x30x52), H=40, d=64, P=8, bf16, no RoPE, |i-j|>=2 reused",
            "ms": round(ms, 4), "pair_ms": round(pair_ms, 4), "pair_tflops": round(tflops, 1),
            "pair_frac_of_burst": round(tflops / burst, 4),
            "sfu_per_clk_per_sm": round(sfu, 2),
            "sfu_frac": round(sfu / SFU_EXP2_PER_CLK_SM, 4)}


def planner_cycle(w, q, k, v, dev, cycles=2, anchor_every=4, tau=1e-3, group=2, sigma=0.02):
    """The anchor-guided planner driving the layer: AnchorPlanner chooses every step's mask
    (anchors every `anchor_every` steps, threshold tau, groups of `group` KV partitions) while
    the inputs drift, x_t = x_0 + sigma * t * eps (eps ~ N(0,1), seeded, made on the device
    before timing). Times `cycles` cycles as a whole (CUDA events and the host clock: the
    planner reads the drift back to the host each step), and each planner part once: the
    anchor's importance and snapshot, the per-step drift and the host selection."""
    import numpy as np
    import torch

    import attention_state_reuse_gb300 as dt

    B, N, H, d, P = w.B, w.N, q.shape[2], w.d, w.P
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 * w.index + 900)
    steps = cycles * anchor_every
    eps = [torch.randn(q.shape, generator=gen, device=dev, dtype=torch.float32) for _ in range(3)]
    drifted = [[(x.float() + sigma * t * e).to(q.dtype) for x, e in zip((q, k, v), eps)]
               for t in range(anchor_every)]
    del eps
    plan = dt.Plan(N, P)
    cO, cL = dt.new_state_cache(B, H, P, N, d, q.dtype, dev)
    grp = dt.new_group_state(B, H, N, d, dev)
    out = torch.empty_like(q)
    out_lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    rope = None
    if w.rope:
        dtt, dhh, dww = w.rope_dims
        rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                             start_frame=w.start_frame, device=dev)
    ws = torch.empty(max(1, dt.workspace_size(plan, B, H, d, q.dtype, w.rope)), dtype=torch.uint8,
                     device=dev)
    ap = dt.AnchorPlanner(plan, cO, cL, anchor_every=anchor_every, tau=tau, group=group)

    def run(n):
        fracs = []
        for t in range(n):
            m = ap.mask()
            qq, kk, vv = drifted[t % anchor_every]
            dt.attn_step(plan, qq, kk, vv, cO, cL, out, out_lse, reuse_mask=m, rope=rope,
                         softmax_scale=w.scale, workspace=ws, group=grp)
            ap.after_step(m)
            fracs.append(float(np.asarray(m).mean()))
        return fracs

    run(steps)  # warm-up cycles (the planner's first anchor has no prediction yet)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    e0.record()
    fracs = run(steps)
    e1.record()
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - h0) * 1e3 / steps
    dev_ms = e0.elapsed_time(e1) / steps
    st = dt.device_status()
    if st != (0, 0):
        raise RuntimeError(f"device status after the planner cycle: {st}")

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        r = fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b), r

    reps = 10  # back to back, so that the host's launch work overlaps the device's
    imp_ms, wgt = timed(lambda: [dt.planner_importance(plan, cO, cL) for _ in range(reps)][-1])
    snap_ms, _ = timed(lambda: [dt.planner_snapshot(plan, cO, cL, ap.snapshot)
                                for _ in range(reps)])
    drift_ms, delta = timed(lambda: [dt.planner_drift(plan, cO, cL, ap.snapshot)
                                     for _ in range(reps)][-1])
    imp_ms, snap_ms, drift_ms = imp_ms / reps, snap_ms / reps, drift_ms / reps
    wn, dn = wgt.cpu().numpy(), delta.cpu().numpy()
    h0 = time.perf_counter()
    dt.planner_select(plan, wn, dn, tau, group)
    select_ms = (time.perf_counter() - h0) * 1e3
    return {"anchor_every": anchor_every, "tau": tau, "group": group, "drift_sigma": sigma,
            "ms_per_step": round(dev_ms, 4), "wall_ms_per_step": round(wall_ms, 4),
            "reuse_fraction_per_step": [round(f, 4) for f in fracs[:anchor_every]],
            "importance_ms": round(imp_ms, 4), "snapshot_ms": round(snap_ms, 4),
            "drift_ms": round(drift_ms, 4), "select_host_ms": round(select_ms, 4)}


def reuse_sweep(dev, steps=10, use_group=True):
    """Step time against the fraction of reused pairs (the reuse-fraction sweep workload).

    N = 32760 (21x30x52 latent), H = 40, d = 128, bf16, P in {4, 8, 16}, no RoPE, seeded
    N(0,1) inputs. Masks: every distance threshold |i - j| >= D from D = P (all pairs
    computed) down to the smallest D with at most 87.5% of pairs reused, plus the seeded random
    mask (reuse probability 0.5, local pairs always computed). After an all-compute anchor
    step, each mask is timed over `steps` steps (CUDA events, inputs larger than L2). Reports
    ms/step, effective TFLOP/s over computed pairs, the pair kernel's time, and per P a
    least-squares fit ms = a * computed_fraction + b with its R^2. With group states (default)
    the untimed first step of each mask builds them and the timed steps reuse them.
    """
    import numpy as np
    import torch

    import attention_state_reuse_gb300 as dt
    from attention_state_reuse_gb300 import workloads as wl

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record()
    w0 = wl.get("sweep_P8")
    q, k, v = (torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in wl.InputStream(w0).next())
    out = torch.empty_like(q)
    out_lse = torch.empty((w0.B, w0.H, w0.N), dtype=torch.float32, device=dev)
    result = {}
    for P in (4, 8, 16):
        w = wl.get(f"sweep_P{P}")
        plan = dt.Plan(w.N, P)
        cO, cL = dt.new_state_cache(w.B, w.H, P, w.N, w.d, torch.bfloat16, dev)
        grp = dt.new_group_state(w.B, w.H, w.N, w.d, dev) if use_group else None
        step = lambda m: dt.attn_step(plan, q, k, v, cO, cL, out, out_lse, reuse_mask=m,
                                      softmax_scale=w.scale, group=grp)
        masks = []
        for kind in w.schedule:
            if kind[0] == "all":
                masks.append(("all computed", wl.distance_mask(P, P)))
            elif kind[0] == "dist":
                masks.append((f"|i-j|>={kind[1]}", wl.distance_mask(P, kind[1])))
            else:
                masks.append(("random p=0.5", wl.random_mask(P, 1000 * w.index + 7 + P)))
        step(masks[0][1])  # anchor
        rows = []
        for name, m in masks:
            step(m)
            torch.cuda.synchronize()
            plan.set_profile_events(evs)
            t0.record()
            for _ in range(steps):
                step(m)
            t1.record()
            torch.cuda.synchronize()
            pair_ms = evs[1].elapsed_time(evs[2])  # last step's pair kernel
            plan.set_profile_events(None)
            ms = t0.elapsed_time(t1) / steps
            f = pair_flops(w, m)
            rows.append({"mask": name, "reuse_fraction": round(float(np.asarray(m).mean()), 4),
                         "ms": round(ms, 4), "effective_tflops": round(f / (ms * 1e-3) / 1e12, 1),
                         "pair_ms": round(pair_ms, 4),
                         "pair_tflops": round(f / (pair_ms * 1e-3) / 1e12, 1)})
        dist = [r for r in rows if r["mask"] != "random p=0.5"]
        comp = np.array([1.0 - r["reuse_fraction"] for r in dist])
        msv = np.array([r["ms"] for r in dist])
        a, b = np.polyfit(comp, msv, 1)
        pred = a * comp + b
        r2 = 1.0 - ((msv - pred) ** 2).sum() / max(((msv - msv.mean()) ** 2).sum(), 1e-12)
        result[f"P{P}"] = {"points": rows,
                           "fit": {"ms_per_computed_fraction": round(float(a), 4),
                                   "ms_at_full_reuse": round(float(b), 4), "r2": round(float(r2), 5)}}
        del cO, cL, grp, plan
        torch.cuda.empty_cache()
    return result


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    """The largest of every rank's x (a timing), on the process group's own device."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ CPU oracle
SAMPLE_ROWS = 12288  # query rows of head 0 the oracle computes per timed step


class OracleBaseline:
    """Times the CPU oracle on a fixed sample of the reuse step, extrapolated to a full step.

    Sample: head 0 only; RoPE of that head's q and k over all N tokens, then the fresh states
    of the computed pairs and the merge of all P states for SAMPLE_ROWS query rows spread evenly
    over the sequence. Full-step estimate = t_rope * H * B + t_rows * (B * H * N / rows).
    The anchor step that fills the sample's state cache runs once, untimed. Both arms of the
    benchmark (the CPU baseline of ours, and --impl reference) use this same sample.
    """

    def __init__(self, w, nthreads=None):
        import numpy as np

        import oracle
        from attention_state_reuse_gb300 import workloads as wl

        self.w = w
        self.nthreads = nthreads or oracle.default_threads()
        self.q, self.k, self.v = wl.InputStream(w, heads=[0]).next()
        self.mask = wl.step_mask(w, 1)
        self.rope_cfg = None
        if w.rope:
            dtt, dhh, dww = w.rope_dims
            self.rope_cfg = dict(Hl=w.Hl, Wl=w.Wl, start_frame=w.start_frame, dt=dtt, dh=dhh,
                                 dw=dww)
        rnd = oracle.ROUND_BF16 if w.dtype == "bf16" else oracle.ROUND_F32
        self.rows_n = min(w.N, SAMPLE_ROWS)
        rows = [(0, 0, int(r)) for r in np.linspace(0, w.N - 1, self.rows_n).astype(np.int64)]
        self.orc = oracle.OracleRun(w.B, w.N, 1, w.d, w.P, w.scale, rows=rows,
                                    cache_round=rnd, input_round=rnd, rope=self.rope_cfg,
                                    nthreads=self.nthreads)
        self.orc.step(self.q, self.k, self.v)  # anchor, untimed

    def time_step(self):
        t0 = time.perf_counter()
        if self.rope_cfg:
            qq, kk = self.orc.rotate(self.q), self.orc.rotate(self.k)
        else:
            qq, kk = self.q, self.k
        t1 = time.perf_counter()
        rope, self.orc.rope = self.orc.rope, None  # this step's inputs are rotated above
        self.orc.step(qq, kk, self.v, self.mask)
        self.orc.rope = rope
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    def estimate_ms(self):
        w = self.w
        t_rope, t_rows = self.time_step()
        est = (t_rope * w.H * w.B + t_rows * (w.B * w.H * w.N / self.rows_n)) * 1e3
        return est, t_rope + t_rows

    def sample_text(self):
        w = self.w
        return (f"head 0 of {w.H}: RoPE of q,k over all {w.N} tokens + {self.rows_n} query "
                f"rows (computed pairs + merge of all {w.P} states) of the reuse step; "
                f"extrapolated x{w.H * w.B} (RoPE) and x{w.B * w.H * w.N / self.rows_n:.0f} (rows)")


def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo), or the platform's processor string."""
    import platform

    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip().lower() in ("model name", "cpu model", "hardware"):
                    return val.strip()
    except OSError:
        pass
    try:  # Arm hosts name the core in lscpu only
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            if key.strip().lower() == "model name":
                return val.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(w, steps):
    """The oracle's extrapolated step time: median over `steps` timed sample steps."""
    base = OracleBaseline(w)
    vals, spent = [], 0.0
    for _ in range(steps):
        est, sec = base.estimate_ms()
        vals.append(est)
        spent += sec
    return base, statistics.median(vals), spent


def run_reference(args, w, world=1):
    """The oracle's time for one step of the whole layer, W untimed and K timed sample steps
    (median). With `world` ranks our arm splits that same layer's heads over the ranks, so the
    job is still one layer step; rank 0 alone runs this."""
    import numpy as np

    from attention_state_reuse_gb300 import workloads as wl

    base = OracleBaseline(w)
    vals = []
    for s in range(args.warmup + args.steps):
        est_ms, _ = base.estimate_ms()
        if s >= args.warmup:
            vals.append(est_ms)
    ms = statistics.median(vals)
    flops = pair_flops(w, wl.step_mask(w, 1))
    return {
        "metric": METRIC, "value": round(ms, 2), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": False,
        "scaling": "strong", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": config_of(w, world),
        "effective_tflops": round(flops / (ms * 1e-3) / 1e12, 6),
        "cpu_baseline": {"value": round(ms, 2), "unit": "ms", "cores": base.nthreads,
                         "cpu": cpu_model(),
                         "kind": "oracle", "sample": base.sample_text()},
        "e2e": {"value": round(ms, 2), "unit": "ms", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_720p")
    ap.add_argument("--cpu-steps", type=int, default=3,
                    help="timed oracle sample steps of the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="skip the reuse-fraction sweep")
    ap.add_argument("--no-offload", dest="offload", action="store_false",
                    help="skip the schedule cycle with the far pairs' states in host memory")
    ap.add_argument("--no-group", dest="group", action="store_false",
                    help="merge every reused state each step instead of one group state per row")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count (smaller cases for profiler captures)")
    args = ap.parse_args()

    from attention_state_reuse_gb300 import workloads as wl

    w = wl.get(args.workload)
    if args.heads is not None and args.heads != w.H:
        w = wl.scaled(w, f"{w.name}_h{args.heads}", H=args.heads)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    line = run_ours(args, w, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            base, est_ms, spent = cpu_baseline(w, args.cpu_steps)
            line["cpu_baseline"] = {"value": round(est_ms, 1), "unit": "ms",
                                    "cores": base.nthreads, "cpu": cpu_model(), "kind": "oracle",
                                    "sample": base.sample_text(),
                                    "seconds_spent": round(spent, 1)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
