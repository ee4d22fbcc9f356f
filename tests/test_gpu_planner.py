"""GPU parity of the anchor-guided planner's reductions, and a planner-driven run.

Importance, snapshot and drift run on seeded synthetic state caches made on the host, and are
compared with the oracle on the same arrays (importance and drift within fp32 summation error,
the snapshot byte for byte). The planner-driven run lets AnchorPlanner choose every step's
mask on a small bf16 layer and checks each step against the oracle, and checks the
importance weights taken at the anchor against the oracle's own states.
"""
import numpy as np
import pytest
import torch

import attention_state_reuse_gb300 as dt
import oracle
from attention_state_reuse_gb300 import workloads as wl
from gpu_harness import ParityRun
from oracle import planner as oplan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dt.build()
    dt.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()


def _lse(rng, B, H, P, N):
    lse = (rng.normal(size=(B, H, P, N)) * 3.0 + rng.normal(size=(1, 1, P, 1)) * 2.0).astype(np.float32)
    return torch.from_numpy(lse).to("cuda"), lse.astype(np.float64)


def _cache(rng, B, H, P, N, d, dtype):
    O = rng.standard_normal(size=(B, H, P, N, d), dtype=np.float32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    cO = torch.from_numpy(O).to("cuda").to(tdt)
    cL, lse = _lse(rng, B, H, P, N)
    return cO, cL, lse


def _empty_O(B, H, P, N, d, dtype):
    # importance reads only the lse; the O cache just has to be a valid tensor of its shape
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return torch.empty((B, H, P, N, d), dtype=tdt, device="cuda")


@pytest.mark.parametrize("B,H,P,N,d,dtype", [(2, 3, 8, 1000, 128, "bf16"), (1, 2, 3, 129, 64, "fp32"),
                                             (1, 1, 64, 64 * 3 + 5, 64, "bf16"),
                                             (1, 40, 8, 32760, 128, "bf16")])
def test_importance_matches_oracle(B, H, P, N, d, dtype):
    rng = np.random.default_rng(P * 1000 + N)
    cL, lse = _lse(rng, B, H, P, N)
    cO = _empty_O(B, H, P, N, d, dtype)
    plan = dt.Plan(N, P)
    w = dt.planner_importance(plan, cO, cL).cpu().numpy()
    ref = oplan.importance(lse, oracle.partition_offsets(N, P))
    assert np.abs(w - ref).max() < 2e-6, np.abs(w - ref).max()
    assert np.abs(w.sum(axis=1) - 1.0).max() < 1e-5


@pytest.mark.parametrize("B,H,P,N,d,dtype", [(2, 3, 8, 1000, 128, "bf16"), (1, 2, 5, 333, 64, "fp32"),
                                             (1, 1, 64, 64 * 3 + 5, 128, "bf16")])
def test_snapshot_and_drift_match_oracle(B, H, P, N, d, dtype):
    rng = np.random.default_rng(P * 7 + N)
    cO, cL, _ = _cache(rng, B, H, P, N, d, dtype)
    plan = dt.Plan(N, P)
    offs = oracle.partition_offsets(N, P)
    part = np.searchsorted(offs, np.arange(N), side="right") - 1
    snap = torch.empty((B, H, N, d), dtype=cO.dtype, device="cuda")
    dt.planner_snapshot(plan, cO, cL, snap)
    diag = cO[:, :, torch.as_tensor(part, device="cuda"), torch.arange(N, device="cuda")]
    assert torch.equal(snap, diag)
    # drift of the cache's diagonal against a perturbed copy of it (host arrays both sides)
    anchor = diag.float().cpu().numpy() * (1.0 + rng.normal(size=(1, 1, N, 1)) * 0.05)
    anchor = anchor.astype(np.float32)
    snap.copy_(torch.from_numpy(anchor).to(snap.dtype))
    anchor = snap.float().cpu().numpy().astype(np.float64)
    got = dt.planner_drift(plan, cO, cL, snap).cpu().numpy()
    want = oplan.drift(diag.float().cpu().numpy().astype(np.float64), anchor, offs)
    assert np.allclose(got, want, rtol=2e-5, atol=1e-9), (got, want)
    zero = torch.zeros_like(snap)
    assert np.all(dt.planner_drift(plan, cO, cL, zero).cpu().numpy() == 0.0)


def test_planner_argument_checks():
    plan = dt.Plan(100, 4)
    cO, cL = dt.new_state_cache(1, 2, 4, 100, 64, torch.bfloat16, "cuda")
    snap = torch.empty((1, 2, 100, 64), dtype=torch.float32, device="cuda")  # wrong dtype
    with pytest.raises(dt.DitangoError) as e:
        dt.planner_drift(plan, cO, cL, snap)
    assert e.value.name == "DTYPE"
    other = dt.Plan(100, 5)
    with pytest.raises(dt.DitangoError) as e:
        dt.planner_importance(other, cO, cL)
    assert e.value.name == "SHAPE"


def test_anchor_planner_drives_steps():
    # small bf16 layer, P = 8; the planner chooses every mask: anchors every 4 steps, groups of
    # two partitions, a threshold that leaves some groups reused and some recomputed
    sched = [("all",)] * 9
    w = wl.Workload("planned", 1, 1, 3, 64, 4, 16, 16, 8, "bf16", len(sched), 0.05,
                    schedule=sched)
    pr = ParityRun(w, group=True)
    ap = dt.AnchorPlanner(pr.plan, pr.cO, pr.cL, anchor_every=4, tau=1e-3, group=2)
    masks = []
    for t in range(len(sched)):
        m = ap.mask()
        masks.append(m)
        e = pr.step(mask=m)
        assert e["ok"], (t, e)
        if t == 0:
            # importance at the anchor against the oracle's own states of that step
            B, H, P, N = w.B, w.H, w.P, w.N
            lse = pr.orc.cache_lse.reshape(B, H, N, P).transpose(0, 1, 3, 2)
            ap.after_step(m)
            ref = oplan.importance(lse, oracle.partition_offsets(N, P))
            assert np.abs(ap.w - ref).max() < 1e-5
        else:
            ap.after_step(m)
    assert not masks[0].any() and not masks[4].any() and not masks[8].any()  # anchors
    between = [m for t, m in enumerate(masks) if t % 4]
    assert all(np.all(np.diag(m) == 0) for m in between)
    assert any(m.any() for m in between)          # something was reused
    assert any((m == 0).sum() > 8 for m in between)  # and something beyond the diagonal computed


def test_anchor_planner_builds_group_states_ahead():
    # two planner-driven runs on the same inputs, with and without the ahead-of-time group
    # build: the masks agree, every step matches the oracle, and the non-anchor steps agree bit
    # for bit (a group state built at the anchor holds the same values as one built at the
    # first reuse step, from the same cached states)
    sched = [("all",)] * 10
    w = wl.Workload("planned_ahead", 2, 1, 3, 64, 4, 16, 16, 8, "bf16", len(sched), 0.05,
                    schedule=sched)
    runs = [ParityRun(w, group=True), ParityRun(w, group=True)]
    aps = [dt.AnchorPlanner(r.plan, r.cO, r.cL, anchor_every=4, tau=1e-3, group=2,
                            build_ahead=b) for r, b in zip(runs, (True, False))]
    for t in range(len(sched)):
        ms = [ap.mask() for ap in aps]
        assert np.array_equal(ms[0], ms[1]), t
        for r, ap, m in zip(runs, aps, ms):
            e = r.step(mask=m)
            assert e["ok"], (t, e)
            ap.after_step(m)
        if ms[0].any():
            assert torch.equal(runs[0].out, runs[1].out), t
            assert torch.equal(runs[0].out_lse, runs[1].out_lse), t
    assert aps[0].predicted is not None and aps[0].predicted.any()
