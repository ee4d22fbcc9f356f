"""GPU: a state cache that keeps part of its states in host memory.

DiTango's closing limitations paragraph names the state cache's memory as a constraint and CPU
offloading as the remedy. Here the device cache keeps S of the P states of a row (the pairs
nearest the diagonal) and page-locked host memory keeps the rest; the kernels read and write
those in place. Storage moves nothing through arithmetic, so every output, lse and stored state
must be bit-identical to the same steps run with the whole cache on the device, which the
parity tests check against the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_state_reuse_gb300 as dt
import oracle
from attention_state_reuse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dt.build()
    dt.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


class Layer:
    """One layer's buffers, with the whole cache on the device (S = None) or S slots per row."""

    def __init__(self, w, S=None, group=True):
        dev = torch.device("cuda")
        B, N, H, d, P = w.B, w.N, w.H, w.d, w.P
        self.w, self.S = w, S
        self.dtype = wl.torch_dtype(w)
        self.plan = dt.Plan(N, P)
        self.cO, self.cL = dt.new_state_cache(B, H, S or P, N, d, self.dtype, dev)
        self.host = dt.new_host_states(B, H, P, N, d, self.dtype) if S else None
        self.group = dt.new_group_state(B, H, N, d, dev) if group else None
        self.out = torch.empty((B, N, H, d), dtype=self.dtype, device=dev)
        self.out_lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.rope = None
        if w.rope:
            dtt, dhh, dww = w.rope_dims
            self.rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                                      start_frame=w.start_frame, device=dev)
        n = dt.workspace_size(self.plan, B, H, d, self.dtype, w.rope)
        self.ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)

    def step(self, q, k, v, mask):
        dt.attn_step(self.plan, q, k, v, self.cO, self.cL, self.out, self.out_lse,
                     reuse_mask=mask, rope=self.rope, softmax_scale=self.w.scale,
                     workspace=self.ws, group=self.group, host=self.host)

    def full_cache(self):
        """The cache as [B, H, P, N, d] / [B, H, P, N] device tensors, every pair's state taken
        from wherever it is kept (device slot or host storage)."""
        if self.S is None:
            return self.cO, self.cL
        P = self.w.P
        hO, hL = self.host[0].cuda(), self.host[1].cuda()
        O, L = torch.empty_like(hO), torch.empty_like(hL)
        off = self.plan.offsets()
        slot = dt.cache_slot_map(P, self.S)
        for i in range(P):
            r0, r1 = int(off[i]), int(off[i + 1])
            for j in range(P):
                s = int(slot[i, j])
                srcO, srcL, x = (self.cO, self.cL, s) if s >= 0 else (hO, hL, j)
                O[:, :, j, r0:r1] = srcO[:, :, x, r0:r1]
                L[:, :, j, r0:r1] = srcL[:, :, x, r0:r1]
        return O, L


def run_pair(w, S, masks, group=True, default_mask=None):
    res, off = Layer(w, None, group), Layer(w, S, group)
    if default_mask is not None:  # the anchors also build the default mask's group states
        res.plan.set_mask(default_mask)
        off.plan.set_mask(default_mask)
    stream = wl.InputStream(w)
    dev = torch.device("cuda")
    for t, mask in enumerate(masks):
        q, k, v = (torch.from_numpy(a).to(dev).to(res.dtype) for a in stream.next())
        res.step(q, k, v, mask)
        off.step(q, k, v, mask)
        torch.cuda.synchronize()
        assert dt.device_status() == (0, 0)
        assert torch.equal(res.out, off.out), t
        assert torch.equal(res.out_lse, off.out_lse), t
        # every schedule starts with an anchor, after which every pair holds a state
        (rO, rL), (oO, oL) = res.full_cache(), off.full_cache()
        assert torch.equal(rO, oO) and torch.equal(rL, oL), t
    return res, off


@pytest.mark.parametrize("ahead", [False, True])
def test_720p_layer_schedule_with_host_storage_matches_device_cache(ahead):
    # the 720p-shaped layer at its stated N (75600 tokens, P = 16, RoPE) on 4 heads, over its
    # eight-step schedule (anchor, |i - j| >= 3 reused, refresh at step 4), with S = 2 * 3 - 1
    # device slots per row: the steady steps compute device-resident pairs only; the anchors
    # write the far pairs into host memory and the group rebuilds read them back (ahead: the
    # plans' default mask is the reuse mask, so the anchors' merges build the group states)
    w = wl.scaled(wl.get("long_720p"), "long_offload", H=4)
    masks = [wl.step_mask(w, t) for t in range(w.steps)]
    run_pair(w, 5, masks, default_mask=masks[1] if ahead else None)


@pytest.mark.parametrize("dtype,S", [("bf16", 3), ("bf16", 1), ("fp32", 2)])
def test_changing_masks_with_host_storage(dtype, S):
    # masks that compute far pairs (random) and change the reused sets, so that pair kernels
    # write host-resident states and group rebuilds read them, without and with group states
    base = wl.get("small_bf16") if dtype == "bf16" else wl.get("tiny_fp32")
    sched = [("all",), ("dist", 2), ("random",), ("dist", 3), ("dist", 3), ("all",), ("dist", 2)]
    w = wl.Workload(f"offload_{dtype}", base.index, 1, 3, base.d, base.T, base.Hl, base.Wl,
                    base.P, dtype, len(sched), 0.03, schedule=sched)
    masks = [wl.step_mask(w, t) for t in range(w.steps)]
    for group in (True, False):
        run_pair(w, S, masks, group)


def test_host_storage_matches_oracle():
    # the offloaded path against the oracle on every row (RoPE, ragged partitions)
    w = wl.scaled(wl.get("wan14b_layer"), "offload_oracle", H=2, T=3, Hl=10, Wl=13, P=6,
                  start_frame=2, steps=3)
    lay = Layer(w, 3)
    dtt, dhh, dww = w.rope_dims
    orc = oracle.OracleRun(w.B, w.N, w.H, w.d, w.P, w.scale,
                           rope=dict(Hl=w.Hl, Wl=w.Wl, start_frame=w.start_frame, dt=dtt, dh=dhh,
                                     dw=dww))
    stream = wl.InputStream(w)
    for t in range(3):
        q, k, v = stream.next()
        mask = np.zeros((w.P, w.P), np.uint8) if t == 0 else wl.distance_mask(w.P, 2)
        lay.step(*(torch.from_numpy(a).cuda().to(torch.bfloat16) for a in (q, k, v)), mask)
        torch.cuda.synchronize()
        ref = orc.step(q, k, v, mask)
        got = lay.out.float().cpu().numpy().transpose(0, 2, 1, 3).reshape(-1, w.d)
        got_lse = lay.out_lse.cpu().numpy().reshape(-1)
        assert np.abs(got - ref["out"]).max() <= 2e-2
        assert np.abs(got_lse - ref["out_lse"]).max() <= 1e-3


def test_planner_reads_host_storage():
    # importance reads every pair's lse (host-resident ones too); snapshot and drift the local
    # pairs (always on the device): equal to the device-resident cache's results
    w = wl.scaled(wl.get("small_bf16"), "offload_planner", H=2, steps=2)
    res, off = run_pair(w, 3, [np.zeros((w.P, w.P), np.uint8)])
    wi_r = dt.planner_importance(res.plan, res.cO, res.cL)
    wi_o = dt.planner_importance(off.plan, off.cO, off.cL, host=off.host)
    snap_r = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device="cuda")
    snap_o = torch.empty_like(snap_r)
    dt.planner_snapshot(res.plan, res.cO, res.cL, snap_r)
    dt.planner_snapshot(off.plan, off.cO, off.cL, snap_o, host=off.host)
    torch.cuda.synchronize()
    assert torch.equal(snap_r, snap_o)
    # the reductions sum with atomics (order-dependent rounding)
    np.testing.assert_allclose(wi_o.cpu().numpy(), wi_r.cpu().numpy(), rtol=1e-5, atol=1e-9)


def test_host_storage_errors():
    w = wl.scaled(wl.get("small_bf16"), "offload_err", H=2, steps=1)
    lay = Layer(w, 3)
    q = torch.zeros((w.B, w.N, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    # pageable host memory cannot be handed to the kernels
    with pytest.raises(ValueError):
        dt.attn_step(lay.plan, q, q, q, lay.cO, lay.cL, lay.out,
                     host=(torch.empty_like(lay.host[0], pin_memory=False), lay.host[1]))
    lib = dt.load_library()
    arr = np.zeros(lay.host[0].numel(), dtype=np.uint16)  # ordinary (pageable) host memory
    cache = dt._state_cache(lay.cO, lay.cL, None, lay.host)
    cache.host_O.ptr = arr.ctypes.data
    qd, od = dt.tensor_desc(q), dt.tensor_desc(lay.out)
    st = lib.ditango_attn_step(lay.plan.handle, ctypes.byref(qd), ctypes.byref(qd),
                               ctypes.byref(qd), None, None, ctypes.byref(cache),
                               ctypes.byref(od), None, ctypes.c_float(0.125), None,
                               ctypes.c_size_t(0), None)
    assert dt.STATUS[st] == "INVALID_ARG"
    # S < P needs host storage; S > P is a shape error
    cache = dt._state_cache(lay.cO, lay.cL, None, None)
    st = lib.ditango_attn_step(lay.plan.handle, ctypes.byref(qd), ctypes.byref(qd),
                               ctypes.byref(qd), None, None, ctypes.byref(cache),
                               ctypes.byref(od), None, ctypes.c_float(0.125), None,
                               ctypes.c_size_t(0), None)
    assert dt.STATUS[st] == "SHAPE"
    assert lay.plan.cache_state()[2] == 0


def test_anchor_planner_drives_an_offloaded_cache():
    # the planner's reductions read the host-resident states through the slot map; its masks
    # drive steps whose outputs match the oracle
    w = wl.scaled(wl.get("small_bf16"), "offload_anchor", H=2, steps=6)
    lay = Layer(w, 3)
    planner = dt.AnchorPlanner(lay.plan, lay.cO, lay.cL, anchor_every=3, tau=0.0, group=2,
                               budget=w.P + 8, host=lay.host)
    orc = oracle.OracleRun(w.B, w.N, w.H, w.d, w.P, w.scale)
    stream = wl.InputStream(w)
    for t in range(6):
        q, k, v = stream.next()
        mask = planner.mask()
        assert mask.shape == (w.P, w.P) and (np.diag(mask) == 0).all()
        lay.step(*(torch.from_numpy(a).cuda().to(torch.bfloat16) for a in (q, k, v)), mask)
        planner.after_step(mask)
        torch.cuda.synchronize()
        ref = orc.step(q, k, v, mask)
        got = lay.out.float().cpu().numpy().transpose(0, 2, 1, 3).reshape(-1, w.d)
        assert np.abs(got - ref["out"]).max() <= 2e-2
        assert np.abs(lay.out_lse.cpu().numpy().reshape(-1) - ref["out_lse"]).max() <= 1e-3
