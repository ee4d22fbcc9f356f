"""The attention step for callers that cannot allocate device memory.

ditango_attn_step_static_workspace takes no workspace: its scratch (the rotated q and k of the
RoPE prologue) lives in a fixed 64 MiB device array inside the library, for callers such as
plugins whose host framework forbids allocation during execution, or processes whose memory
pool already holds the GPU's free memory. These tests call it through the C ABI and compare it
with ditango_attn_step on the same inputs, over two calls in a row (an all-compute step, then
a reuse step): both run the same deterministic kernels, so outputs, lse and state caches must
be bit-identical; and check that a step whose scratch
would exceed the array is refused before anything is launched.

This file is named to be collected last, so that a run stopping at the first failure has run
every other test before it.
"""
import numpy as np
import pytest
import torch

import attention_state_reuse_gb300 as dt
from attention_state_reuse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dt.build()
    dt.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _setup(w, dev):
    B, N, H, d, P = w.B, w.N, w.H, w.d, w.P
    plan = dt.Plan(N, P)
    cO, cL = dt.new_state_cache(B, H, P, N, d, torch.bfloat16, dev)
    out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    return plan, cO, cL, out, out_lse


def test_static_workspace_step_matches_workspace_step():
    dev = torch.device("cuda")
    w = wl.scaled(wl.get("wan14b_layer"), "no_alloc", H=3, T=3, Hl=8, Wl=16, P=4,
                  start_frame=3, steps=2)
    dtt, dhh, dww = w.rope_dims
    rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                         start_frame=w.start_frame, device=dev)
    ref = _setup(w, dev)
    new = _setup(w, dev)
    ws = torch.empty(dt.workspace_size(ref[0], w.B, w.H, w.d, torch.bfloat16, True),
                     dtype=torch.uint8, device=dev)
    stream = wl.InputStream(w)
    for t in range(2):  # two calls in a row: all pairs computed, then |i-j| >= 2 reused
        q, k, v = (torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in stream.next())
        mask = wl.distance_mask(w.P, 2) if t else np.zeros((w.P, w.P), np.uint8)
        dt.attn_step(ref[0], q, k, v, ref[1], ref[2], ref[3], ref[4], reuse_mask=mask,
                     rope=rope, softmax_scale=w.scale, workspace=ws)
        dt.attn_step_static_workspace(new[0], q, k, v, new[1], new[2], new[3], new[4],
                                      reuse_mask=mask, rope=rope, softmax_scale=w.scale)
        torch.cuda.synchronize()
        assert dt.device_status() == (0, 0)
        # the same deterministic kernels on the same inputs: identical bits, not just close
        assert torch.equal(new[3], ref[3]) and torch.equal(new[4], ref[4]), t
        assert torch.equal(new[1], ref[1]) and torch.equal(new[2], ref[2]), t
        assert new[0].cache_state()[2] == ref[0].cache_state()[2] == t + 1


def test_static_workspace_refuses_oversized_scratch():
    dev = torch.device("cuda")
    # rotated q and k of 8192 x 17 x 128 bf16 need 2 x 35.7 MB > 64 MiB
    B, N, H, d, P = 1, 8192, 17, 128, 4
    plan = dt.Plan(N, P)
    q = torch.zeros((B, N, H, d), dtype=torch.bfloat16, device=dev)
    cO, cL = dt.new_state_cache(B, H, P, N, d, torch.bfloat16, dev)
    out = torch.empty_like(q)
    rope = dt.RopeTables(2, 64, 64, 44, 42, 42, device=dev)
    with pytest.raises(dt.DitangoError) as e:
        dt.attn_step_static_workspace(plan, q, q, q, cO, cL, out, rope=rope)
    assert e.value.name == "WORKSPACE"
    assert plan.cache_state()[2] == 0
