"""Failure detection on the GPU without a fault: a bounded barrier wait that runs out.

The plan's test hook makes the pair kernel's first CTA skip the copy of its first K tile. The
MMA warp's wait for that tile then gives up after its limit (about one second); the CTA stops,
drains what it has in flight, frees its TMEM and sets the device error word, which
ditango_device_status reports and clears. Nothing traps, faults or hangs, and the context stays
usable: the next steps match the oracle again.
"""
import time

import numpy as np
import pytest
import torch

import attention_state_reuse_gb300 as dt
from attention_state_reuse_gb300 import workloads as wl
from gpu_harness import ParityRun

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dt.build()
    dt.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()


@pytest.mark.parametrize("rope", [False, True])
def test_device_timeout_is_reported_and_the_context_recovers(rope):
    w = wl.scaled(wl.get("small_bf16"), "fault", H=2, steps=3)
    w.rope = rope
    pr = ParityRun(w)
    P = w.P
    compute_all = np.zeros((P, P), np.uint8)
    assert pr.step(mask=compute_all)["ok"]

    # the armed step: the launch returns, the device reports the timeout
    pr.plan.inject_fault(1)
    q, k, v = pr.stream.next()
    t0 = time.time()
    dt.attn_step(pr.plan, pr._to_dev(q), pr._to_dev(k), pr._to_dev(v), pr.cO, pr.cL, pr.out,
                 pr.out_lse, reuse_mask=compute_all, rope=pr.rope, softmax_scale=w.scale,
                 workspace=pr.ws)
    status, code = dt.device_status()
    elapsed = time.time() - t0
    assert dt.STATUS[status] == "DEVICE_TIMEOUT" and code != 0, (status, code)
    assert 0.5 < elapsed < 60.0, elapsed
    pr.orc.book.advance(compute_all)  # the plan recorded the armed step like any other
    pr.t += 1
    assert dt.device_status() == (0, 0)  # reading the status cleared it

    # the hook is one-shot, and the context works: recompute everything, then reuse
    e = pr.step(mask=compute_all)
    assert e["ok"], e
    e = pr.step(mask=wl.distance_mask(P, 2))
    assert e["ok"], e
