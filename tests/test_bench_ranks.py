"""bench.py's multi-rank plumbing on CPU: two gloo ranks, no GPU.

Under torchrun every rank runs its own replica of the layer (weak scaling, no data-path
collective); the only cross-rank operations are the barriers around the timed region and the
max over ranks of the measured times. These tests run that plumbing with world size 2 over gloo.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        bench.barrier(world)
        got = bench.max_over_ranks(10.0 + 3.5 * rank, world)  # rank 1 is the slow one
        bench.barrier(world)
        queue.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(queue.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert got == [(0, 13.5), (1, 13.5)]
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_needs_no_process_group():
    import bench

    bench.barrier(1)
    assert bench.max_over_ranks(4.25, 1) == 4.25


def test_replicas_have_own_inputs_and_same_shapes():
    import bench
    from attention_state_reuse_gb300 import workloads as wl

    w = wl.scaled(wl.get("wan14b_layer"), "tiny_replica", H=2, T=1, Hl=4, Wl=8)
    r0, r1 = bench.replica_workload(w, 0), bench.replica_workload(w, 1)
    assert (r0.N, r0.H, r0.d, r0.P) == (r1.N, r1.H, r1.d, r1.P) == (w.N, w.H, w.d, w.P)
    a0 = wl.InputStream(r0).next()
    a1 = wl.InputStream(r1).next()
    for x, y in zip(a0, a1):
        assert x.shape == y.shape
        assert not np.array_equal(x, y)
    assert w.index == r0.index  # the caller's workload is left alone


def test_algorithmic_work_accounting():
    # hand-computed for the Wan-14B-shaped layer (B=1, H=40, d=128, N=32760, P=8, partitions of
    # 4095 rows, |i-j| >= 2 reused: 22 computed pairs; rows of partitions 0 and 7 keep 2 computed
    # states, the other six keep 3)
    import bench
    from attention_state_reuse_gb300 import workloads as wl

    w = wl.get("wan14b_layer")
    mask = wl.distance_mask(w.P, 2)
    assert int((mask == 0).sum()) == 22
    assert bench.pair_flops(w, mask) == 4 * 1 * 40 * 128 * 22 * 4095 * 4095
    rows = 40 * 4095
    state = 128 * 2 + 4
    no_group = rows * 8 * (8 * state + state)
    with_group = rows * (2 * (2 * state + (128 * 4 + 4) + state) + 6 * (3 * state + (128 * 4 + 4) + state))
    assert bench.merge_bytes(w, mask, False) == no_group == 3066336000
    assert bench.merge_bytes(w, mask, True) == with_group
    assert abs(with_group - 1.9538e9) < 1e5
    # all computed: no group state is read
    zero = np.zeros((w.P, w.P), np.uint8)
    assert bench.merge_bytes(w, zero, True) == bench.merge_bytes(w, zero, False)


def test_reference_arm_counts_every_rank_replica(monkeypatch):
    # the oracle does the whole job's work: one replica per rank of the GPU arm, same host cores
    import argparse

    import bench
    from attention_state_reuse_gb300 import workloads as wl

    class FixedOracle:
        nthreads = 4

        def __init__(self, w, budget):
            pass

        def estimate_ms(self):
            return 1000.0, 0.1

        def sample_text(self):
            return "fixed"

    monkeypatch.setattr(bench, "OracleBaseline", FixedOracle)
    args = argparse.Namespace(steps=3, warmup=3)
    w = wl.get("wan14b_layer")
    one = bench.run_reference(args, w)
    four = bench.run_reference(args, w, world=4)
    assert one["value"] == 1000.0 and one["n_gpus"] == 1
    assert four["value"] == 4000.0 and four["n_gpus"] == 4
    assert four["effective_tflops"] == pytest.approx(one["effective_tflops"], rel=1e-6)
    for line in (one, four):
        assert line["impl"] == "reference" and line["higher_is_better"] is False
        assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
