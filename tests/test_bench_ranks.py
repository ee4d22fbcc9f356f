"""bench.py's multi-rank plumbing on CPU: two gloo ranks, no GPU.

Under torchrun the ranks split one layer's heads (every (b, h) of the method is independent:
DiTango page, Methodology 2, Group State Computation, of which this is the single-node
analogue): rank r computes heads [r H / N, (r + 1) H / N) with no data-path collective; the only
cross-rank operations are the barriers around the timed region and the max over ranks of the
measured times. These tests run that plumbing with world size 2 over gloo, check that the head
ranges tile [0, H), and that per-rank oracle runs on their head ranges reassemble the whole
layer's oracle result bit for bit.
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


@pytest.mark.parametrize("H", [1, 2, 7, 40])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_head_ranges_tile_the_layer(H, world):
    import bench

    if world > H:
        pytest.skip("more ranks than heads")
    ranges = [bench.head_range(r, world, H) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == H
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def _shard_main(rank, world, port, queue):
    # each rank runs the oracle over its own heads of one small layer with RoPE and a reuse
    # step, then rank 0 gathers the shards
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from attention_state_reuse_gb300 import workloads as wl

        w = wl.scaled(wl.get("wan14b_layer"), "shard", H=5, T=2, Hl=4, Wl=6, P=4, start_frame=3)
        h0, h1 = bench.head_range(rank, world, w.H)
        dtt, dhh, dww = w.rope_dims
        stream = wl.InputStream(w)
        orc = oracle.OracleRun(w.B, w.N, h1 - h0, w.d, w.P, w.scale, nthreads=1,
                               rope=dict(Hl=w.Hl, Wl=w.Wl, start_frame=w.start_frame, dt=dtt,
                                         dh=dhh, dw=dww))
        outs = []
        for t in range(2):
            q, k, v = (a[:, :, h0:h1] for a in stream.next())
            res = orc.step(q, k, v, wl.step_mask(w, t))
            # rows are (b, h_local, r) in order: back to [B, H_r, N, d]
            outs.append(torch.from_numpy(res["out"].reshape(w.B, h1 - h0, w.N, w.d)))
            outs.append(torch.from_numpy(res["out_lse"].reshape(w.B, h1 - h0, w.N)))
        gathered = [None] * world if rank == 0 else None
        dist.gather_object(outs, gathered, dst=0)
        if rank == 0:
            queue.put([[x.numpy() for x in g] for g in gathered])
    finally:
        dist.destroy_process_group()


def test_head_shards_reassemble_the_layer_bit_for_bit():
    import torch.multiprocessing as mp

    import oracle
    from attention_state_reuse_gb300 import workloads as wl

    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        shards = queue.get(timeout=300)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    w = wl.scaled(wl.get("wan14b_layer"), "shard", H=5, T=2, Hl=4, Wl=6, P=4, start_frame=3)
    dtt, dhh, dww = w.rope_dims
    full = oracle.OracleRun(w.B, w.N, w.H, w.d, w.P, w.scale, nthreads=3,
                            rope=dict(Hl=w.Hl, Wl=w.Wl, start_frame=w.start_frame, dt=dtt,
                                      dh=dhh, dw=dww))
    stream = wl.InputStream(w)
    for t in range(2):
        res = full.step(*stream.next(), wl.step_mask(w, t))
        out = res["out"].reshape(w.B, w.H, w.N, w.d)
        lse = res["out_lse"].reshape(w.B, w.H, w.N)
        got_out = np.concatenate([sh[2 * t] for sh in shards], axis=1)
        got_lse = np.concatenate([sh[2 * t + 1] for sh in shards], axis=1)
        assert np.array_equal(got_out, out) and np.array_equal(got_lse, lse)


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


def test_reference_arm_is_one_layer_step_for_any_rank_count(monkeypatch):
    # our arm splits one layer's heads over the ranks, so the oracle's job is one layer step
    # whatever the rank count; its config is the one our arm prints
    import argparse

    import bench
    from attention_state_reuse_gb300 import workloads as wl

    class FixedOracle:
        nthreads = 4

        def __init__(self, w):
            pass

        def estimate_ms(self):
            return 1000.0, 0.1

        def sample_text(self):
            return "fixed"

    monkeypatch.setattr(bench, "OracleBaseline", FixedOracle)
    args = argparse.Namespace(steps=3, warmup=3)
    w = wl.get("long_720p")
    one = bench.run_reference(args, w)
    four = bench.run_reference(args, w, world=4)
    assert one["value"] == four["value"] == 1000.0
    assert one["n_gpus"] == 1 and four["n_gpus"] == 4
    assert one["config"] == bench.config_of(w, 1) and four["config"] == bench.config_of(w, 4)
    assert one["config"]["workload"] == "long_720p" and one["config"]["reuse_mask"] == "|i-j|>=3"
    for line in (one, four):
        assert line["impl"] == "reference" and line["higher_is_better"] is False
        assert line["scaling"] == "strong"
        assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
