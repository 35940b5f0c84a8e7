"""The multi-replica host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The path shards by sequence with no exchange, so N GPUs run N replicas; the job's time
is the slowest rank's and its rate counts every rank's batch. The reference arm runs
on rank 0 only.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from speculative_decoding_draft_dflash_gb300 import synth
        t = bench.max_over_ranks(times[rank], world, device="cpu")
        w = synth.WORKLOADS["serve_b32"]
        rate = bench.whole_job_rate(world, w, t)
        q.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    world, times = 2, [0.31, 0.47]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    from speculative_decoding_draft_dflash_gb300 import synth
    w = synth.WORKLOADS["serve_b32"]
    for rank, t, rate in got:
        assert t == pytest.approx(max(times))                  # every rank sees the slowest
        assert rate == pytest.approx(world * w.batch * w.n_layers / (max(times) * 1e-3))


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(0.25, 1) == 0.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse
    import bench
    from speculative_decoding_draft_dflash_gb300 import synth
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=0, gpus=2, impl="reference", workload="serve_b32",
                              no_cpu_baseline=True, no_graph=False)
    bench.run_reference(args, synth.WORKLOADS["serve_b32"])  # returns without work
    assert capsys.readouterr().out == ""
