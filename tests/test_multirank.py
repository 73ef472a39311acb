"""Host logic of the multi-rank bench path, on CPU: two gloo ranks stand in for
two GPUs.  Each rank runs its own batch (weak scaling); the job's time is the
slowest rank's, and only rank 0 prints."""
import os
import socket
import types

import torch.multiprocessing as mp

import bench
from synth import gen


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, xs, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        out.put((rank, bench._max_over_ranks(xs[rank], world, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_reaches_every_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    xs = [1.25, 3.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, xs, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    assert bench._max_over_ranks(2.0, 1, "cpu") == 2.0


def test_job_throughput_is_weak_scaling():
    ops = 2 * 512 * 3584 * 3584
    one = bench._job_tops(1, ops, 100, 3.3)
    assert abs(one - ops * 100 / 3.3e-3 / 1e12) < 1e-9 * one
    # two ranks, each its own 100 steps, slowest rank 3.3 ms: twice the work in the same time
    assert abs(bench._job_tops(2, ops, 100, 3.3) - 2 * one) < 1e-9 * one


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = types.SimpleNamespace(steps=3, warmup=3, gpus=2)
    assert bench.run_reference(args, gen.config_by_name("q6_K_tiny_256x512_nt16"), rank=1) is None
    assert capsys.readouterr().out == ""
