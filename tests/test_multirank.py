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


# --------------------------------------------------------------------------
# column-parallel split of the GEMM over ranks (shard.py)
def test_od_slices_cover_the_rows_in_tile_multiples():
    from quantized_int8_gemm_gb300 import shard
    for od in (1, 127, 128, 300, 3584, 18944, 1000):
        for world in (1, 2, 3, 4, 8):
            sl = shard.od_slices(od, world)
            assert len(sl) == world
            assert sl[0][0] == 0 and sl[-1][1] == od
            for (a0, a1), (b0, b1) in zip(sl, sl[1:]):
                assert a1 == b0                        # contiguous, no overlap
            for o0, o1 in sl[:-1]:
                assert o0 % 128 == 0 and (o1 - o0) % 128 == 0 or o1 == od
            widths = [o1 - o0 for o0, o1 in sl]
            units = [-(-w // 128) for w in widths]
            assert max(units) - min(units) <= 1        # balanced to one tile
    assert shard.od_slices(3584, 8) == [(0, 512), (512, 1024), (1024, 1536), (1536, 2048),
                                        (2048, 2432), (2432, 2816), (2816, 3200), (3200, 3584)]


def _shard_rank_main(rank, world, port, qtype, od, id_, nt, out):
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from quantized_int8_gemm_gb300 import shard
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = gen.weights(qtype, od, id_, 5)
        Q = oracle.quantize_q8_0(gen.activations(nt, id_, 6))   # replicated activations
        slices = shard.od_slices(od, world)
        o0, o1 = slices[rank]
        Ws = np.ascontiguousarray(shard.weight_rows(W, qtype, id_, o0, o1))
        qt = oracle.Q4_K if qtype == "q4_K" else oracle.Q6_K
        # the rank's own GEMM (here the oracle on its row slice: this test checks
        # the partition and the gather, not the kernel)
        y_loc = oracle.gemm(qt, Ws, o1 - o0, id_, Q, nt) if o1 > o0 else np.zeros((nt, 0))
        y = shard.gather_columns(torch.from_numpy(y_loc), slices)
        if rank == 0:
            out.put(y.numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_column_parallel_gemm_reassembles_the_single_rank_result():
    """Two gloo ranks, ragged od (300 rows: slices of 256 and 44): every rank
    computes its row slice of W against the replicated activations, the
    column slices are gathered, and the assembled Y equals the single-rank
    result bit for bit (each output is the same sum either way)."""
    import numpy as np

    import oracle
    qtype, od, id_, nt = "q4_K", 300, 512, 37
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, 2, port, qtype, od, id_, nt, out))
             for r in range(2)]
    for p in procs:
        p.start()
    y = out.get(timeout=180)
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    W = gen.weights(qtype, od, id_, 5)
    Q = oracle.quantize_q8_0(gen.activations(nt, id_, 6))
    assert np.array_equal(y, oracle.gemm(oracle.Q4_K, W, od, id_, Q, nt))
