#!/usr/bin/env python
"""Throughput of the k-quant x q8_0 prefill GEMM hot path on GB300.

One step = the whole hot path over one batch of activations: q8_0
quantization of X fused with the activation operand plane, then the GEMM
against a registered weight (mmq_gemm_f32; --step two times mmq_quantize_act
followed by mmq_gemm instead).  Registration is a one-time, per-weight cost
(the pages call its amortization infinite); it is timed once and reported
separately.

Default workload: q4_K q-proj, od = id = 3584, nt = 512.  Inputs rotate over
enough independent sets (activations, weights, outputs) to exceed twice the
L2 size, so every step reads its operands from HBM.  The K timed steps are
captured into CUDA graphs and replayed; that pass gives `value`.  A second
pass over the same K steps, with CUDA events around every GEMM kernel, gives
the kernel's live average duration for the roofline.  The events stay out of
the first pass: an event record between the two kernels of a step adds
latency and stops the GEMM's programmatic launch behind the quantization.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

The default run also times the q6_K q-proj workload (same shape) in the
same process and reports it under "also", and times quantize_act, gemm and
the fused call separately, each with cold (rotating) and warm inputs, under
"timings".

For N > 1 (under torchrun) the problem is split column-parallel: rank r
registers weight rows [o0, o1) (shard.od_slices: multiples of the 128-row
weight tile) and computes Y[:, o0:o1] from the replicated activations, with no
data-path collective (total work fixed: strong scaling); --parallel replicas
runs an independent whole problem per rank instead (weak scaling).  Rank 0
prints one JSON line with the whole-job throughput over the slowest rank's
time.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int8 TOPS and GEMM tokens/s at 1 GB300; % of roofline (q4_K/q6_K x q8_0)"
UNIT = "TOPS"  # 2*nt*od*id integer multiply-adds counted as 2 ops, per second, / 1e12
DEFAULT_WORKLOAD = "q4_K_qproj_3584x3584_nt512"
# the GEMM arm every call of the run asks for (--arm; 0: the library's choice)
ARM = [0]
# The pages' own q4_K q-proj kernel (nt=512, od=id=3584): 555 us after the
# split-phase A staging step, i.e. 2*512*3584*3584 / 555e-6 = 23.7 TOPS, on an
# unnamed GPU ("25 · r20: Split-phase A staging", §5).  Context only.
PAGES_TOPS = {"q4_K_qproj_3584x3584_nt512": 2 * 512 * 3584 * 3584 / 555e-6 / 1e12}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------- helpers
def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_sha1(path):
    """sha1 of a C/CUDA source with comments removed and whitespace runs
    collapsed, so that a comment edit does not orphan its profile."""
    src = open(path).read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    code = " ".join("".join(out).split())
    return hashlib.sha1(code.encode()).hexdigest()


def _workload_name(cfg, args):
    """The workload's name, marked when its q6_K scales are not the recipe's
    and when the operand plane is built from the W_exp plane."""
    return (cfg.name + ("_int8scales" if cfg.qtype == "q6_K" and args.q6_scales == "int8" else "")
            + ("_wexp" if getattr(args, "reg_wexp", False) else ""))


def _profiled_traffic(workload, kernel):
    """DRAM bytes per GEMM launch from the committed ncu summary of this kernel
    on this workload (profiles/<kernel>_<workload>.md), if it was taken on the
    current kernel source; else None."""
    src = os.path.join(ROOT, "quantized_int8_gemm_gb300", "csrc", "gemm.cu")
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"gemm_cu_code_sha1:\s*([0-9a-f]{40})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if m_sha and m_b and m_sha.group(1) == _code_sha1(src):
        return int(m_b.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.out.name)
        inwin = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        use = inwin or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({n for r in use for n, v in zip(self.NAMES, r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inwin)}


def _max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks of the process group (x itself at world 1):
    the job's time is its slowest rank's."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_tops(world: int, ops_per_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank runs `steps` steps of `ops_per_step`
    (weak scaling) in `ms`, the slowest rank's time."""
    return world * ops_per_step * steps / (ms * 1e-3) / 1e12


def _gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------- CPU oracle timing
def _cpu_model():
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else the machine)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip().lower() in ("model name", "cpu model") and v.strip():
                    return v.strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_plan(cfg, W, X, target_s, threads):
    """Size a bounded sample of the workload for the oracle: q8_0 quantization
    of all nt tokens plus the fp64 GEMM of those tokens against n_rows weight
    rows (a multiple of the thread count), about target_s seconds.  Returns
    (n_rows, Q)."""
    import oracle
    qt = oracle.Q4_K if cfg.qtype == "q4_K" else oracle.Q6_K
    row_bytes = (cfg.id // 256) * (144 if cfg.qtype == "q4_K" else 210)
    t = time.perf_counter()
    Q = oracle.quantize_q8_0(X)
    tq = time.perf_counter() - t
    probe = min(cfg.od, max(2, threads))
    t = time.perf_counter()
    oracle.gemm_mt(qt, W[:probe * row_bytes], probe, cfg.id, Q, cfg.nt, threads)
    per_row = (time.perf_counter() - t) / probe
    n_rows = int(max(1, min(cfg.od, (target_s - tq) / max(per_row, 1e-9))))
    if n_rows >= threads:
        n_rows -= n_rows % threads
    return n_rows, Q


def _oracle_baseline(cfg, W, X, target_s):
    """The oracle as it stands on every host core: median of three timed runs of
    the bounded sample (quantization of all tokens + the threaded fp64 GEMM of
    those tokens x a row sample), ~target_s in all."""
    import oracle
    qt = oracle.Q4_K if cfg.qtype == "q4_K" else oracle.Q6_K
    row_bytes = (cfg.id // 256) * (144 if cfg.qtype == "q4_K" else 210)
    threads = oracle.host_threads()
    n_rows, _ = _oracle_plan(cfg, W, X, target_s / 3.0, threads)
    Ws = W[:n_rows * row_bytes]
    runs = []
    for _ in range(3):
        t = time.perf_counter()
        Q = oracle.quantize_q8_0(X)
        oracle.gemm_mt(qt, Ws, n_rows, cfg.id, Q, cfg.nt, threads)
        runs.append(time.perf_counter() - t)
    dt = statistics.median(runs)
    ops = 2 * cfg.nt * n_rows * cfg.id
    return {"value": ops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_model": _cpu_model(),
            "sample": (f"oracle q8_0 quantization of {cfg.nt}x{cfg.id} activations + fp64 GEMM of "
                       f"{cfg.nt} tokens x {n_rows} of {cfg.od} weight rows over {threads} threads; "
                       f"median of 3 runs ({', '.join(f'{r:.2f}' for r in runs)} s)")}


def run_reference(args, cfg, rank):
    """The oracle as it stands, on every host core.  Each step is a bounded
    sample of the workload -- q8_0 quantization of nt_s tokens and the fp64
    GEMM of those tokens against n_rows weight rows, threaded over the rows --
    sized so the whole warm-up + timed run takes about two and a half
    minutes."""
    if rank != 0:
        return
    import oracle
    from synth import gen
    oracle.build()
    W, X = gen.config_inputs(cfg)
    if cfg.qtype == "q6_K" and args.q6_scales != "small":
        W = gen.weights(cfg.qtype, cfg.od, cfg.id, cfg.seed, q6_scales=args.q6_scales)
    qt = oracle.Q4_K if cfg.qtype == "q4_K" else oracle.Q6_K
    row_bytes = (cfg.id // 256) * (144 if cfg.qtype == "q4_K" else 210)
    threads = oracle.host_threads()
    target = max(1e-3, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    # calibrate: quantization of all tokens, and `threads` weight rows against all tokens
    t = time.perf_counter()
    Qf = oracle.quantize_q8_0(X)
    tq = time.perf_counter() - t
    probe = min(cfg.od, max(2, threads))
    t = time.perf_counter()
    oracle.gemm_mt(qt, W[:probe * row_bytes], probe, cfg.id, Qf, cfg.nt, threads)
    t_row = (time.perf_counter() - t) / probe
    # enough rows that the GEMM, not the quantization, dominates each step
    n_rows = int(min(cfg.od, max(math.ceil(4 * tq / t_row), (target - tq) / t_row, 1)))
    if n_rows >= threads:
        n_rows -= n_rows % threads
    nt_s = int(min(cfg.nt, max(1, cfg.nt * target / (tq + t_row * n_rows))))
    Xs = np.ascontiguousarray(X[:nt_s])
    Ws = W[:n_rows * row_bytes]

    def step():
        Q = oracle.quantize_q8_0(Xs)
        oracle.gemm_mt(qt, Ws, n_rows, cfg.id, Q, nt_s, threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    ops = 2 * nt_s * n_rows * cfg.id * args.steps
    value = ops / dt / 1e12
    sample = (f"per step: oracle q8_0 quantization of {nt_s} of {cfg.nt} tokens (id={cfg.id}) + "
              f"fp64 GEMM of those tokens x {n_rows} of {cfg.od} weight rows over {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "strong" if args.gpus > 1 else "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_name(cfg, args), "qtype": cfg.qtype, "od": cfg.od, "id": cfg.id,
                   "nt": cfg.nt, "sample_tokens": nt_s, "sample_rows": n_rows},
        "tokens_per_s": value * 1e12 / (2 * cfg.od * cfg.id),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "cpu_model": _cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- GPU arm
def _graph_time_us(stream, calls, reps=3):
    """Average device time of one call of `calls` (a list of zero-argument
    callables run in order, one "call" each) captured as one CUDA graph and
    replayed `reps` times; CUDA events on the launching stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    with torch.cuda.stream(stream):
        g.replay()  # upload and first-touch costs
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            e0.record()
            g.replay()
            e1.record()
        stream.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / len(calls))
    del g
    return statistics.median(times)


class _Workload:
    """A workload's device inputs on one rank: rotating sets of (weight
    handle, X, Q, Y), larger than twice the L2 together.  With an od slice
    (column-parallel split over ranks) the handles hold rows [o0, o1) only."""

    def __init__(self, args, cfg, rank, dev, o0=0, o1=None, rank_seed=True):
        import torch

        import quantized_int8_gemm_gb300 as mmq
        from quantized_int8_gemm_gb300 import shard
        from synth import gen
        self.cfg = cfg
        self.nt, self.id = cfg.nt, cfg.id
        self.o0, self.o1 = o0, cfg.od if o1 is None else o1
        self.od = self.o1 - self.o0
        seed = cfg.seed + (1000 * rank if rank_seed else 0)
        self.W_host = gen.weights(cfg.qtype, cfg.od, cfg.id, seed, q6_scales=args.q6_scales)
        W_dev = torch.from_numpy(shard.weight_rows(self.W_host, cfg.qtype, cfg.id, self.o0, self.o1)).to(dev)
        self.flags = (mmq.MMQ_REG_WEXP if args.reg_wexp else 0) | (mmq.MMQ_REG_RAW if args.arm == "raw" else 0)
        torch.cuda.synchronize()
        t = time.perf_counter()
        w0 = mmq.mmq_register_weights(cfg.qtype, W_dev, self.od, cfg.id, self.flags)
        self.register_ms = (time.perf_counter() - t) * 1e3
        self.info = mmq.mmq_weights_info(w0)
        nt, id_, od = cfg.nt, cfg.id, self.od
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.per_set = (nt * id_ * 4 + nt * (id_ // 32) * 40 + nt * od * 4 + self.info["operand_bytes"]
                        + self.info["scale_bytes"] + self.info["wexp_bytes"] + nt * id_ * 4
                        + nt * (id_ // 32) * 8)
        self.n_sets = int(min(64, max(2, math.ceil(2 * self.l2 / self.per_set))))
        self.ws = [w0] + [mmq.mmq_register_weights(cfg.qtype, W_dev, od, id_, self.flags)
                          for _ in range(self.n_sets - 1)]
        self.Xs = [torch.from_numpy(gen.activations(nt, id_, seed + 7 * i, cfg.sigma, cfg.outlier_p,
                                                    cfg.outlier_scale)).to(dev) for i in range(self.n_sets)]
        self.Qs = [torch.empty((nt, id_ // 32, 40), dtype=torch.uint8, device=dev) for _ in range(self.n_sets)]
        self.Ys = [torch.empty((nt, od), dtype=torch.float32, device=dev) for _ in range(self.n_sets)]
        del W_dev

    def release(self):
        for w in self.ws:
            w.release()
        self.ws = []


def _measure(args, wl, stream, world, dev, main=True):
    """One workload's numbers on this rank: `value` over K steps captured in
    CUDA graphs (with nvidia-smi clock samples when `main`), the GEMM kernel's
    live event time (second pass), and, when `main`, the separate warm/cold
    timings of quantize_act, gemm and the fused call."""
    import torch

    import quantized_int8_gemm_gb300 as mmq
    cfg, nt, od, id_ = wl.cfg, wl.nt, wl.od, wl.id
    n_sets, ws, Xs, Qs, Ys = wl.n_sets, wl.ws, wl.Xs, wl.Qs, wl.Ys
    fused = args.step == "fused"

    def step(i, ev=None):
        j = i % n_sets
        if fused:  # X -> operand plane -> Y: two kernels
            if ev is None:
                mmq.mmq_gemm_f32(ws[j], Xs[j], Ys[j], flags=ARM[0])
            else:
                mmq.mmq_gemm_f32_profiled(ws[j], Xs[j], Ys[j], ev[0], ev[1], flags=ARM[0])
            return
        mmq.mmq_quantize_act(Xs[j], Qs[j])  # X -> pad40 Q -> operand plane -> Y: three kernels
        if ev is None:
            mmq.mmq_gemm(ws[j], Qs[j], nt, Ys[j], flags=ARM[0])
        else:
            mmq.mmq_gemm_profiled(ws[j], Qs[j], nt, Ys[j], ev[0], ev[1], flags=ARM[0])

    K, Wu = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(Wu):
            step(i)
        if fused:  # one more untimed call that reports the arm the library picked
            arm = mmq.mmq_gemm_f32(ws[0], Xs[0], Ys[0], flags=ARM[0], return_arm=True)[1]
        else:
            mmq.mmq_quantize_act(Xs[0], Qs[0])
            arm = mmq.mmq_gemm(ws[0], Qs[0], nt, Ys[0], flags=ARM[0], return_arm=True)[1]
    stream.synchronize()
    if mmq.mmq_last_device_error() != 0:
        raise RuntimeError("device wait expired during warm-up")
    arm_name = mmq.ARM_NAMES.get(arm, str(arm))
    kernel_name = {mmq.MMQ_ARM_SPLIT: "mmq_gemm_split_kernel",
                   mmq.MMQ_ARM_PAIR: "mmq_gemm_pair_kernel"}.get(arm, "mmq_gemm_kernel")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with torch.cuda.stream(stream):
        for a, b in evs:  # torch creates CUDA events lazily, at the first record
            a.record()
            b.record()
    stream.synchronize()

    # K steps captured as CUDA graphs of at most --graph-chunk steps each:
    # `graphs` plain (the timed pass), `pgraphs` with the GEMM events
    use_graph = not args.no_graph
    graphs, pgraphs = [], []
    if use_graph:
        try:
            for with_ev, out in ((False, graphs), (True, pgraphs)):
                for c0 in range(0, K, args.graph_chunk):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for k in range(c0, min(K, c0 + args.graph_chunk)):
                            step(k, evs[k] if with_ev else None)
                    out.append(g)
            with torch.cuda.stream(stream):
                for g in graphs + pgraphs:  # untimed pass: upload and first-touch costs
                    g.replay()
            stream.synchronize()
        except Exception as e:  # capture unsupported here: time eager launches
            print(f"[bench] graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graphs, pgraphs, use_graph = [], [], False
            torch.cuda.synchronize()

    sampler = ClockSampler(_gpu_uuid(dev)).start() if main else None
    if main:
        time.sleep(0.6)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev_all0, ev_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        ev_all0.record()
        if graphs:
            for g in graphs:
                g.replay()
        else:
            for k in range(K):
                step(k)
        ev_all1.record()
    stream.synchronize()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None
    if mmq.mmq_last_device_error() != 0:
        raise RuntimeError("device wait expired in the timed region")

    # the same K steps again, with CUDA events around every GEMM kernel
    torch.cuda.synchronize()
    ev_p0, ev_p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev_p0.record()
        if pgraphs:
            for g in pgraphs:
                g.replay()
        else:
            for k in range(K):
                step(k, evs[k])
        ev_p1.record()
    stream.synchronize()
    if mmq.mmq_last_device_error() != 0:
        raise RuntimeError("device wait expired in the profiled pass")
    del graphs, pgraphs

    elapsed_ms = _max_over_ranks(ev_all0.elapsed_time(ev_all1), world, dev)
    gemm_ms = [a.elapsed_time(b) for a, b in evs]
    gemm_avg_ms = _max_over_ranks(sum(gemm_ms) / len(gemm_ms), world, dev)

    # ---- roofline of the GEMM kernel (tensor-bound: fp16 UMMA carrying exact integers)
    ops_local = 2 * nt * od * id_
    peaks, peak_src = _peaks()
    long_region = elapsed_ms > 1000.0
    peak = peaks["bf16_tflops_sustained" if long_region else "bf16_tflops"]
    achieved = ops_local / (gemm_avg_ms * 1e-3) / 1e12
    wname = _workload_name(cfg, args)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": _profiled_traffic(wname, kernel_name) if world == 1 else None,
                "peak_source": f"{peak_src} {'sustained' if long_region else 'burst'} bf16 "
                               f"(fp16 UMMA runs at the bf16 rate)",
                "kernel": kernel_name, "arm": arm_name, "gemm_ms_avg": gemm_avg_ms,
                "timing": "CUDA events around each GEMM launch, second pass over the same K steps "
                          f"(that pass: {ev_p0.elapsed_time(ev_p1) / K * 1e3:.1f} us per step)",
                "hbm_floor_us": (wl.info["operand_bytes"] + nt * id_ * 2 + nt * od * 4) /
                                (peaks["hbm_gbs"] * 1e9) * 1e6}
    out = {"elapsed_ms": elapsed_ms, "ms_per_step": elapsed_ms / K, "arm": arm_name, "kernel": kernel_name,
           "roofline": roofline, "clocks": clocks, "use_graph": use_graph, "n_graphs": -(-K // args.graph_chunk)}

    if main and use_graph and not args.no_timings:
        out["timings"] = _separate_timings(wl, stream, peaks)
    return out


def _separate_timings(wl, stream, peaks, reps=200):
    """quantize_act, gemm (from pad40 Q) and the fused call, each as a CUDA
    graph of `reps` calls: "cold" rotates over the input sets (operands come
    from HBM), "warm" repeats set 0 (operands that fit stay in L2)."""
    import quantized_int8_gemm_gb300 as mmq
    nt, id_ = wl.nt, wl.id
    n = wl.n_sets
    res = {}
    for mode in ("cold", "warm"):
        pick = (lambda i: i % n) if mode == "cold" else (lambda i: 0)
        res[f"quantize_act_{mode}_us"] = _graph_time_us(
            stream, [lambda j=pick(i): mmq.mmq_quantize_act(wl.Xs[j], wl.Qs[j]) for i in range(reps)])
        res[f"gemm_{mode}_us"] = _graph_time_us(
            stream, [lambda j=pick(i): mmq.mmq_gemm(wl.ws[j], wl.Qs[j], nt, wl.Ys[j], flags=ARM[0]) for i in range(reps)])
        res[f"fused_{mode}_us"] = _graph_time_us(
            stream, [lambda j=pick(i): mmq.mmq_gemm_f32(wl.ws[j], wl.Xs[j], wl.Ys[j], flags=ARM[0]) for i in range(reps)])
    if mmq.mmq_last_device_error() != 0:
        raise RuntimeError("device wait expired in the separate timings")
    qbytes = nt * id_ * 4 + nt * (id_ // 32) * 40  # read X, write the pad40 blocks: 168 B per block
    gbs = qbytes / (res["quantize_act_cold_us"] * 1e-6) / 1e9
    res["quantize_act_roofline"] = {"bound": "hbm", "bytes_per_call": qbytes, "achieved": gbs,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": gbs / peaks["hbm_gbs"], "timing": "cold"}
    res["how"] = (f"each a CUDA graph of {reps} calls, median of 3 replays, CUDA events; gemm = "
                  "mmq_gemm from pad40 blocks (its prepass + GEMM kernels); fused = mmq_gemm_f32; "
                  f"cold rotates over {n} input sets > 2 x L2, warm repeats one set")
    return res


def _e2e(args, wl, stream, world, dev, ops, d2h_bytes):
    """The same metric end to end through the C ABI: pinned host X -> device,
    the GEMM, Y -> pinned host, every step."""
    import torch

    import quantized_int8_gemm_gb300 as mmq
    from synth import gen
    cfg, nt, od, id_ = wl.cfg, wl.nt, wl.od, wl.id
    n_sets, ws, Xs, Qs, Ys = wl.n_sets, wl.ws, wl.Xs, wl.Qs, wl.Ys
    fused = args.step == "fused"
    E = max(5, min(args.steps, args.e2e_steps))
    Xh = [torch.from_numpy(gen.activations(nt, id_, cfg.seed + 7 * i, cfg.sigma, cfg.outlier_p,
                                           cfg.outlier_scale)).pin_memory()
          for i in range(2)]
    Yh = [torch.empty((nt, od), dtype=torch.float32).pin_memory() for _ in range(2)]
    # Three streams, pipelined across steps: step i's host->device copy runs
    # while step i-1 computes and step i-2's result goes back.  Every step
    # still copies its own input in and its own result out.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    done_c = [torch.cuda.Event() for _ in range(n_sets)]  # compute of the last step on set j
    done_o = [torch.cuda.Event() for _ in range(n_sets)]  # read-back of the last step on set j
    started = [False] * n_sets

    def e2e_step(i):
        j = i % n_sets
        ev_in = torch.cuda.Event()
        with torch.cuda.stream(s_in):
            if started[j]:
                s_in.wait_event(done_c[j])  # set j's X is free once its last step computed
            Xs[j].copy_(Xh[i % 2], non_blocking=True)
            ev_in.record()
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in)
            if started[j]:
                stream.wait_event(done_o[j])  # set j's Y is free once read back
            if fused:
                mmq.mmq_gemm_f32(ws[j], Xs[j], Ys[j], flags=ARM[0])
            else:
                mmq.mmq_quantize_act(Xs[j], Qs[j])
                mmq.mmq_gemm(ws[j], Qs[j], nt, Ys[j], flags=ARM[0])
            done_c[j].record()
        with torch.cuda.stream(s_out):
            s_out.wait_event(done_c[j])
            Yh[i % 2].copy_(Ys[j], non_blocking=True)
            done_o[j].record()
        started[j] = True

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    # The E steps captured as one CUDA graph (the same calls, copies included;
    # the C ABI takes its scratch from graph memory nodes while capturing), so
    # the host's launch rate does not set the step time.
    ge = None
    if not args.no_graph:
        try:
            started[:] = [False] * n_sets  # no waits on events recorded before the capture
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream):
                for st in (s_in, s_out):
                    st.wait_stream(stream)
                for i in range(E):
                    e2e_step(i)
                stream.wait_stream(s_in)
                stream.wait_stream(s_out)
            ge.replay()
            torch.cuda.synchronize()
        except Exception as ex:
            print(f"[bench] e2e graph capture failed ({ex}); timing eager steps", file=sys.stderr)
            ge = None
            torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        if ge is not None:
            ge.replay()
    if ge is None:
        for st in (s_in, s_out):
            st.wait_event(e0)
        for i in range(E):
            e2e_step(i)
    with torch.cuda.stream(stream):
        stream.wait_stream(s_out)
        e1.record()
    torch.cuda.synchronize()
    e_ms = _max_over_ranks(e0.elapsed_time(e1), world, dev)
    return {"value": ops * E / (e_ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": world * nt * id_ * 4, "d2h_bytes_per_step": d2h_bytes,
            "steps": E, "ms_per_step": e_ms / E,
            "path": ("pinned host X -> device, mmq_gemm_f32, Y -> pinned host" if fused else
                     "pinned host X -> device, mmq_quantize_act, mmq_gemm, Y -> pinned host"),
            "overlap": "copies in, compute and copies out on three streams, pipelined across steps",
            "launch": "the E steps as one CUDA graph" if ge is not None else "eager"}


def run_engines():
    """One JSON line: the rates of the exact-integer-capable engines -- the
    library's own probe loops (tcgen05 kind::f16 per SM, mma.sync s8 and f16)
    and, as library references, torch._int_mm (int8) and torch fp16 matmul at
    8192^3, best of 10 each."""
    import torch

    import quantized_int8_gemm_gb300 as mmq
    from quantized_int8_gemm_gb300 import build as mbuild
    mbuild.build()
    torch.cuda.set_device(0)
    rates = mmq.mmq_probe_engine_rates()
    dev = torch.device("cuda")
    props = torch.cuda.get_device_properties(dev)
    n = 8192

    def best_ms(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return min(ts)

    a8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
    b8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
    int_mm = 2 * n ** 3 / (best_ms(lambda: torch._int_mm(a8, b8)) * 1e-3) / 1e12
    a16, b16 = a8.half(), b8.half()
    f16 = 2 * n ** 3 / (best_ms(lambda: torch.matmul(a16, b16)) * 1e-3) / 1e12
    clocks = _clock_snapshot()
    out = {"engines": rates, "torch_int_mm_8192_tops": int_mm, "torch_fp16_matmul_8192_tflops": f16,
           "sms": props.multi_processor_count, "gpu": props.name, "sm_clock_mhz_after": clocks}
    m = rates["umma_f16_mac_per_clk_per_sm"]["N128"]
    if clocks:
        out["umma_f16_tflops_at_that_clock"] = 2 * m * props.multi_processor_count * clocks * 1e6 / 1e12
    print(json.dumps(out), flush=True)


def _clock_snapshot():
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm", "--format=csv,noheader,nounits", "-i", "0"],
                           capture_output=True, text=True, timeout=10)
        return float(r.stdout.strip().splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        return None


# the other q-proj workload, timed beside the default one in the same run
ALSO_WORKLOADS = {DEFAULT_WORKLOAD: ["q6_K_qproj_3584x3584_nt512"]}


def run_mine(args, cfg, rank, world):
    import torch

    from quantized_int8_gemm_gb300 import build as mbuild
    from quantized_int8_gemm_gb300 import shard
    from synth import gen

    mbuild.build()
    local = _env_int("LOCAL_RANK", 0)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream()
    split_od = world > 1 and args.parallel == "od-split"
    # N > 1, od-split: rank r registers rows [o0, o1) of the one weight and
    # computes Y[:, o0:o1] from the same activations (column-parallel, total
    # work fixed); replicas: every rank runs the whole problem on its own batch
    o0, o1 = shard.od_slices(cfg.od, world)[rank] if split_od else (0, cfg.od)
    wl = _Workload(args, cfg, rank, dev, o0, o1, rank_seed=not split_od)
    res = _measure(args, wl, stream, world, dev, main=True)
    K, Wu = args.steps, args.warmup
    ops_step = cfg.ops if split_od else world * cfg.ops  # the whole job's work per step
    value = ops_step * K / (res["elapsed_ms"] * 1e-3) / 1e12
    tokens_per_s = (1 if split_od else world) * cfg.nt * K / (res["elapsed_ms"] * 1e-3)
    d2h = cfg.nt * (cfg.od if split_od else world * cfg.od) * 4  # every Y element read back once
    e2e = None if args.no_e2e else _e2e(args, wl, stream, world, dev, ops_step, d2h)
    wname = _workload_name(cfg, args)

    also = {}
    if world == 1 and not args.no_also:
        for name in ALSO_WORKLOADS.get(cfg.name, []):
            acfg = gen.config_by_name(name)
            awl = _Workload(args, acfg, rank, dev)
            ares = _measure(args, awl, stream, world, dev, main=False)
            also[_workload_name(acfg, args)] = {
                "value": acfg.ops * K / (ares["elapsed_ms"] * 1e-3) / 1e12, "unit": UNIT,
                "ms_per_step": ares["ms_per_step"], "steps": K, "warmup": Wu,
                "tokens_per_s": acfg.nt * K / (ares["elapsed_ms"] * 1e-3),
                "config": {"workload": _workload_name(acfg, args), "qtype": acfg.qtype, "od": acfg.od,
                           "id": acfg.id, "nt": acfg.nt},
                "roofline": ares["roofline"], "gpu_launches": (2 if args.step == "fused" else 3) * K}
            awl.release()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = _oracle_baseline(cfg, wl.W_host, wl.Xs[0].cpu().numpy(), args.cpu_seconds)

    if rank == 0:
        fused = args.step == "fused"
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": Wu, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "strong" if split_od else "weak",
            "vs_baseline": (value / PAGES_TOPS[wname]) if wname in PAGES_TOPS else None,
            "dtype": "s8 x k-quant ints on f16 UMMA, f32 accumulate", "data": "synthetic",
            "config": {"workload": wname, "qtype": cfg.qtype, "od": cfg.od, "id": cfg.id, "nt": cfg.nt,
                       "step": ("mmq_gemm_f32 (fused q8_0 quantization + GEMM)" if fused
                                else "mmq_quantize_act + mmq_gemm"),
                       "cuda_graph": (f"{res['n_graphs']} graphs of <= {args.graph_chunk} steps"
                                      if res["use_graph"] else False),
                       "gemm_launch": "programmatic (overlaps the quantization kernel's tail)",
                       "l2": f"inputs larger than L2: {wl.n_sets} rotating sets x "
                             f"{wl.per_set / 2**20:.1f} MiB > 2 x {wl.l2 / 2**20:.0f} MiB",
                       "register_ms_once": wl.register_ms,
                       "registration": "MMQ_REG_WEXP (operand plane built from W_exp)" if args.reg_wexp
                                       else "default",
                       "parallelism": (f"od-split column-parallel over {world} GPUs: rank r owns weight rows "
                                       f"{shard.od_slices(cfg.od, world)}[r], activations replicated, "
                                       "Y column slices not gathered (the consumer is sharded)")
                                      if split_od else ("replicas" if world > 1 else "single GPU")},
            "tokens_per_s": tokens_per_s,
            "impl": "mine",
            "roofline": res["roofline"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (2 if fused else 3) * K,
            "clocks": res["clocks"],
        }
        if "timings" in res:
            line["timings"] = res["timings"]
        if also:
            line["also"] = also
        print(json.dumps(line), flush=True)
    wl.release()
    if world > 1:
        torch.distributed.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("mine", "reference"), default="mine")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--graph-chunk", type=int, default=500)
    ap.add_argument("--step", choices=("fused", "two"), default="fused",
                    help="fused: mmq_gemm_f32; two: mmq_quantize_act then mmq_gemm")
    ap.add_argument("--q6-scales", choices=("small", "int8"), default="small",
                    help="q6_K sub-block scales: small = the workloads' recipe, uniform in [-32, 31]; "
                         "int8 = the format's usual encoding over the int8 range (two-plane operand); "
                         "the workload is then named <workload>_int8scales")
    ap.add_argument("--parallel", choices=("od-split", "replicas"), default="od-split",
                    help="N > 1: od-split = each rank one slice of the weight rows (column-parallel); "
                         "replicas = each rank the whole problem on its own batch")
    ap.add_argument("--reg-wexp", action="store_true",
                    help="register with MMQ_REG_WEXP: the operand plane is built from the dense W_exp "
                         "plane (the workload is then named <workload>_wexp)")
    ap.add_argument("--no-also", action="store_true", help="skip the other q-proj workload")
    ap.add_argument("--arm", choices=("auto", "f16", "raw", "split", "pair"), default="auto",
                    help="force one GEMM arm (default: the library's choice)")
    ap.add_argument("--engines", action="store_true",
                    help="print the tensor engines' rates (the library's probe, torch._int_mm and fp16 matmul) "
                         "instead of a bench line")
    ap.add_argument("--nt", type=int, default=None,
                    help="run the workload's shape and generators at this many tokens (the name's _nt suffix "
                         "follows)")
    ap.add_argument("--no-timings", action="store_true",
                    help="skip the separate quantize_act / gemm / fused timings")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ARM[0] = {"auto": 0, "f16": 1, "raw": 2, "split": 3, "pair": 4}[args.arm]
    from synth import gen
    cfg = gen.config_by_name(args.workload)
    if args.nt is not None:  # the workload's weights and generators at another token count
        import dataclasses
        if args.nt <= 0:
            ap.error("--nt must be positive")
        cfg = dataclasses.replace(cfg, nt=args.nt, name=re.sub(r"_nt\d+$", f"_nt{args.nt}", cfg.name))
    rank, world = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1)
    if args.engines:
        run_engines()
        return
    if args.impl == "reference":
        run_reference(args, cfg, rank)
    else:
        run_mine(args, cfg, rank, world)


if __name__ == "__main__":
    main()
