"""mmq_gemm_noalloc: the GEMM entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc -- a process whose device
memory is owned by another allocator, or a path that cannot accept
cudaMalloc's implicit synchronization -- by using a fixed 16 MiB scratch
array compiled into the library.  These tests call it through the C ABI and
compare it with mmq_gemm's fp16-plane arm (bit for bit where that arm, like
the no-alloc one, runs whole tiles) and with the oracle.  The file name
makes pytest collect it last, so a failure here never hides the rest of the
suite.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle
from synth import gen

pytestmark = pytest.mark.gpu

MMQ_ERR_SCRATCH_LIMIT = -9
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
QT = {"q4_K": oracle.Q4_K, "q6_K": oracle.Q6_K}


@pytest.fixture(scope="module")
def mmq():
    from quantized_int8_gemm_gb300 import build
    build.build()
    import quantized_int8_gemm_gb300 as m
    m.load()
    return m


def _noalloc(mmq, w, Q, nt, Y):
    return mmq.load().mmq_gemm_noalloc(w.handle, Q.data_ptr(), nt, Y.data_ptr(), None)


def _sampled(nt, od, n, seed):
    rng = np.random.default_rng(seed)
    ts = np.concatenate([rng.integers(0, nt, n), [0, nt - 1, min(127, nt - 1), min(128, nt - 1)]])
    os_ = np.concatenate([rng.integers(0, od, n), [od - 1, 0, min(128, od - 1), min(127, od - 1)]])
    return ts.astype(np.int64), os_.astype(np.int64)


# Shapes whose fp16-plane GEMM in mmq_gemm runs whole tiles (no stream-K
# split), as the no-alloc entry point always does: the two results are then
# the same kernel on the same operands, equal bit for bit.
@pytest.mark.parametrize("qtype,od,id_,nts", [("q4_K", 3584, 3584, (512, 640)),
                                              ("q6_K", 256, 512, (16, 129))])
def test_noalloc_matches_gemm_on_two_calls_in_a_row(mmq, qtype, od, id_, nts):
    dev = torch.device("cuda")
    W = gen.weights(qtype, od, id_, 71)
    w = mmq.mmq_register_weights(qtype, torch.from_numpy(W).to(dev), od, id_)
    for call, nt in enumerate(nts):  # the second call reuses the buffer the first left behind
        X = gen.activations(nt, id_, seed=80 + call, outlier_p=0.01, outlier_scale=20.0)
        Q = mmq.mmq_quantize_act(torch.from_numpy(X).to(dev))
        Y_ref = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_F16)
        Y = torch.full((nt, od), float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc(mmq, w, Q, nt, Y) == 0
        torch.cuda.synchronize()
        assert mmq.mmq_last_device_error() == 0
        assert torch.equal(Y, Y_ref), call
        # and against the oracle, within the GEMM tolerance
        ts, os_ = _sampled(nt, od, 2000, 90 + call)
        y_ref = oracle.gemm_entries(QT[qtype], W, od, id_, Q.cpu().numpy(), nt, ts, os_)
        err = np.abs(Y.cpu().numpy()[ts, os_].astype(np.float64) - y_ref).max()
        assert err <= 1e-3 * np.abs(y_ref).max() + 1e-5, (call, err)
    w.release()


def test_noalloc_matches_gemm_where_gemm_splits_tiles(mmq):
    """A shape where mmq_gemm's fp16-plane arm splits tiles between CTAs
    (stream-K, another summation order): equal within the GEMM tolerance, and
    the no-alloc result against the oracle element by element."""
    dev = torch.device("cuda")
    qtype, od, id_, nt = "q6_K", 1000, 2048, 129
    W = gen.weights(qtype, od, id_, 73)
    w = mmq.mmq_register_weights(qtype, torch.from_numpy(W).to(dev), od, id_)
    X = gen.activations(nt, id_, seed=74, outlier_p=0.01, outlier_scale=20.0)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).to(dev))
    Y = torch.full((nt, od), float("nan"), dtype=torch.float32, device=dev)
    for _ in range(2):
        assert _noalloc(mmq, w, Q, nt, Y) == 0
    Y_ref = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_F16)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    a, b = Y.cpu().numpy().astype(np.float64), Y_ref.cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    assert np.abs(a - b).max() <= 1e-3 * np.abs(b).max() + 1e-5
    y_or = oracle.gemm(oracle.Q6_K, W, od, id_, Q.cpu().numpy(), nt)
    assert np.abs(a - y_or).max() <= 1e-3 * np.abs(y_or).max() + 1e-5
    w.release()


def test_noalloc_rejects_problems_beyond_its_fixed_scratch(mmq):
    dev = torch.device("cuda")
    od, id_ = 128, 3584
    w = mmq.mmq_register_weights("q4_K", torch.from_numpy(gen.weights("q4_K", od, id_, 72)).to(dev),
                                 od, id_)
    nt_ok, nt_big = 2048, 2049  # 16 MiB holds 2048 tokens at id = 3584 (q4_K)
    X = torch.zeros((nt_big, id_), dtype=torch.float32, device=dev)
    Q = mmq.mmq_quantize_act(X)
    Y = torch.empty((nt_big, od), dtype=torch.float32, device=dev)
    assert _noalloc(mmq, w, Q, nt_big, Y) == MMQ_ERR_SCRATCH_LIMIT
    assert _noalloc(mmq, w, Q, nt_ok, Y) == 0
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert not Y[:nt_ok].any()
    w.release()


# Run in a fresh interpreter: registration, then the no-alloc GEMM as the very
# first GEMM call of the process, with the device's free memory read before
# and after it.  Registration has loaded the GEMM's module and kernels, so
# the call must not lower the free memory (lazy module loading would take the
# 16 MiB array and the kernels' code right there).
_FIRST_CALL = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import quantized_int8_gemm_gb300 as mmq
    from synth import gen
    L = mmq.load()
    dev = torch.device("cuda")
    for qtype, od, id_, nt, seed in (("q4_K", 3584, 3584, 512, 75), ("q6_K", 384, 1024, 200, 76)):
        W = gen.weights(qtype, od, id_, seed)
        X = gen.activations(nt, id_, seed=seed + 1)
        w = mmq.mmq_register_weights(qtype, torch.from_numpy(W).to(dev), od, id_)
        Q = mmq.mmq_quantize_act(torch.from_numpy(X).to(dev))
        Y = torch.full((nt, od), float("nan"), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = L.mmq_gemm_noalloc(w.handle, Q.data_ptr(), nt, Y.data_ptr(), None)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert rc == 0, rc
        assert mmq.mmq_last_device_error() == 0
        assert free1 >= free0, (qtype, free0, free1)
        Yf = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_F16)
        torch.cuda.synchronize()
        assert torch.equal(Y, Yf), qtype
        w.release()
    print("FIRST_CALL_OK")
""")


def test_noalloc_first_gemm_call_of_a_process_allocates_nothing(mmq):
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL.format(root=ROOT)], capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "FIRST_CALL_OK" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
