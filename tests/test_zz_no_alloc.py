"""mmq_gemm_noalloc: the GEMM entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc -- a process whose device
memory is owned by another allocator, or a path that cannot accept
cudaMalloc's implicit synchronization -- by using a fixed 16 MiB scratch
array compiled into the library.  These tests call it through the C ABI and
compare it with mmq_gemm.  The file name makes pytest collect it last, so a
failure here never hides the rest of the suite.
"""
import numpy as np
import pytest
import torch

from synth import gen

pytestmark = pytest.mark.gpu

MMQ_ERR_SCRATCH_LIMIT = -9


@pytest.fixture(scope="module")
def mmq():
    from quantized_int8_gemm_gb300 import build
    build.build()
    import quantized_int8_gemm_gb300 as m
    m.load()
    return m


def _noalloc(mmq, w, Q, nt, Y):
    return mmq.load().mmq_gemm_noalloc(w.handle, Q.data_ptr(), nt, Y.data_ptr(), None)


@pytest.mark.parametrize("qtype,od,id_,nts", [("q4_K", 3584, 3584, (512, 300)),
                                              ("q6_K", 1000, 2048, (129, 700))])
def test_noalloc_matches_gemm_on_two_calls_in_a_row(mmq, qtype, od, id_, nts):
    dev = torch.device("cuda")
    w = mmq.mmq_register_weights(qtype, torch.from_numpy(gen.weights(qtype, od, id_, 71)).to(dev),
                                 od, id_)
    for call, nt in enumerate(nts):  # the second call reuses the buffer the first left behind
        X = gen.activations(nt, id_, seed=80 + call, outlier_p=0.01, outlier_scale=20.0)
        Q = mmq.mmq_quantize_act(torch.from_numpy(X).to(dev))
        Y_ref = mmq.mmq_gemm(w, Q, nt)
        Y = torch.full((nt, od), float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc(mmq, w, Q, nt, Y) == 0
        torch.cuda.synchronize()
        assert mmq.mmq_last_device_error() == 0
        a, b = Y.cpu().numpy().astype(np.float64), Y_ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all()
        err = np.abs(a - b).max()
        assert err <= 1e-3 * np.abs(b).max() + 1e-5, (call, err)
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
