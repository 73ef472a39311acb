"""GEMM calls captured in a CUDA graph and replayed with new inputs give the
eager calls' results bit for bit.  A replayed graph repeats each launch's
arguments -- its epoch among them -- and its scratch, so every hand-off
between CTAs that lives in scratch has to start clear in each replay: the
fp16-plane arm's stream-K flags (tagged with the epoch), the split arm's
per-tile piece counters; the pair arm holds none."""
import pytest
import torch

from synth import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mmq():
    from quantized_int8_gemm_gb300 import build
    build.build()
    import quantized_int8_gemm_gb300 as m
    m.load()
    assert torch.cuda.is_available()
    return m


def _graph_replays_match(mmq, w, id_, nt, flags, seed):
    """Two calls captured in one CUDA graph on static inputs; the inputs are
    rewritten and the graph replayed three times; each replay's outputs equal
    eager calls on the same inputs."""
    X1 = torch.empty((nt, id_), dtype=torch.float32, device="cuda")
    X2 = torch.empty_like(X1)
    X1.copy_(torch.from_numpy(gen.activations(nt, id_, seed=seed)))
    X2.copy_(torch.from_numpy(gen.activations(nt, id_, seed=seed + 1)))
    arm = mmq.mmq_gemm_f32(w, X1, flags=flags, return_arm=True)[1]  # (outside the capture: module loading)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        Y1 = mmq.mmq_gemm_f32(w, X1, flags=flags)
        Y2 = mmq.mmq_gemm_f32(w, X2, flags=flags)
    for r in range(3):
        X1.copy_(torch.from_numpy(gen.activations(nt, id_, seed=seed + 10 + 2 * r, outlier_p=0.01,
                                                  outlier_scale=20.0)))
        X2.copy_(torch.from_numpy(gen.activations(nt, id_, seed=seed + 11 + 2 * r)))
        g.replay()
        torch.cuda.synchronize()
        assert mmq.mmq_last_device_error() == 0
        E1 = mmq.mmq_gemm_f32(w, X1, flags=flags)
        E2 = mmq.mmq_gemm_f32(w, X2, flags=flags)
        torch.cuda.synchronize()
        assert torch.equal(Y1, E1), r
        assert torch.equal(Y2, E2), r
    del g
    return arm


@pytest.mark.parametrize("name,od,id_,nt,flags,arm", [
    ("q4_K", 3584, 3584, 512, 0, 4),   # the pair arm (library choice)
    ("q6_K", 3584, 3584, 512, 0, 4),
    ("q6_K", 3584, 3584, 16, 0, 3),    # the split arm's pieces of tiles (per-tile counters)
    ("q6_K", 1000, 4096, 300, 1, 1),   # the fp16-plane arm's stream-K split tiles (tagged flags)
    ("q4_K", 700, 3072, 200, 1, 1),
])
def test_graph_replays_equal_eager_calls(mmq, name, od, id_, nt, flags, arm):
    W = gen.weights(name, od, id_, seed=1400 + nt)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    assert _graph_replays_match(mmq, w, id_, nt, flags, 1410 + od) == arm
    w.release()
