"""GPU parity of the pair arm (MMQ_ARM_PAIR: the split arm's operands on 2-CTA
clusters with cta_group::2 UMMAs) against the oracle, element by element on
small shapes and on sampled outputs at the q-proj workloads' full size, and
against the 128-row split arm, whose exact products and epilogue operations it
repeats per output with the tile transposed."""
import numpy as np
import pytest
import torch

import oracle
from synth import gen

pytestmark = pytest.mark.gpu

QT = {"q4_K": oracle.Q4_K, "q6_K": oracle.Q6_K}


@pytest.fixture(scope="module")
def mmq():
    from quantized_int8_gemm_gb300 import build
    build.build()
    import quantized_int8_gemm_gb300 as m
    m.load()
    assert torch.cuda.is_available()
    return m


def _within_tol(y_gpu, y_ref):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref).max() if y_ref.size else 0.0
    bound = 1e-3 * (np.abs(y_ref).max() if y_ref.size else 0.0) + 1e-5
    return err, bound


def _sample_entries(nt, od, n, seed):
    rng = np.random.default_rng(seed)
    ts = list(rng.integers(0, nt, n))
    os_ = list(rng.integers(0, od, n))
    for t in {0, min(63, nt - 1), min(64, nt - 1), min(127, nt - 1), min(128, nt - 1), nt - 1}:
        for o in {0, min(127, od - 1), min(128, od - 1), min(255, od - 1), min(256, od - 1), od - 1}:
            ts.append(t)
            os_.append(o)
    return np.array(ts, dtype=np.int64), np.array(os_, dtype=np.int64)


PAIR_SHAPES = [
    ("q6_K", 256, 512, 16, 1),     # one pair, one token tile
    ("q4_K", 260, 512, 129, 2),    # 3 weight tiles: the second pair repeats its tile; ragged tokens
    ("q6_K", 300, 768, 200, 3),
    ("q4_K", 131, 256, 1, 4),      # one super-block, one token
    ("q4_K", 384, 1024, 256, 5),
    ("q6_K", 1000, 4096, 300, 6),
    ("q6_K", 3456, 3584, 300, 7),  # 27 weight tiles
    ("q4_K", 896, 7168, 200, 8),   # 28 super-blocks per tile
    ("q6_K", 130, 22016, 70, 9),
]


@pytest.mark.parametrize("name,od,id_,nt,seed", PAIR_SHAPES)
def test_pair_arm_parity(mmq, name, od, id_, nt, seed):
    W = gen.weights(name, od, id_, seed=900 + seed)
    X = gen.activations(nt, id_, seed=950 + seed, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Q = mmq.mmq_quantize_act(Xd)
    Yp, arm = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_PAIR, return_arm=True)
    assert arm == mmq.MMQ_ARM_PAIR
    Yf = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_PAIR)
    Ys = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_SPLIT)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert torch.equal(Yp, Yf)          # the same operands from X or from Q
    Y_ref = oracle.gemm(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt)
    err, bound = _within_tol(Yp.cpu().numpy(), Y_ref)
    assert err <= bound, (err, bound)
    scale = float(np.abs(Y_ref).max()) + 1e-30
    assert float((Yp - Ys).abs().max()) / scale < 1e-5
    w.release()


@pytest.mark.parametrize("name", ["q4_K", "q6_K"])
def test_pair_arm_against_split_arm(mmq, name):
    """Per output the same exact products and the same fp32 epilogue
    operations as the 128-row split kernel, but the tensor core sums a
    super-block of the transposed tile in its own internal order: the arms
    agree to about one fp32 unit of the largest output, not bit for bit (a
    shape where the split arm runs whole 128-row tiles)."""
    od, id_, nt = 1000, 4096, 300
    W = gen.weights(name, od, id_, seed=990)
    X = gen.activations(nt, id_, seed=991)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Yp = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_PAIR)
    Ys = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert float((Yp - Ys).abs().max()) <= 2.0 ** -20 * float(Ys.abs().max())
    w.release()


@pytest.mark.parametrize("name", ["q4_K", "q6_K"])
def test_pair_arm_many_units_per_pair(mmq, name):
    """More units than pairs: each pair loops over several tiles, carrying its
    ring, region and scale-entry phases across them."""
    od, id_, nt = 3584, 512, 2176
    W = gen.weights(name, od, id_, seed=992)
    X = gen.activations(nt, id_, seed=993, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Y = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_PAIR)
    Y2 = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_PAIR)
    Y16 = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_F16)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert torch.equal(Y, Y2)           # deterministic
    ts, os_ = _sample_entries(nt, od, 4000, 994)
    y_ref = oracle.gemm_entries(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt, ts, os_)
    err, bound = _within_tol(Y.cpu().numpy()[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    assert float((Y - Y16).abs().max()) <= 1e-5 * float(Y16.abs().max())
    w.release()


@pytest.mark.parametrize("cfg", [c for c in gen.CONFIGS if c.od == 3584 and c.id == 3584],
                         ids=lambda c: c.name)
def test_pair_arm_qproj_workloads_sampled(mmq, cfg):
    W, X = gen.config_inputs(cfg)
    w = mmq.mmq_register_weights(cfg.qtype, torch.from_numpy(W).cuda(), cfg.od, cfg.id)
    Xd = torch.from_numpy(X).cuda()
    Y = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_PAIR)
    Ys = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    ts, os_ = _sample_entries(cfg.nt, cfg.od, 3000, cfg.seed + 5)
    y_ref = oracle.gemm_entries(QT[cfg.qtype], W, cfg.od, cfg.id, oracle.quantize_q8_0(X), cfg.nt, ts, os_)
    err, bound = _within_tol(Y.cpu().numpy()[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    assert float((Y - Ys).abs().max()) <= 1e-5 * float(Ys.abs().max())
    w.release()


def test_pair_arm_refuses_two_plane_handles(mmq):
    od, id_ = 256, 512
    W = gen.weights("q6_K", od, id_, seed=995, q6_scales="int8")
    w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), od, id_)
    X = torch.from_numpy(gen.activations(16, id_, seed=996)).cuda()
    with pytest.raises(mmq.MMQError):
        mmq.mmq_gemm_f32(w, X, flags=mmq.MMQ_ARM_PAIR)
    w.release()


@pytest.mark.parametrize("cfg", [c for c in gen.CONFIGS if c.od * c.id > 3584 * 3584], ids=lambda c: c.name)
def test_pair_arm_ffn_workloads_sampled(mmq, cfg):
    """The FFN workloads: many tiles per SM pair, 128-token tiles."""
    W, X = gen.config_inputs(cfg)
    w = mmq.mmq_register_weights(cfg.qtype, torch.from_numpy(W).cuda(), cfg.od, cfg.id)
    Y = mmq.mmq_gemm_f32(w, torch.from_numpy(X).cuda(), flags=mmq.MMQ_ARM_PAIR).cpu().numpy()
    assert mmq.mmq_last_device_error() == 0
    ts, os_ = _sample_entries(cfg.nt, cfg.od, 800, cfg.seed + 6)
    y_ref = oracle.gemm_entries(QT[cfg.qtype], W, cfg.od, cfg.id, oracle.quantize_q8_0(X), cfg.nt, ts, os_)
    err, bound = _within_tol(Y[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    w.release()
