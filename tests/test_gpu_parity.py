"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact for the q8_0 activation blocks and the W_exp plane; for the fp32
GEMM output  max|Y_gpu - Y_ref| <= 1e-3 * max|Y_ref| + 1e-5  (the tolerance
the task states), Y_ref in fp64 from the oracle.  Small shapes are compared
element by element (several tiles, ragged tails); the five workloads at full
size are compared on sampled outputs the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import gen

pytestmark = pytest.mark.gpu

RTOL_MAX = 1e-3
ATOL = 1e-5
QT = {"q4_K": oracle.Q4_K, "q6_K": oracle.Q6_K}
# the four layer-sized workloads (q-proj 3584 x 3584 and the FFN matrices)
FULL_SIZE = [c for c in gen.CONFIGS if c.od * c.id >= 3584 * 3584]


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
    bound = RTOL_MAX * (np.abs(y_ref).max() if y_ref.size else 0.0) + ATOL
    return err, bound


def _run(mmq, qtype, W, od, id_, X, flags=0):
    dev = torch.device("cuda")
    Wd = torch.from_numpy(W).to(dev)
    Xd = torch.from_numpy(X).to(dev)
    Qd = mmq.mmq_quantize_act(Xd)
    w = mmq.mmq_register_weights(qtype, Wd, od, id_, flags)
    Y, arm = mmq.mmq_gemm(w, Qd, X.shape[0], return_arm=True)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    return w, Qd.cpu().numpy(), Y.cpu().numpy(), arm


# ---------------------------------------------------------------- quantizer
@pytest.mark.parametrize("cfg", gen.CONFIGS, ids=lambda c: c.name)
def test_quantize_bit_exact_workloads(mmq, cfg):
    X = gen.activations(cfg.nt, cfg.id, cfg.seed, cfg.sigma, cfg.outlier_p, cfg.outlier_scale)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda()).cpu().numpy()
    assert np.array_equal(Q, oracle.quantize_q8_0(X))


def test_quantize_bit_exact_edge_values(mmq):
    rng = np.random.default_rng(0)
    X = rng.standard_normal((37, 256)).astype(np.float32)
    X[0, :32] = 0.0                                  # all-zero block
    X[1, :32] = 3.0                                  # all-equal block
    X[2, :32] = np.arange(32) - 15.5                 # halves
    X[3, :32] = 0.0
    X[3, 0] = 127.0
    X[3, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5]  # exact ties
    X[4] *= 1e-30                                    # d16 underflows to zero
    X[5] *= 1e-6                                     # subnormal d16
    X[6] *= 7e4                                      # large
    X[7, 32:64] = -0.0
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda()).cpu().numpy()
    assert np.array_equal(Q, oracle.quantize_q8_0(X))


# ---------------------------------------------------------------- W_exp plane
@pytest.mark.parametrize("od,id_", [(256, 512), (70, 256), (3584, 3584), (3584, 18944)])
def test_wexp_plane_bit_exact(mmq, od, id_):
    W = gen.weights("q6_K", od, id_, seed=od + id_)
    w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), od, id_, mmq.MMQ_REG_WEXP)
    plane = mmq.mmq_weights_wexp(w).cpu().numpy()
    assert plane.shape == (od, id_)
    assert np.array_equal(plane, oracle.expand_q6k_dense(W, od, id_))
    info = mmq.mmq_weights_info(w)
    assert info["wexp_bytes"] == od * id_
    w.release()


# ---------------------------------------------------------------- GEMM, full compare
SMALL = [
    ("q6_K", 256, 512, 16, 0),     # workload 0, the tiny q6_K case
    ("q6_K", 300, 768, 200, 1),    # ragged rows and tokens, 3 super-blocks
    ("q4_K", 260, 512, 129, 2),
    ("q4_K", 131, 256, 1, 3),      # one token, od not a multiple of 4
    ("q6_K", 5, 256, 130, 4),      # od < 4, one super-block
    ("q4_K", 384, 1024, 256, 5),   # second token tile starts at i0 = 128
    ("q6_K", 129, 2048, 127, 6),
    ("q4_K", 128, 768, 128, 7),
    # few tiles, many super-blocks: the (tile, super-block) work is split over
    # all SMs, each tile between several CTAs that hand partial sums over
    ("q6_K", 1000, 4096, 300, 8),
    ("q4_K", 700, 3072, 200, 9),
]


@pytest.mark.parametrize("name,od,id_,nt,seed", SMALL)
def test_gemm_parity_full_compare(mmq, name, od, id_, nt, seed):
    W = gen.weights(name, od, id_, seed=100 + seed)
    X = gen.activations(nt, id_, seed=200 + seed, outlier_p=0.01, outlier_scale=20.0)
    _, Q, Y, arm = _run(mmq, name, W, od, id_, X)
    Q_ref = oracle.quantize_q8_0(X)
    assert np.array_equal(Q, Q_ref)
    Y_ref = oracle.gemm(QT[name], W, od, id_, Q_ref, nt)
    err, bound = _within_tol(Y, Y_ref)
    assert err <= bound, (err, bound)
    assert arm in mmq.ARM_NAMES


@pytest.mark.parametrize("od,id_,nt", [(256, 256, 130), (300, 768, 129), (131, 3584, 64)])
def test_gemm_consumes_wexp_plane_with_dense_strides(mmq, od, id_, nt):
    """Offsets gate for the pre-expanded plane: with MMQ_REG_WEXP the q6_K
    operand is rebuilt from the dense W_exp plane, so the GEMM only matches
    the oracle if the plane is read with row pitch id and super-block pitch
    256 (a padded-pitch read shifts every row but row 0)."""
    W = gen.weights("q6_K", od, id_, seed=300 + od)
    X = gen.activations(nt, id_, seed=301 + od)
    w, Q, Y, _ = _run(mmq, "q6_K", W, od, id_, X, flags=mmq.MMQ_REG_WEXP)
    assert np.array_equal(mmq.mmq_weights_wexp(w).cpu().numpy(), oracle.expand_q6k_dense(W, od, id_))
    Y_ref = oracle.gemm(oracle.Q6_K, W, od, id_, oracle.quantize_q8_0(X), nt)
    err, bound = _within_tol(Y, Y_ref)
    assert err <= bound, (err, bound)


# ---------------------------------------------------------------- GEMM, the five workloads at full size
def _sample_entries(nt, od, n, seed):
    rng = np.random.default_rng(seed)
    ts = list(rng.integers(0, nt, n))
    os_ = list(rng.integers(0, od, n))
    # tile edges and the ragged tail
    for t in {0, min(127, nt - 1), min(128, nt - 1), nt - 1}:
        for o in {0, min(127, od - 1), min(128, od - 1), od - 1}:
            ts.append(t)
            os_.append(o)
    return np.array(ts, dtype=np.int64), np.array(os_, dtype=np.int64)


@pytest.mark.parametrize("cfg", gen.CONFIGS, ids=lambda c: c.name)
def test_gemm_parity_workloads_sampled(mmq, cfg):
    W, X = gen.config_inputs(cfg)
    _, Q, Y, _ = _run(mmq, cfg.qtype, W, cfg.od, cfg.id, X)
    Q_ref = oracle.quantize_q8_0(X)
    assert np.array_equal(Q, Q_ref)
    n = 3000 if cfg.id <= 4096 else 800
    ts, os_ = _sample_entries(cfg.nt, cfg.od, n, cfg.seed)
    y_ref = oracle.gemm_entries(QT[cfg.qtype], W, cfg.od, cfg.id, Q_ref, cfg.nt, ts, os_)
    err, bound = _within_tol(Y[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    assert np.isfinite(Y).all()


# ---------------------------------------------------------------- boundary behaviour
def test_error_codes(mmq):
    dev = torch.device("cuda")
    W = torch.from_numpy(gen.weights("q6_K", 8, 256, seed=1)).to(dev)
    with pytest.raises(mmq.MMQError) as e:
        mmq.mmq_register_weights("q6_K", W, 8, 300)
    assert e.value.code == -1
    with pytest.raises(mmq.MMQError) as e:
        mmq.mmq_register_weights(7, W, 8, 256)
    assert e.value.code == -3
    with pytest.raises(mmq.MMQError) as e:
        mmq.mmq_register_weights("q4_K", W, 8, 256, 0x80)  # no such flag
    assert e.value.code == -1
    # a q6_K sub-block scale beyond +-64 (one, in otherwise small scales) takes
    # the two-plane operand; the raw arm has no B0 image and refuses it
    Wb = gen.weights("q6_K", 8, 256, seed=2, q6_scales="small").reshape(8, 210)
    Wb[3, 192 + 5] = np.uint8(np.int8(-100).view(np.uint8))
    wb = mmq.mmq_register_weights("q6_K", torch.from_numpy(Wb.reshape(-1)).to(dev), 8, 256, mmq.MMQ_REG_RAW)
    Xb = gen.activations(4, 256, seed=3)
    Qb4 = mmq.mmq_quantize_act(torch.from_numpy(Xb).to(dev))
    with pytest.raises(mmq.MMQError) as e:
        mmq.mmq_gemm(wb, Qb4, 4, flags=mmq.MMQ_ARM_RAW)
    assert e.value.code == -7
    for arm in (mmq.MMQ_ARM_F16, mmq.MMQ_ARM_SPLIT):
        Yb = mmq.mmq_gemm(wb, Qb4, 4, flags=arm).cpu().numpy()
        err, bound = _within_tol(Yb, oracle.gemm(oracle.Q6_K, Wb.reshape(-1), 8, 256, oracle.quantize_q8_0(Xb), 4))
        assert err <= bound, (arm, err, bound)
    wb.release()
    # misaligned activations
    X = torch.zeros(4 * 256 + 4, dtype=torch.float32, device=dev)
    Qb = torch.empty(4 * 8 * 40, dtype=torch.uint8, device=dev)
    rc = mmq.load().mmq_quantize_act(X.data_ptr() + 4, 4, 256, Qb.data_ptr(), None)
    assert rc == -2
    w = mmq.mmq_register_weights("q6_K", W, 8, 256)
    Q = mmq.mmq_quantize_act(torch.zeros(4, 256, device=dev))
    Y = torch.empty(4 * 8 + 4, dtype=torch.float32, device=dev)
    rc = mmq.load().mmq_gemm(w.handle, Q.data_ptr(), 4, Y.data_ptr() + 4, None, 0, None)
    assert rc == -2
    rc = mmq.load().mmq_gemm(w.handle, Q.data_ptr(), 4, Y.data_ptr(), None, 99, None)
    assert rc == -7
    # nt == 0 is a no-op
    assert mmq.load().mmq_gemm(w.handle, Q.data_ptr(), 0, Y.data_ptr(), None, 0, None) == 0


def test_zero_and_constant_activations(mmq):
    od, id_ = 200, 512
    W = gen.weights("q4_K", od, id_, seed=9)
    X = np.zeros((3, id_), dtype=np.float32)
    X[1] = 0.75
    X[2] = -2.0
    _, _, Y, _ = _run(mmq, "q4_K", W, od, id_, X)
    assert not Y[0].any()
    Y_ref = oracle.gemm(oracle.Q4_K, W, od, id_, oracle.quantize_q8_0(X), 3)
    err, bound = _within_tol(Y, Y_ref)
    assert err <= bound


def _fp16_bits(v):
    return np.frombuffer(np.float16(v).tobytes(), dtype=np.uint8)


def test_extreme_weight_blocks(mmq):
    """The exactness boundary of the fp16 operands and extreme block scales:
    q6_K sub-block scales of exactly +-64 with codes 0 and 63 give |sc*(q-32)|
    up to 2048 (one operand plane); scales -128 and 127 up to 4096 (the B1 + B0
    planes), against rows of +-1 activations (qs = +-127), so a 32-K partial
    reaches 32 * 127 * 4096; q4_K scales and mins of 63 with codes 15; d and
    dmin at the fp16 maximum, at a subnormal and at zero."""
    od, id_, nt = 160, 768, 130
    X = gen.activations(nt, id_, seed=61, outlier_p=0.02, outlier_scale=30.0)
    X[0:8] = 1.0
    X[8:16] = np.where(np.arange(id_) % 64 < 32, 1.0, -1.0).astype(np.float32)
    Q_ref = oracle.quantize_q8_0(X)
    rng = np.random.default_rng(62)
    # q6_K: 210-byte blocks, ql @0, qh @128, sc @192 (int8), d @208
    W6 = gen.weights("q6_K", od, id_, seed=63).reshape(-1, 210).copy()
    n = W6.shape[0]
    W6[:, 192:208] = np.where(rng.random((n, 16)) < 0.5, 64, np.uint8(np.int8(-64).view(np.uint8)))
    W6[0::3, 0:192] = 0xFF       # q = 63
    W6[1::3, 0:192] = 0x00       # q = 0: q - 32 = -32, |sc (q - 32)| = 2048
    # d: the fp16 maximum (on blocks with small codes, so |Y| stays finite), a
    # subnormal, zero, and the generator's values elsewhere
    W6[0::20, 208:210] = _fp16_bits(65504.0)
    W6[0::20, 0:192] = 0x22
    W6[5::20, 208:210] = _fp16_bits(6e-8)
    W6[10::20, 208:210] = _fp16_bits(0.0)
    W6 = W6.reshape(-1)
    # q6_K at the ends of the int8 scale range: the two-plane operand
    W8 = gen.weights("q6_K", od, id_, seed=65).reshape(-1, 210).copy()
    W8[:, 192:208] = np.where(rng.random((n, 16)) < 0.5, 127, np.uint8(np.int8(-128).view(np.uint8)))
    W8[0::3, 0:192] = 0xFF       # q = 63: (q - 32) = 31, 127 * 31 = 3937 (odd)
    W8[1::3, 0:192] = 0x00       # q = 0: -32, -128 * -32 = 4096
    W8 = W8.reshape(-1)
    # q4_K: 144-byte blocks, d @0, dmin @2, packed scales/mins @4, qs @16
    W4 = gen.weights("q4_K", od, id_, seed=64).reshape(-1, 144).copy()
    W4[0::2, 4:16] = 0xFF        # every 6-bit scale and min = 63
    W4[0::4, 16:144] = 0xFF      # codes 15
    W4[1::4, 16:144] = 0x00      # codes 0: only the min term
    for i, (dv, mv) in enumerate([(65504.0, 0.0), (0.0, 2.0), (6e-8, 6e-8), (1e-3, 65504.0)]):
        W4[i::20, 0:2] = _fp16_bits(dv)
        W4[i::20, 2:4] = _fp16_bits(mv)
    big4 = (W4[:, 0:2].view(np.uint16)[:, 0] == 0x7BFF) | (W4[:, 2:4].view(np.uint16)[:, 0] == 0x7BFF)
    W4[big4, 4:16] = 0x41        # small scales and mins there
    W4 = W4.reshape(-1)
    for name, W in (("q6_K", W6), ("q6_K", W8), ("q4_K", W4)):
        _, Q, Y, _ = _run(mmq, name, W, od, id_, X)
        assert np.array_equal(Q, Q_ref)
        Y_ref = oracle.gemm(QT[name], W, od, id_, Q_ref, nt)
        assert np.isfinite(Y_ref).all()
        # the task's bound, applied per weight row (stricter than over all of Y,
        # whose maximum the fp16-maximum blocks dominate)
        err = np.abs(Y.astype(np.float64) - Y_ref).max(axis=0)
        bound = RTOL_MAX * np.abs(Y_ref).max(axis=0) + ATOL
        assert (err <= bound).all(), (name, int(np.argmax(err - bound)))


def test_many_token_tiles(mmq):
    """nt = 16384: 128 token tiles, persistent CTAs over many tiles, sampled."""
    od, id_, nt = 256, 512, 16384
    W = gen.weights("q4_K", od, id_, seed=71)
    X = gen.activations(nt, id_, seed=72)
    _, Q, Y, _ = _run(mmq, "q4_K", W, od, id_, X)
    Q_ref = oracle.quantize_q8_0(X)
    assert np.array_equal(Q, Q_ref)
    ts, os_ = _sample_entries(nt, od, 4000, 73)
    y_ref = oracle.gemm_entries(oracle.Q4_K, W, od, id_, Q_ref, nt, ts, os_)
    err, bound = _within_tol(Y[ts, os_], y_ref)
    assert err <= bound, (err, bound)


def test_bounded_wait_reports_and_context_survives(mmq):
    rc = mmq.mmq_selftest_wait_timeout(50_000_000)  # 50 ms, nothing ever arrives
    assert rc == mmq.mmq.MMQ_ERR_DEVICE_TIMEOUT
    assert mmq.mmq_last_device_error() == 0         # the status word was cleared
    # the context still works
    od, id_, nt = 128, 256, 8
    W = gen.weights("q6_K", od, id_, seed=3)
    X = gen.activations(nt, id_, seed=4)
    _, _, Y, _ = _run(mmq, "q6_K", W, od, id_, X)
    err, bound = _within_tol(Y, oracle.gemm(oracle.Q6_K, W, od, id_, oracle.quantize_q8_0(X), nt))
    assert err <= bound


@pytest.mark.parametrize("name,od,id_,nt", [("q6_K", 3584, 18944, 2630), ("q4_K", 18944, 3584, 2630)])
def test_persistent_tiles_deterministic_with_outliers(mmq, name, od, id_, nt):
    """Many tiles per persistent CTA, outlier activations: repeated runs must
    agree bit for bit (a stage buffer refilled too early shows up here first)."""
    W = gen.weights(name, od, id_, seed=7)
    X = gen.activations(nt, id_, seed=8, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda())
    Y0 = mmq.mmq_gemm(w, Q, nt).clone()
    for _ in range(3):
        assert torch.equal(mmq.mmq_gemm(w, Q, nt), Y0)
    assert mmq.mmq_last_device_error() == 0
    w.release()


def test_repeat_calls_are_deterministic(mmq):
    od, id_, nt = 256, 1024, 300
    W = gen.weights("q6_K", od, id_, seed=5)
    X = gen.activations(nt, id_, seed=6)
    w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), od, id_)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda())
    Y1 = mmq.mmq_gemm(w, Q, nt).clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Y2 = mmq.mmq_gemm(w, Q, nt, stream=s)
    s.synchronize()
    assert torch.equal(Y1, Y2)


# --------------------------------------------------------------------------
# fused quantization: fp32 activations straight into the operand plane
@pytest.mark.parametrize("name,od,id_,nt,seed", [
    ("q4_K", 260, 512, 129, 21),
    ("q6_K", 300, 768, 200, 22),
    ("q4_K", 3584, 3584, 512, 23),
    ("q6_K", 1000, 4096, 300, 24),
    ("q4_K", 130, 22016, 70, 25),   # 688 blocks per token, stashed
    ("q4_K", 64, 196864, 5, 26),    # 6152 blocks per token, past the stash: two passes over X
])
def test_gemm_f32_matches_quantize_then_gemm(mmq, name, od, id_, nt, seed):
    W = gen.weights(name, od, id_, seed=300 + seed)
    X = gen.activations(nt, id_, seed=400 + seed, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Y2 = mmq.mmq_gemm(w, mmq.mmq_quantize_act(Xd), nt)
    Y1 = mmq.mmq_gemm_f32(w, Xd)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    # the same q8_0 operands reach the same kernel: bit-identical outputs
    assert torch.equal(Y1, Y2)
    if od * id_ * nt <= 1e8:
        err, bound = _within_tol(Y1.cpu().numpy(), oracle.gemm(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt))
        assert err <= bound, (err, bound)
    w.release()


def _tie_blocks(nt, id_, seed):
    """Activation rows whose q8_0 quotients x / d sit on half-integers, one ulp
    beside them, and just inside and outside 1e-4 of them, for block scales
    from 1e-3 to 7e4 (d = 1 exactly when amax = 127); every block's first value
    is +-amax."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((nt, id_)).astype(np.float32)
    one = np.float32(1)
    for t in range(nt):
        for c in range(id_ // 32):
            kind = (t * 7 + c) % 5
            amax = np.float32(rng.choice([127.0, 1.2345, 3.0e-3, 7.7e4, 0.5]))
            d = np.float32(amax / np.float32(127))
            x = ((rng.integers(-126, 126, size=31) + 0.5).astype(np.float32) * d).astype(np.float32)
            if kind == 1:
                x = np.nextafter(x, np.float32(np.inf))
            elif kind == 2:
                x = np.nextafter(x, np.float32(-np.inf))
            elif kind == 3:
                x = (x * (one + np.float32(3e-6))).astype(np.float32)
            elif kind == 4:
                x = (x * (one - np.float32(3e-6))).astype(np.float32)
            X[t, c * 32] = amax if rng.random() < 0.5 else -amax
            X[t, c * 32 + 1:(c + 1) * 32] = x
    return X


@pytest.mark.parametrize("name", ["q4_K", "q6_K"])
def test_fused_quantization_at_rounding_ties(mmq, name):
    """The fused quantization rounds x * fl(1/d) and divides only within 1e-4 of
    a half-integer; quotients on and around the ties must still give the
    blocks of the dividing quantizer (and so the oracle's), on both arms."""
    nt, od, id_ = 40, 256, 512
    X = _tie_blocks(nt, id_, 90)
    Xd = torch.from_numpy(X).cuda()
    Q = mmq.mmq_quantize_act(Xd)
    assert np.array_equal(Q.cpu().numpy(), oracle.quantize_q8_0(X))
    W = gen.weights(name, od, id_, seed=91)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    for arm in (mmq.MMQ_ARM_F16, mmq.MMQ_ARM_SPLIT):
        Y1 = mmq.mmq_gemm_f32(w, Xd, flags=arm)
        Y2 = mmq.mmq_gemm(w, Q, nt, flags=arm)
        torch.cuda.synchronize()
        assert mmq.mmq_last_device_error() == 0
        assert torch.equal(Y1, Y2), arm
    w.release()


# --------------------------------------------------------------------------
# integer exactness: the raw per-chunk TMEM partials against the oracle's int64
def _extreme_q6k(od, id_, seed):
    """q6_K blocks at the ends of both ranges: sc in {-128, 127}, codes 0 or 63."""
    W = gen.weights("q6_K", od, id_, seed=seed).reshape(-1, 210).copy()
    rng = np.random.default_rng(seed)
    n = W.shape[0]
    W[:, 192:208] = np.where(rng.random((n, 16)) < 0.5, 127, np.uint8(np.int8(-128).view(np.uint8)))
    W[:, 0:192] = np.where(rng.random((n, 1)) < 0.5, 0x00, 0xFF).astype(np.uint8)
    return W.reshape(-1)


@pytest.mark.parametrize("case", ["q6_K one plane", "q6_K two planes", "q4_K", "q6_K extremes"])
def test_chunk_partials_are_exact_integers(mmq, case):
    """Every 32-K chunk partial the tensor core leaves in TMEM equals the
    oracle's int64 sum exactly (two-plane q6_K: the B1 and B0 UMMAs summed);
    the extreme case drives partials to 32 * 127 * 4096, just under 2^24."""
    if case == "q4_K":
        name, od, id_, nt = "q4_K", 200, 768, 130
        W = gen.weights(name, od, id_, seed=93)
    else:
        name, od, id_, nt = "q6_K", 256, 512, 40
        if case == "q6_K extremes":
            W = _extreme_q6k(od, id_, 94)
        else:
            W = gen.weights(name, od, id_, seed=95, q6_scales="int8" if "two" in case else "small")
    X = gen.activations(nt, id_, seed=96, outlier_p=0.02, outlier_scale=30.0)
    X[0:8] = 1.0                                                   # qs = 127 everywhere
    X[8:16] = np.where(np.arange(id_) % 64 < 32, 1.0, -1.0).astype(np.float32)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda())
    P = mmq.mmq_debug_chunk_partials(w, Q, nt).cpu().numpy()
    assert mmq.mmq_last_device_error() == 0
    S = oracle.chunk_partials(QT[name], W, od, id_, Q.cpu().numpy(), nt)
    assert np.abs(S).max() < 2 ** 24
    assert np.array_equal(P.astype(np.int64), S) and np.array_equal(P, S.astype(np.float32))
    if case == "q6_K extremes":
        assert np.abs(S).max() > 2 ** 23   # the boundary was reached
    w.release()


# --------------------------------------------------------------------------
# raw arm: packed weight bytes unpacked inside the GEMM
RAW_SHAPES = [
    ("q6_K", 256, 512, 16, 31),
    ("q4_K", 260, 512, 129, 32),
    ("q6_K", 300, 768, 200, 33),
    ("q4_K", 131, 256, 1, 34),
    ("q6_K", 1000, 4096, 300, 35),   # stream-K split tiles
    ("q4_K", 3584, 3584, 512, 36),   # the q-proj workload
    ("q6_K", 3584, 18944, 300, 37),  # many super-blocks, whole tiles
]


@pytest.mark.parametrize("name,od,id_,nt,seed", RAW_SHAPES)
def test_raw_arm_bit_identical_to_operand_plane(mmq, name, od, id_, nt, seed):
    # (q6_K scales within +-64: the raw arm unpacks into one operand image)
    W = gen.weights(name, od, id_, seed=500 + seed, q6_scales="small")
    X = gen.activations(nt, id_, seed=600 + seed, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_, mmq.MMQ_REG_RAW)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda())
    Y16, a16 = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_F16, return_arm=True)
    Yraw, araw = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_RAW, return_arm=True)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert (a16, araw) == (mmq.MMQ_ARM_F16, mmq.MMQ_ARM_RAW)
    # the unpacked operand images equal the registered ones: same results
    assert torch.equal(Y16, Yraw)
    if od * id_ * nt <= 1e8:
        err, bound = _within_tol(Yraw.cpu().numpy(),
                                 oracle.gemm(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt))
        assert err <= bound, (err, bound)
    w.release()


def test_raw_arm_argument_errors(mmq):
    W = gen.weights("q6_K", 128, 256, seed=7)
    w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), 128, 256)
    Q = mmq.mmq_quantize_act(torch.randn(4, 256, device="cuda"))
    with pytest.raises(mmq.MMQError) as ei:
        mmq.mmq_gemm(w, Q, 4, flags=mmq.MMQ_ARM_RAW)  # handle has no raw plane
    assert ei.value.code == -7
    with pytest.raises(mmq.MMQError) as ei:
        mmq.mmq_gemm(w, Q, 4, flags=7)  # no such arm
    assert ei.value.code == -7
    w.release()


# --------------------------------------------------------------------------
# the W_exp code plane carried to q4_K, and the dequantization fallback
@pytest.mark.parametrize("od,id_,nt", [(300, 768, 70), (131, 2048, 129)])
def test_q4k_wexp_plane_and_consumer(mmq, od, id_, nt):
    W = gen.weights("q4_K", od, id_, seed=41)
    X = gen.activations(nt, id_, seed=42)
    w, Q, Y, _ = _run(mmq, "q4_K", W, od, id_, X, mmq.MMQ_REG_WEXP)
    # producer gate: the plane's bytes; consumer gate: the GEMM built from it
    assert np.array_equal(mmq.mmq_weights_wexp(w).cpu().numpy(), oracle.expand_q4k_dense(W, od, id_))
    err, bound = _within_tol(Y, oracle.gemm(oracle.Q4_K, W, od, id_, oracle.quantize_q8_0(X), nt))
    assert err <= bound, (err, bound)
    w.release()


@pytest.mark.parametrize("name,od,id_", [("q6_K", 300, 768), ("q4_K", 131, 2048), ("q6_K", 5, 256)])
def test_dequantize_weights_bit_exact(mmq, name, od, id_):
    W = gen.weights(name, od, id_, seed=43)
    Wd = torch.from_numpy(W).cuda()
    ref = oracle.dequant_weights(QT[name], W, od, id_)
    for dt, npt in ((torch.float16, np.float16), (torch.float32, np.float32)):
        got = mmq.mmq_dequantize_weights(name, Wd, od, id_, dt).cpu().numpy()
        want = ref.astype(npt)  # one rounding, to nearest even, from the exact fp64 weight
        assert np.array_equal(got.view(np.uint16 if npt is np.float16 else np.uint32),
                              want.view(np.uint16 if npt is np.float16 else np.uint32))


# --------------------------------------------------------------------------
# split arm: the activation scale folded into A as an exact fp16 hi + lo pair
SPLIT_SHAPES = [
    ("q6_K", 256, 512, 16, 41),
    ("q4_K", 260, 512, 129, 42),
    ("q6_K", 300, 768, 200, 43),
    ("q4_K", 131, 256, 1, 44),
    ("q4_K", 384, 1024, 256, 45),
    ("q6_K", 1000, 4096, 300, 46),
    # 27 weight tiles, 14 super-blocks, ragged tokens
    ("q6_K", 3456, 3584, 300, 47),
    # 28 super-blocks per tile: the min term's region hand-off over a long tile
    ("q4_K", 896, 7168, 200, 48),
    # 688 blocks per token: the quantization kernel keeps them in shared memory
    ("q6_K", 130, 22016, 70, 49),
    # 1280 blocks per token, past the shared-memory stash: two passes over X
    ("q4_K", 64, 40960, 5, 50),
    ("q6_K", 64, 40960, 5, 51),
]


@pytest.mark.parametrize("name,od,id_,nt,seed", SPLIT_SHAPES)
def test_split_arm_parity(mmq, name, od, id_, nt, seed):
    W = gen.weights(name, od, id_, seed=500 + seed)
    X = gen.activations(nt, id_, seed=600 + seed, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Q = mmq.mmq_quantize_act(Xd)
    Ys, arm = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_SPLIT, return_arm=True)
    assert arm == mmq.MMQ_ARM_SPLIT
    Yf = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    # the same quantized operands from X or from Q: bit-identical
    assert torch.equal(Ys, Yf)
    Y_ref = oracle.gemm(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt)
    err, bound = _within_tol(Ys.cpu().numpy(), Y_ref)
    assert err <= bound, (err, bound)
    # and close to the exact-partials arm: both are within fp32 summation of Y_ref
    Y16 = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_F16)
    scale = float(np.abs(Y_ref).max()) + 1e-30
    assert float((Ys - Y16).abs().max()) / scale < 1e-5
    w.release()


@pytest.mark.parametrize("od,id_,nt", [(300, 768, 200), (1000, 4096, 300), (3584, 512, 2176)])
def test_q6k_one_plane_and_two_plane_operands(mmq, od, id_, nt):
    """q6_K with every |sc| <= 64 registers one operand plane, with the int8
    range two (B1 + B0); both arms on both against the oracle."""
    X = gen.activations(nt, id_, seed=70 + od, outlier_p=0.01, outlier_scale=20.0)
    Q_ref = oracle.quantize_q8_0(X)
    Q = mmq.mmq_quantize_act(torch.from_numpy(X).cuda())
    operand_bytes = {}
    for scales in ("small", "int8"):
        W = gen.weights("q6_K", od, id_, seed=71 + od, q6_scales=scales)
        w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), od, id_)
        operand_bytes[scales] = mmq.mmq_weights_info(w)["operand_bytes"]
        ts, os_ = _sample_entries(nt, od, 2000, od)
        y_ref = oracle.gemm_entries(oracle.Q6_K, W, od, id_, Q_ref, nt, ts, os_)
        for arm in (mmq.MMQ_ARM_F16, mmq.MMQ_ARM_SPLIT):
            Y = mmq.mmq_gemm(w, Q, nt, flags=arm).cpu().numpy()
            assert mmq.mmq_last_device_error() == 0
            err, bound = _within_tol(Y[ts, os_], y_ref)
            assert err <= bound, (scales, arm, err, bound)
        w.release()
    # the two-plane handle holds twice the operand bytes
    assert operand_bytes["int8"] == 2 * operand_bytes["small"]


@pytest.mark.parametrize("cfg", [c for c in FULL_SIZE if c.qtype == "q6_K"], ids=lambda c: c.name)
def test_two_plane_q6k_workloads_sampled(mmq, cfg):
    """The q6_K workloads' shapes with scales over the int8 range (the format's
    usual encoding): the two-plane operand on both arms, at full size, sampled
    against the oracle; the library's choice is the fp16-plane arm."""
    W = gen.weights("q6_K", cfg.od, cfg.id, cfg.seed, q6_scales="int8")
    _, X = gen.config_inputs(cfg)
    w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), cfg.od, cfg.id)
    Xd = torch.from_numpy(X).cuda()
    ts, os_ = _sample_entries(cfg.nt, cfg.od, 3000 if cfg.id <= 4096 else 800, cfg.seed)
    y_ref = oracle.gemm_entries(oracle.Q6_K, W, cfg.od, cfg.id, oracle.quantize_q8_0(X), cfg.nt, ts, os_)
    for arm in (mmq.MMQ_ARM_AUTO, mmq.MMQ_ARM_SPLIT):
        Y, used = mmq.mmq_gemm_f32(w, Xd, flags=arm, return_arm=True)
        assert mmq.mmq_last_device_error() == 0
        assert used == (mmq.MMQ_ARM_F16 if arm == mmq.MMQ_ARM_AUTO else mmq.MMQ_ARM_SPLIT)
        err, bound = _within_tol(Y.cpu().numpy()[ts, os_], y_ref)
        assert err <= bound, (arm, err, bound)
    w.release()


@pytest.mark.parametrize("cfg", FULL_SIZE, ids=lambda c: c.name)
def test_split_arm_workloads_sampled(mmq, cfg):
    W, X = gen.config_inputs(cfg)
    w = mmq.mmq_register_weights(cfg.qtype, torch.from_numpy(W).cuda(), cfg.od, cfg.id)
    Y = mmq.mmq_gemm_f32(w, torch.from_numpy(X).cuda(), flags=mmq.MMQ_ARM_SPLIT).cpu().numpy()
    assert mmq.mmq_last_device_error() == 0
    ts, os_ = _sample_entries(cfg.nt, cfg.od, 3000 if cfg.id <= 4096 else 800, cfg.seed)
    y_ref = oracle.gemm_entries(QT[cfg.qtype], W, cfg.od, cfg.id, oracle.quantize_q8_0(X), cfg.nt, ts, os_)
    err, bound = _within_tol(Y[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    w.release()


@pytest.mark.parametrize("name", ["q6_K", "q4_K"])
@pytest.mark.parametrize("od", [3584, 3456])   # 28 weight tiles, and 27 (the last pair repeats a tile)
def test_split_arm_wide_tiles(mmq, name, od):
    """Enough tiles for the split arm's 256-row tiles (for q4_K the min term then
    shares the accumulator's TMEM region); two super-blocks per tile, so a CTA
    carries the pending min term across tile boundaries."""
    id_, nt = 512, 2176
    W = gen.weights(name, od, id_, seed=81 + od)
    X = gen.activations(nt, id_, seed=82 + od, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Y = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    Y16 = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_F16)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    Yn = Y.cpu().numpy()
    ts, os_ = _sample_entries(nt, od, 4000, od)
    y_ref = oracle.gemm_entries(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt, ts, os_)
    err, bound = _within_tol(Yn[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    # every output written, and within fp32 summation of the exact-partials arm
    assert float((Y - Y16).abs().max()) <= 1e-5 * float(Y16.abs().max())
    w.release()


# --------------------------------------------------------------------------
# the FFN-down workload with the pre-expanded W_exp plane, at full size
def test_ffn_down_workload_with_wexp_plane_through_the_gemm(mmq):
    """q6_K 3584 x 18944, nt = 2630, registered with MMQ_REG_WEXP: the operand
    plane is then rebuilt from the dense W_exp plane, so this is the consumer
    gate of "47 · r44 — W_exp stride mismatch root cause" (§2.5) on the
    workload's own shape -- the plane byte-exact, and the GEMM through it on
    every arm that reads it against the oracle on sampled outputs and the
    tile edges."""
    cfg = gen.config_by_name("q6_K_ffn_down_3584x18944_nt2630")
    W, X = gen.config_inputs(cfg)
    w = mmq.mmq_register_weights("q6_K", torch.from_numpy(W).cuda(), cfg.od, cfg.id, mmq.MMQ_REG_WEXP)
    assert np.array_equal(mmq.mmq_weights_wexp(w).cpu().numpy(), oracle.expand_q6k_dense(W, cfg.od, cfg.id))
    Xd = torch.from_numpy(X).cuda()
    ts, os_ = _sample_entries(cfg.nt, cfg.od, 800, cfg.seed + 11)
    y_ref = oracle.gemm_entries(oracle.Q6_K, W, cfg.od, cfg.id, oracle.quantize_q8_0(X), cfg.nt, ts, os_)
    for arm in (mmq.MMQ_ARM_AUTO, mmq.MMQ_ARM_SPLIT, mmq.MMQ_ARM_F16):
        Y, used = mmq.mmq_gemm_f32(w, Xd, flags=arm, return_arm=True)
        torch.cuda.synchronize()
        assert mmq.mmq_last_device_error() == 0
        Yn = Y.cpu().numpy()
        assert np.isfinite(Yn).all()
        err, bound = _within_tol(Yn[ts, os_], y_ref)
        assert err <= bound, (mmq.ARM_NAMES[used], err, bound)
    w.release()


@pytest.mark.parametrize("name", ["q4_K_qproj_3584x3584_nt512", "q6_K_ffn_down_3584x18944_nt2630"])
def test_raw_arm_workloads_sampled_against_oracle(mmq, name):
    """The raw arm (packed weight bytes unpacked inside the GEMM) on the q-proj
    and FFN-down workloads at full size, against the oracle directly (sampled
    outputs and tile edges), not only against the fp16-plane arm."""
    cfg = gen.config_by_name(name)
    W, X = gen.config_inputs(cfg)
    w = mmq.mmq_register_weights(cfg.qtype, torch.from_numpy(W).cuda(), cfg.od, cfg.id, mmq.MMQ_REG_RAW)
    Y, used = mmq.mmq_gemm_f32(w, torch.from_numpy(X).cuda(), flags=mmq.MMQ_ARM_RAW, return_arm=True)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert used == mmq.MMQ_ARM_RAW
    Yn = Y.cpu().numpy()
    assert np.isfinite(Yn).all()
    ts, os_ = _sample_entries(cfg.nt, cfg.od, 3000 if cfg.id <= 4096 else 800, cfg.seed + 13)
    y_ref = oracle.gemm_entries(QT[cfg.qtype], W, cfg.od, cfg.id, oracle.quantize_q8_0(X), cfg.nt, ts, os_)
    err, bound = _within_tol(Yn[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    w.release()


# --------------------------------------------------------------------------
# few tiles (small nt): the split arm cuts each tile's super-blocks into pieces
@pytest.mark.parametrize("name", ["q4_K", "q6_K"])
@pytest.mark.parametrize("nt", [1, 16, 32, 33, 64, 100, 128, 129, 200, 256])
def test_small_nt_pieces_against_oracle(mmq, name, nt):
    """q-proj weights (3584 x 3584) at token counts whose 128-row tiles fill
    at most half the SMs: every tile's super-blocks are shared out as pieces
    over CTAs, the activation copies stop at the last token row, and the
    last piece of a tile adds all pieces in order.  Full element-by-element
    compare with the oracle, on the library's arm and the split arm; repeat
    calls bit-identical (the order of the pieces' sum is fixed)."""
    od = id_ = 3584
    W = gen.weights(name, od, id_, seed=700 + nt)
    X = gen.activations(nt, id_, seed=701 + nt, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Y_ref = oracle.gemm_mt(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt)
    for arm in (mmq.MMQ_ARM_AUTO, mmq.MMQ_ARM_SPLIT):
        Y, used = mmq.mmq_gemm_f32(w, Xd, flags=arm, return_arm=True)
        Y2 = mmq.mmq_gemm_f32(w, Xd, flags=arm)
        torch.cuda.synchronize()
        assert mmq.mmq_last_device_error() == 0
        # the library takes the pieces up to 128 tokens, the pair arm above
        assert used == (mmq.MMQ_ARM_PAIR if arm == mmq.MMQ_ARM_AUTO and nt > 128 else mmq.MMQ_ARM_SPLIT)
        assert torch.equal(Y, Y2)
        err, bound = _within_tol(Y.cpu().numpy(), Y_ref)
        assert err <= bound, (arm, err, bound)
    Y16 = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_F16)
    assert float((Y - Y16).abs().max()) <= 1e-5 * float(Y16.abs().max())
    w.release()


@pytest.mark.parametrize("name,od,id_,nt", [("q6_K", 3584, 18944, 16), ("q4_K", 1000, 2048, 50),
                                            ("q6_K", 130, 512, 7), ("q4_K", 131, 768, 5),
                                            ("q4_K", 257, 1024, 31)])
def test_small_nt_pieces_other_shapes(mmq, name, od, id_, nt):
    """Pieces on the FFN-down shape (74 super-blocks per tile), a ragged od
    (8 tiles, one super-block per piece), two- and three-tile weights with od
    not a multiple of 4 (the last piece's sum stored element by element) and
    up to 31 tokens (the trimmed activation regions); from pad40 blocks and
    from fp32 X, against the oracle."""
    W = gen.weights(name, od, id_, seed=710 + nt)
    X = gen.activations(nt, id_, seed=711 + nt, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Q = mmq.mmq_quantize_act(Xd)
    Yf = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    Yq = mmq.mmq_gemm(w, Q, nt, flags=mmq.MMQ_ARM_SPLIT)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert torch.equal(Yf, Yq)
    Y_ref = oracle.gemm_mt(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt)
    err, bound = _within_tol(Yf.cpu().numpy(), Y_ref)
    assert err <= bound, (err, bound)
    w.release()


@pytest.mark.parametrize("name,od,id_,nt", [("q6_K", 2048, 3584, 2630), ("q6_K", 3584, 3584, 2048),
                                            ("q4_K", 2048, 3584, 2630)])
def test_last_wave_in_pieces(mmq, name, od, id_, nt):
    """Several waves of 256-row q6_K tiles whose last wave would leave SMs idle
    (168 and 224 tiles on the GPU's SMs): those tiles run as pieces over every
    CTA after the whole tiles (q4_K's 256-row tiles stay whole: the same shape
    as a control).  Sampled outputs against the oracle, tile edges included;
    repeat calls bit-identical."""
    W = gen.weights(name, od, id_, seed=720 + od)
    X = gen.activations(nt, id_, seed=721 + od, outlier_p=0.01, outlier_scale=20.0)
    w = mmq.mmq_register_weights(name, torch.from_numpy(W).cuda(), od, id_)
    Xd = torch.from_numpy(X).cuda()
    Y = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    Y2 = mmq.mmq_gemm_f32(w, Xd, flags=mmq.MMQ_ARM_SPLIT)
    torch.cuda.synchronize()
    assert mmq.mmq_last_device_error() == 0
    assert torch.equal(Y, Y2)
    Yn = Y.cpu().numpy()
    assert np.isfinite(Yn).all()
    ts, os_ = _sample_entries(nt, od, 3000, od + nt)
    # the last rows of the output (the tiles of the last wave)
    ts = np.concatenate([ts, np.full(64, nt - 1), np.arange(nt - 64, nt)])
    os_ = np.concatenate([os_, np.arange(od - 64, od), np.full(64, od - 1)])
    y_ref = oracle.gemm_entries(QT[name], W, od, id_, oracle.quantize_q8_0(X), nt, ts, os_)
    err, bound = _within_tol(Yn[ts, os_], y_ref)
    assert err <= bound, (err, bound)
    w.release()
