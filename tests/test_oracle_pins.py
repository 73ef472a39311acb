"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one part of the oracle to something it cannot simply echo: a
value printed on the pages (golden fixtures, cited there), a second statement
of the same map on another page, a closed form, an invariant, a bijection, or
brute force against a library matmul.  A plausible mistake in any oracle
function (a dropped term, a wrong shift or index, a transposed operand) fails
at least one of them.
"""
import numpy as np
import pytest

import oracle
from synth import gen

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

F16_ONE = 0x3C00  # fp16 1.0


def _f16_bytes(v):
    return np.array([v], dtype=np.float16).view(np.uint8)


# --------------------------------------------------------------------------
# fp16 conversion: the oracle's vs numpy's (an independent implementation)
# --------------------------------------------------------------------------
def test_f32_to_f16_matches_numpy():
    rng = np.random.default_rng(7)
    parts = [
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8,
                  1 / 3, 1e-4, 1e-3, 2049.0, 2051.0, 4097.0], dtype=np.float32),
    ]
    x = np.concatenate(parts).astype(np.float32)
    # ties: halfway between consecutive fp16 values, both signs
    h = np.arange(0x0001, 0x7BFF, 97, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    got = oracle.f32_to_f16(x)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    back = oracle.f16_to_f64(want)
    assert np.array_equal(back, want.view(np.float16).astype(np.float64), equal_nan=True)


# --------------------------------------------------------------------------
# q8_0 pad40 quantizer
# --------------------------------------------------------------------------
def test_pad40_layout_golden(golden):
    rows = {r[0]: r[1:] for r in golden("pad40_layout.txt")}
    assert rows["pitch"] == ["40"]
    # amax = 127 gives d = 1 exactly: every value is its own code.
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, 32:64] = np.arange(-15, 17, dtype=np.float32) * 4  # block (1, 1)
    x[1, 32] = 127.0
    Q = oracle.quantize_q8_0(x)
    assert Q.shape == (2, 2, 40)
    flat = Q.reshape(-1)
    blk = flat[(1 * 2 + 1) * 40:(1 * 2 + 1) * 40 + 40]  # plane index (t*nb32 + c)*40
    d_off, d_n = map(int, rows["d"])
    qs_off, qs_n = map(int, rows["qs"])
    ss_off, ss_n = map(int, rows["ssum"])
    assert int(blk[d_off:d_off + d_n].view("<u2")[0]) == F16_ONE
    assert blk[2:4].tolist() == [0, 0]
    qs = blk[qs_off:qs_off + qs_n].view(np.int8)
    want = x[1, 32:64].astype(np.int64)
    assert qs.tolist() == want.tolist()
    assert int(blk[ss_off:ss_off + ss_n].view("<i4")[0]) == int(want.sum())
    # the three other blocks are all-zero chunks
    assert not flat[:120].any()


def test_quantize_ties_round_half_away_from_zero():
    # d = 127/127 = 1 exactly, so x = k + 0.5 is an exact tie.
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 127.0
    vals = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5, 3.5, -3.5, 0.49999997, -0.49999997]
    x[0, 1:1 + len(vals)] = vals
    qs = oracle.quantize_q8_0(x)[0, 0, 4:36].view(np.int8)
    assert qs[1:1 + len(vals)].tolist() == [3, -3, 1, -1, 2, -2, 127, -127, 4, -4, 0, 0]


def test_quantize_zero_block():
    Q = oracle.quantize_q8_0(np.zeros((3, 96), dtype=np.float32))
    assert not Q.any()
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 5] = -0.0
    assert not oracle.quantize_q8_0(x).any()


@pytest.mark.parametrize("v", [1.0, -1.0, 0.37, -123.25, 1e-3, 7e4])
def test_quantize_all_equal_block(v):
    x = np.full((1, 32), v, dtype=np.float32)
    b = oracle.quantize_q8_0(x)[0, 0]
    s = 1 if v > 0 else -1
    assert b[4:36].view(np.int8).tolist() == [127 * s] * 32
    assert int(b[36:40].view("<i4")[0]) == 4064 * s
    d_want = np.float16(np.float32(abs(v)) / np.float32(127.0))
    assert int(b[0:2].view("<u2")[0]) == int(np.array([d_want]).view(np.uint16)[0])


def test_quantize_invariants_random():
    X = gen.activations(64, 1024, seed=11, sigma=1.0, outlier_p=0.02, outlier_scale=30.0)
    X[3, :32] = 0.0
    X[5, 64:96] *= 1e-6
    Q = oracle.quantize_q8_0(X)
    qs = Q[:, :, 4:36].view(np.int8).astype(np.int64)
    ssum = Q[:, :, 36:40].copy().view("<i4")[..., 0].astype(np.int64)
    assert np.array_equal(ssum, qs.sum(-1))
    assert np.abs(qs).max() <= 127
    assert not Q[:, :, 2:4].any()
    xb = X.reshape(64, 32, 32).astype(np.float64)
    amax = np.abs(xb).max(-1)
    nz = amax > 0
    # the element that attains amax maps to +-127
    assert (np.abs(qs).max(-1)[nz] == 127).all()
    # rounding to nearest with the fp32 step amax/127: |x/d - q| <= 1/2 (+ fp32 rounding)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    r = np.abs(xb[nz] / d32[nz][:, None] - qs[nz])
    assert r.max() <= 0.5 + 1e-5
    # stored d is fp16 of that step
    d16 = Q[:, :, 0:2].copy().view("<u2")[..., 0]
    assert np.array_equal(d16[nz], d32[nz].astype(np.float32).astype(np.float16).view(np.uint16))


# --------------------------------------------------------------------------
# q6_K element map: two statements on two pages must agree
# --------------------------------------------------------------------------
def _q6k_pair_form(blocks):
    """Centered values by the byte-pair statement (page r43, §3.2): for half
    it and r < 64, ql[it*64+r] feeds elements it*128+r (low nibble) and
    it*128+r+64 (high nibble); qh[it*32 + r%32] feeds them at bit 2*(r//32)
    and 2*(r//32)+4."""
    n = blocks.shape[0]
    out = np.empty((n, 256), dtype=np.int64)
    ql = blocks[:, 0:128].astype(np.int64)
    qh = blocks[:, 128:192].astype(np.int64)
    for it in range(2):
        for r in range(64):
            a = ql[:, it * 64 + r]
            h = qh[:, it * 32 + (r % 32)]
            s = 2 * (r // 32)
            out[:, it * 128 + r] = ((a & 15) | (((h >> s) & 3) << 4)) - 32
            out[:, it * 128 + r + 64] = ((a >> 4) | (((h >> (s + 4)) & 3) << 4)) - 32
    return out


def test_q6k_two_statements_agree_random():
    blocks = gen.q6k_blocks(seed=21, nblk=512)
    got = oracle.expand_q6k_dense(blocks.reshape(-1), 512, 256).astype(np.int64)
    assert np.array_equal(got, _q6k_pair_form(blocks))


def test_q6k_two_statements_agree_every_byte_value():
    # every value 0..255 in every ql and qh position (rest zero)
    rows = []
    for pos in range(192):
        b = np.zeros((256, 210), dtype=np.uint8)
        b[:, pos] = np.arange(256, dtype=np.uint8)
        rows.append(b)
    blocks = np.concatenate(rows)
    got = oracle.expand_q6k_dense(blocks.reshape(-1), blocks.shape[0], 256).astype(np.int64)
    assert np.array_equal(got, _q6k_pair_form(blocks))


def test_q6k_element_map_golden(golden):
    for e, qlb, qlbit, qhb, qhbit in (map(int, r) for r in golden("q6k_element_map.txt")):
        # set exactly the golden bits to 1: nibble 1 -> low bit of q, field 1 -> bit 4 of q
        b = np.zeros(210, dtype=np.uint8)
        b[qlb] |= 1 << qlbit
        assert oracle.q6k_centered(b, e) == 1 - 32
        b2 = np.zeros(210, dtype=np.uint8)
        b2[128 + qhb] |= 1 << qhbit
        assert oracle.q6k_centered(b2, e) == 16 - 32
        # and no other element picks those bits up as its own
        others = [oracle.q6k_centered(b, k) for k in range(256) if k != e]
        assert all(v == -32 for v in others)


def test_q6k_nibbles_and_fields_are_a_bijection():
    hit_ql, hit_qh = {}, {}
    for pos in range(128):
        for sh in (0, 4):
            b = np.zeros((1, 210), dtype=np.uint8)
            b[0, pos] = 0xF << sh
            v = oracle.expand_q6k_dense(b.reshape(-1), 1, 256)[0].astype(int)
            idx = np.nonzero(v != -32)[0]
            assert len(idx) == 1 and v[idx[0]] == 15 - 32
            hit_ql[(pos, sh)] = int(idx[0])
    for pos in range(64):
        for sh in (0, 2, 4, 6):
            b = np.zeros((1, 210), dtype=np.uint8)
            b[0, 128 + pos] = 3 << sh
            v = oracle.expand_q6k_dense(b.reshape(-1), 1, 256)[0].astype(int)
            idx = np.nonzero(v != -32)[0]
            assert len(idx) == 1 and v[idx[0]] == 48 - 32
            hit_qh[(pos, sh)] = int(idx[0])
    assert sorted(hit_ql.values()) == list(range(256))
    assert sorted(hit_qh.values()) == list(range(256))


def test_q6k_layout_scales_and_d(golden):
    rows = {r[0]: r[1:] for r in golden("q6k_block_layout.txt")}
    assert int(rows["content"][0]) == 210
    sc_off = int(rows["sc"][0])
    d_off = int(rows["d"][0])
    sub = int(rows["sub_block_elems"][0])
    b = np.zeros(210, dtype=np.uint8)  # ql = qh = 0  ->  q - 32 = -32 everywhere
    scales = np.array([3, -7, 11, -2, 31, -32, 1, 0, 5, -5, 17, -19, 23, 29, -31, 13], dtype=np.int8)
    b[sc_off:sc_off + 16] = scales.view(np.uint8)
    b[d_off:d_off + 2] = _f16_bytes(0.5)
    for e in range(256):
        assert oracle.weight(oracle.Q6_K, b, e) == 0.5 * float(scales[e // sub]) * -32.0


# --------------------------------------------------------------------------
# q4_K (reading of the ggml layout; pinned by round trip, bijection, closed forms)
# --------------------------------------------------------------------------
def _pack_q4k_scales(sc, m):
    """Independent packer: 8 (scale, min) 6-bit pairs -> 12 bytes.  Pairs 0..3
    sit whole in the low 6 bits of bytes j (scale) and j+4 (min); pairs 4..7
    put their low nibbles in byte j+4 (scale low, min high) and their top two
    bits in bits 6..7 of bytes j-4 (scale) and j (min)."""
    s = [0] * 12
    for j in range(8):
        if j < 4:
            s[j] |= sc[j] & 63
            s[j + 4] |= m[j] & 63
        else:
            s[j + 4] |= (sc[j] & 15) | ((m[j] & 15) << 4)
            s[j - 4] |= (sc[j] >> 4) << 6
            s[j] |= (m[j] >> 4) << 6
    return np.array(s, dtype=np.uint8)


def test_q4k_scale_min_round_trip_exhaustive():
    rng = np.random.default_rng(3)
    vals = np.arange(64)
    for j in range(8):
        for a in vals:
            # each (sc, m) value pair at position j, other positions random
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            for bval in (a, 63 - a):
                sc[j], m[j] = a, bval
                blk = np.zeros(144, dtype=np.uint8)
                blk[4:16] = _pack_q4k_scales(sc, m)
                for jj in range(8):
                    assert oracle.q4k_scale_min(blk, jj) == (int(sc[jj]), int(m[jj]))


def test_q4k_nibble_bijection_and_sub_blocks():
    hit = {}
    for pos in range(128):
        for sh in (0, 4):
            b = np.zeros(144, dtype=np.uint8)
            b[16 + pos] = 0x5 << sh
            v = [oracle.q4k_quant(b, e) for e in range(256)]
            idx = [e for e in range(256) if v[e] != 0]
            assert len(idx) == 1 and v[idx[0]] == 5
            hit[(pos, sh)] = idx[0]
    assert sorted(hit.values()) == list(range(256))
    # sub-block of element e is e // 32: distinct scales make it visible
    sc = np.array([1, 2, 3, 4, 5, 6, 7, 8])
    m = np.zeros(8, dtype=int)
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = _f16_bytes(1.0)
    b[4:16] = _pack_q4k_scales(sc, m)
    b[16:144] = 0x11  # every nibble = 1
    for e in range(256):
        assert oracle.weight(oracle.Q4_K, b, e) == float(sc[e // 32])


def test_q4k_nibble_order_reading(golden):
    for e, byte, sh in (map(int, r) for r in golden("q4k_layout_reading.txt")):
        b = np.zeros(144, dtype=np.uint8)
        b[16 + byte] = 0x9 << sh
        assert oracle.q4k_quant(b, e) == 9
        assert oracle.q4k_quant(b, e ^ 32) == 0  # the partner sub-block sees the other nibble
    b = np.zeros(144, dtype=np.uint8)
    b[16:144] = 0x21  # low nibble 1, high nibble 2
    assert [oracle.q4k_quant(b, e) for e in range(0, 256, 32)] == [1, 2] * 4


def test_q4k_closed_forms():
    rng = np.random.default_rng(5)
    sc = rng.integers(0, 64, 8)
    m = rng.integers(0, 64, 8)
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = _f16_bytes(0.25)
    b[2:4] = _f16_bytes(0.125)
    b[4:16] = _pack_q4k_scales(sc, m)
    # qs = 0 -> w = -dmin * m_j
    for e in range(256):
        assert oracle.weight(oracle.Q4_K, b, e) == -0.125 * m[e // 32]
    # all nibbles 15 -> w = d*sc*15 - dmin*m
    b[16:144] = 0xFF
    for e in range(256):
        assert oracle.weight(oracle.Q4_K, b, e) == 0.25 * sc[e // 32] * 15 - 0.125 * m[e // 32]


# --------------------------------------------------------------------------
# W_exp plane and the stride-bug worked example
# --------------------------------------------------------------------------
def test_wexp_plane_layout_matches_dequant():
    od, id_ = 5, 768
    W = gen.weights("q6_K", od, id_, seed=31)
    Wexp = oracle.expand_q6k_dense(W, od, id_)
    deq = oracle.dequant_weights(oracle.Q6_K, W, od, id_)
    blk = W.reshape(od, id_ // 256, 210)
    for o in range(od):
        for sb in range(id_ // 256):
            d = float(blk[o, sb, 208:210].view(np.float16)[0])
            sc = blk[o, sb, 192:208].view(np.int8).astype(np.float64)
            for e in range(0, 256, 7):
                # element (o, sb, e) sits at o*id + sb*256 + e
                assert deq[o, sb * 256 + e] == d * sc[e // 16] * float(Wexp.reshape(-1)[o * id_ + sb * 256 + e])


def test_wexp_stride_worked_example(golden):
    rows = golden("wexp_stride_example.txt")
    ex = [r for r in rows if len(r) == 9]
    drift = [r for r in rows if len(r) == 4]
    od, id_ = 4, 256
    W = gen.weights("q6_K", od, id_, seed=41)
    dense = oracle.expand_q6k_dense(W, od, id_).reshape(-1)
    nsb, padded = id_ // 256, 224
    for r in ex:
        idv, j, start, ra, a0, a1, rb, b0, b1 = map(int, r)
        assert idv == id_
        wrong = j * (nsb * padded)  # padded row pitch applied to the dense plane
        assert wrong == start
        window = dense[wrong:wrong + id_]
        want = np.concatenate([dense[ra * id_ + a0:ra * id_ + a1], dense[rb * id_ + b0:rb * id_ + b1]])
        assert np.array_equal(window, want)
    for r in drift:
        idv, nsb_, pitch, dr = map(int, r)
        assert idv // 256 == nsb_ and nsb_ * padded == pitch and idv - pitch == dr


def test_misstrided_consumer_fails_except_row_zero():
    """Content right, offsets wrong: a consumer reading the dense plane with
    the padded pitch reproduces 'row 0 correct, every other row wrong'."""
    od, id_, nt = 6, 256, 3
    W = gen.weights("q6_K", od, id_, seed=43)
    Q = oracle.quantize_q8_0(gen.activations(nt, id_, seed=44))
    dense = oracle.expand_q6k_dense(W, od, id_).astype(np.float64)
    blk = W.reshape(od, 1, 210)
    d = blk[:, 0, 208:210].copy().view(np.float16)[:, 0].astype(np.float64)
    sc = blk[:, 0, 192:208].copy().view(np.int8).astype(np.float64)
    xh = oracle.dequant_act(Q, nt, id_)
    flat = dense.reshape(-1)

    def consume(pitch):
        Wd = np.stack([flat[o * pitch:o * pitch + id_] for o in range(od)])
        return xh @ (Wd * d[:, None] * np.repeat(sc, 16, axis=1)).T

    Y_ref = oracle.gemm(oracle.Q6_K, W, od, id_, Q, nt)
    good, bad = consume(id_), consume(224)
    assert np.allclose(good, Y_ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(bad[:, 0], Y_ref[:, 0], rtol=1e-12, atol=1e-15)
    for o in range(1, od):
        assert not np.allclose(bad[:, o], Y_ref[:, o], rtol=1e-3)


# --------------------------------------------------------------------------
# GEMM: closed forms, two formulations, brute force
# --------------------------------------------------------------------------
def test_mac_count_golden(golden):
    kv = {r[0]: int(r[1]) for r in golden("mac_count.txt")}
    cfg = gen.config_by_name("q4_K_qproj_3584x3584_nt512")
    assert (cfg.nt, cfg.od, cfg.id) == (kv["nt"], kv["od"], kv["id"])
    assert cfg.ops == 2 * kv["imma_count"] * kv["macs_per_imma"]


@pytest.mark.parametrize("qtype,name", [(oracle.Q6_K, "q6_K"), (oracle.Q4_K, "q4_K")])
def test_gemm_zero_activations(qtype, name):
    od, id_, nt = 3, 512, 2
    W = gen.weights(name, od, id_, seed=51)
    Q = oracle.quantize_q8_0(np.zeros((nt, id_), dtype=np.float32))
    assert not oracle.gemm(qtype, W, od, id_, Q, nt).any()


@pytest.mark.parametrize("qtype,name", [(oracle.Q6_K, "q6_K"), (oracle.Q4_K, "q4_K")])
def test_gemm_all_equal_activations(qtype, name):
    od, id_ = 4, 512
    vs = np.array([0.7, -2.25, 1e-2], dtype=np.float32)
    X = np.repeat(vs[:, None], id_, axis=1)
    W = gen.weights(name, od, id_, seed=52)
    Q = oracle.quantize_q8_0(X)
    Y = oracle.gemm(qtype, W, od, id_, Q, len(vs))
    rowsum = oracle.dequant_weights(qtype, W, od, id_).sum(1)
    for t, v in enumerate(vs):
        d16 = float(np.float16(np.float32(abs(v)) / np.float32(127.0)))
        want = d16 * 127.0 * np.sign(v) * rowsum
        np.testing.assert_allclose(Y[t], want, rtol=1e-12)


def test_gemm_q6k_zero_codes_closed_form():
    od, id_, nt = 3, 512, 4
    W = gen.weights("q6_K", od, id_, seed=53).reshape(od, 2, 210)
    W[:, :, 0:192] = 0  # ql = qh = 0 -> w = -32 * d * sc
    Q = oracle.quantize_q8_0(gen.activations(nt, id_, seed=54))
    Y = oracle.gemm(oracle.Q6_K, W.reshape(-1), od, id_, Q, nt)
    xh = oracle.dequant_act(Q, nt, id_)
    for t in range(nt):
        for o in range(od):
            acc = 0.0
            for sb in range(2):
                d = float(W[o, sb, 208:210].view(np.float16)[0])
                sc = W[o, sb, 192:208].view(np.int8)
                for j in range(16):
                    k0 = sb * 256 + 16 * j
                    acc += d * float(sc[j]) * -32.0 * xh[t, k0:k0 + 16].sum()
            assert Y[t, o] == pytest.approx(acc, rel=1e-12, abs=1e-300)


def test_gemm_q4k_zero_codes_min_term_closed_form():
    """qs = 0 leaves only the min term: y = -sum_c dmin * m_c * da_c * ssum_c."""
    od, id_, nt = 2, 512, 3
    rng = np.random.default_rng(9)
    blocks = np.zeros((od, 2, 144), dtype=np.uint8)
    mins = rng.integers(0, 64, (od, 2, 8))
    for o in range(od):
        for sb in range(2):
            blocks[o, sb, 0:2] = _f16_bytes(0.5)
            blocks[o, sb, 2:4] = _f16_bytes([0.001, 0.003][sb])
            blocks[o, sb, 4:16] = _pack_q4k_scales(rng.integers(0, 64, 8), mins[o, sb])
    Q = oracle.quantize_q8_0(gen.activations(nt, id_, seed=55))
    Y = oracle.gemm(oracle.Q4_K, blocks.reshape(-1), od, id_, Q, nt)
    Qb = Q.reshape(nt, id_ // 32, 40)
    for t in range(nt):
        for o in range(od):
            acc = 0.0
            for c in range(id_ // 32):
                sb, j = divmod(c, 8)
                dmin = float(blocks[o, sb, 2:4].view(np.float16)[0])
                da = float(Qb[t, c, 0:2].view(np.float16)[0])
                ssum = int(Qb[t, c, 36:40].view("<i4")[0])
                acc -= dmin * mins[o, sb, j] * da * ssum
            assert Y[t, o] == pytest.approx(acc, rel=1e-12)


@pytest.mark.parametrize("name,qtype", [("q6_K", oracle.Q6_K), ("q4_K", oracle.Q4_K)])
@pytest.mark.parametrize("od,id_,nt", [(1, 256, 1), (2, 512, 3), (3, 256, 129), (5, 768, 7)])
def test_gemm_brute_force_and_two_formulations(name, qtype, od, id_, nt):
    W = gen.weights(name, od, id_, seed=60 + od)
    X = gen.activations(nt, id_, seed=70 + nt, outlier_p=0.05, outlier_scale=10.0)
    Q = oracle.quantize_q8_0(X)
    Y = oracle.gemm(qtype, W, od, id_, Q, nt)
    # brute force: library matmul of the dequantized operands (X_hat . W^T)
    Yb = oracle.dequant_act(Q, nt, id_) @ oracle.dequant_weights(qtype, W, od, id_).T
    np.testing.assert_allclose(Y, Yb, rtol=1e-11, atol=1e-14)
    ts, os_ = np.meshgrid(np.arange(nt), np.arange(od), indexing="ij")
    ya = oracle.gemm_entries(qtype, W, od, id_, Q, nt, ts.ravel(), os_.ravel())
    yb = oracle.gemm_entries_int(qtype, W, od, id_, Q, nt, ts.ravel(), os_.ravel())
    np.testing.assert_allclose(ya, Y.ravel(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(yb, Y.ravel(), rtol=1e-10, atol=1e-12)


def test_gemm_is_not_transposed():
    """Asymmetric shapes and a one-hot token: row t of Y depends on token t only."""
    od, id_, nt = 7, 256, 5
    W = gen.weights("q4_K", od, id_, seed=80)
    X = np.zeros((nt, id_), dtype=np.float32)
    X[2] = gen.activations(1, id_, seed=81)[0]
    Q = oracle.quantize_q8_0(X)
    Y = oracle.gemm(oracle.Q4_K, W, od, id_, Q, nt)
    assert not Y[[0, 1, 3, 4]].any()
    deq = oracle.dequant_weights(oracle.Q4_K, W, od, id_)
    np.testing.assert_allclose(Y[2], deq @ oracle.dequant_act(Q, nt, id_)[2], rtol=1e-12)


def test_q4k_dense_plane_codes():
    """The dense q4_K code plane against the per-element code reading, and
    a hand-built block: qs byte i = i, so element e reads byte
    32*(e//64) + e%32 and takes its low nibble when (e//32) is even."""
    W = gen.weights("q4_K", 3, 512, seed=9)
    P = oracle.expand_q4k_dense(W, 3, 512)
    B = W.reshape(3, 2, 144)
    for j in range(3):
        for sb in range(2):
            assert [int(P[j, sb * 256 + e]) for e in range(256)] == \
                [oracle.q4k_quant(B[j, sb], e) for e in range(256)]
    blk = np.zeros(144, dtype=np.uint8)
    blk[16:144] = np.arange(128, dtype=np.uint8)
    P1 = oracle.expand_q4k_dense(blk, 1, 256)[0]
    # e=0: byte 0 low = 0; e=33: byte 1 high = 0; e=65: byte 33 low = 1;
    # e=100: byte 36 high (36 = 0x24) = 2; e=255: byte 127 high (0x7f) = 7
    assert (P1[0], P1[33], P1[65], P1[100], P1[255]) == (0, 0, 1, 2, 7)


# --------------------------------------------------------------------------
# exact chunk partials (the integer sums a GPU dump is compared with)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,qtype,scales", [("q6_K", oracle.Q6_K, "small"), ("q6_K", oracle.Q6_K, "int8"),
                                                ("q4_K", oracle.Q4_K, "small")])
def test_chunk_partials_brute_force_and_recombination(name, qtype, scales):
    """S[t][c][o] against a numpy int64 contraction of the dense code plane
    (pinned above) with the sub-block scales read from the block bytes, and
    recombined with d, da (and the q4_K min term) into the fp64 GEMM."""
    od, id_, nt = 5, 512, 7
    W = gen.weights(name, od, id_, seed=81, q6_scales=scales)
    X = gen.activations(nt, id_, seed=82, outlier_p=0.05, outlier_scale=30.0)
    Q = oracle.quantize_q8_0(X)
    S = oracle.chunk_partials(qtype, W, od, id_, Q, nt)
    nsb, nb32 = id_ // 256, id_ // 32
    qs = Q.reshape(nt, nb32, 40)[:, :, 4:36].view(np.int8).astype(np.int64).reshape(nt, id_)
    bb = 210 if name == "q6_K" else 144
    blocks = W.reshape(od, nsb, bb)
    if name == "q6_K":
        codes = oracle.expand_q6k_dense(W, od, id_).astype(np.int64)
        sc = blocks[:, :, 192:208].view(np.int8).astype(np.int64)          # (od, nsb, 16)
        scale_k = np.repeat(sc.reshape(od, nsb * 16), 16, axis=1)         # per element
    else:
        codes = oracle.expand_q4k_dense(W, od, id_).astype(np.int64)
        sc = np.array([[oracle.q4k_scale_min(blocks[o, s], j)[0] for s in range(nsb) for j in range(8)]
                       for o in range(od)], dtype=np.int64)                 # (od, nsb*8)
        scale_k = np.repeat(sc, 32, axis=1)
    B = codes * scale_k                                                     # (od, id)
    want = np.einsum("tck,ock->tco", qs.reshape(nt, nb32, 32), B.reshape(od, nb32, 32))
    assert np.array_equal(S, want)
    # recombined with the float scales: the GEMM
    da = oracle.f16_to_f64(Q.reshape(nt, nb32, 40)[:, :, 0:2].copy().view(np.uint16).reshape(nt, nb32))
    if name == "q6_K":
        d = oracle.f16_to_f64(blocks[:, :, 208:210].copy().view(np.uint16).reshape(od, nsb))
        Y = np.einsum("tco,tc,oc->to", S.astype(np.float64), da, np.repeat(d, 8, axis=1))
    else:
        d = oracle.f16_to_f64(blocks[:, :, 0:2].copy().view(np.uint16).reshape(od, nsb))
        dmin = oracle.f16_to_f64(blocks[:, :, 2:4].copy().view(np.uint16).reshape(od, nsb))
        m = np.array([[oracle.q4k_scale_min(blocks[o, s], j)[1] for s in range(nsb) for j in range(8)]
                      for o in range(od)], dtype=np.float64)
        ssum = Q.reshape(nt, nb32, 40)[:, :, 36:40].copy().view(np.int32).reshape(nt, nb32).astype(np.float64)
        Y = (np.einsum("tco,tc,oc->to", S.astype(np.float64), da, np.repeat(d, 8, axis=1))
             - np.einsum("tc,tc,oc,oc->to", da, ssum, np.repeat(dmin, 8, axis=1), m))
    Y_ref = oracle.gemm(qtype, W, od, id_, Q, nt)
    assert np.allclose(Y, Y_ref, rtol=1e-12, atol=1e-12 * np.abs(Y_ref).max())


def test_threaded_gemm_is_the_same_gemm():
    """The CPU baseline's threaded oracle GEMM shares the weight rows out over
    threads; every output must be the single-threaded value bit for bit, for
    thread counts that do and do not divide od (and more threads than rows)."""
    for qtype, qt, od, id_, nt in (("q4_K", oracle.Q4_K, 37, 512, 9), ("q6_K", oracle.Q6_K, 5, 256, 3)):
        W = gen.weights(qtype, od, id_, 21)
        Q = oracle.quantize_q8_0(gen.activations(nt, id_, 22, outlier_p=0.05, outlier_scale=20.0))
        ref = oracle.gemm(qt, W, od, id_, Q, nt)
        for threads in (1, 2, 3, 8, 64):
            assert np.array_equal(oracle.gemm_mt(qt, W, od, id_, Q, nt, threads), ref), (qtype, threads)
