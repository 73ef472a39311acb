/*
 * mmq_oracle.c -- plain, slow CPU oracle for the k-quant x q8_0 prefill
 * "MMQ" GEMM  Y[t][o] = sum_k W[o][k] * X[t][k].
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
 * bench's CPU-baseline / reference leg may load or call this library.  It
 * shares no code, header, table or constant with the CUDA path: every
 * layout constant below is restated here on purpose.
 *
 * Sources (the "minfer CUDA optimisation steps" log pages):
 *   [P-r21] "26 · r21 — Coalesced block-linear A staging", §2.1: the q8_0
 *           activation block, d (2 B) | qs (32 B at +4) | ssum (4 B at +36),
 *           block pitch 40 B, one block per token per 32-element chunk.
 *   [P-r20] "25 · r20: Split-phase A staging", §2.3: the same 40-B block
 *           read by the GEMM, plane index (t*nb32 + c)*40.
 *   [P-r44] "47 · r44 — W_exp stride mismatch root cause", §2.2: block_q6_K
 *           = ql[128] + qh[64] + sc[16] + d[2] = 210 B, 16 sub-blocks of 16
 *           elements; §3.2 (the in-kernel element expander): element e reads
 *           its low nibble from ql and its 2 high bits from qh, minus 32.
 *   [P-r43] "46 · r43 — PC-sampling attribution", §3.1: the sub-block scale
 *           byte of a block sits at offset 192 (the int8 sc array); §3.2: the
 *           dense centered-int8 W_exp plane, out[j*id + sb*256 + e] = q - 32,
 *           row pitch id, super-block pitch 256, id % 256 == 0.
 *   q4_K:   not printed on the pages.  Reading taken (the plainest one the
 *           task statement supports): the ggml block_q4_K layout, fp16 d at
 *           0, fp16 dmin at 2, 12 bytes of packed 6-bit (scale, min) pairs at
 *           4, qs[128] at 16 (144 B); 8 sub-blocks of 32; w = d*sc*q - dmin*m.
 *
 * Quantizer readings (the pages do not print the quantizer; the task's
 * workload text fixes d = amax/127 and round-half-away-from-zero):
 *   d   = amax / 127.0f in fp32 (IEEE round-to-nearest division),
 *   q_i = roundf(x_i / d) in fp32 (division, not multiplication by 1/d),
 *   d16 = fp16 round-to-nearest-even of the fp32 d (stored; used to
 *         dequantize), bytes [2,4) = 0, ssum = sum of q_i as int32,
 *   amax == 0 gives an all-zero block.
 *
 * Floating point: build with -ffp-contract=off (no fused multiply-add) and
 * without -ffast-math.  Sums are accumulated in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- type codes (ggml numbering) ------------------------------------- */
#define OR_Q4_K 12
#define OR_Q6_K 14

/* ---- q8_0 pad40 block [P-r21 §2.1] ------------------------------------ */
#define OR_Q8_PITCH 40
#define OR_Q8_QS 4
#define OR_Q8_SSUM 36

/* ---- q6_K block [P-r44 §2.2, P-r43 §3.1] ------------------------------ */
#define OR_Q6_BYTES 210
#define OR_Q6_QL 0
#define OR_Q6_QH 128
#define OR_Q6_SC 192
#define OR_Q6_D 208

/* ---- q4_K block (reading, see header) --------------------------------- */
#define OR_Q4_BYTES 144
#define OR_Q4_D 0
#define OR_Q4_DMIN 2
#define OR_Q4_SC 4
#define OR_Q4_QS 16

static int block_bytes(int type) {
    if (type == OR_Q6_K) return OR_Q6_BYTES;
    if (type == OR_Q4_K) return OR_Q4_BYTES;
    return -1;
}

/* ---- fp16 helpers (the compiler's IEEE binary16 type) ------------------ */
static uint16_t f32_to_f16_bits(float f) {
    _Float16 h = (_Float16)f;            /* IEEE round-to-nearest-even */
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static double f16_bits_to_f64(uint16_t b) {
    _Float16 h;
    memcpy(&h, &b, 2);
    return (double)h;                    /* exact */
}

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static int32_t rd_i32(const uint8_t *p) {
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                 ((uint32_t)p[3] << 24);
    return (int32_t)u;
}

void mmq_oracle_f32_to_f16(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16_bits(in[i]);
}

void mmq_oracle_f16_to_f64(const uint16_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f16_bits_to_f64(in[i]);
}

/* ====================================================================== */
/* q8_0 activation quantization                                            */
/* ====================================================================== */

/* One 32-element chunk x[0..31] -> one 40-byte block.  Returns 0, or -1 if
 * a value is not finite (out of contract). */
static int quantize_chunk(const float *x, uint8_t *blk) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
        if (!isfinite(x[i])) return -1;
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    memset(blk, 0, OR_Q8_PITCH);
    if (amax == 0.0f) return 0;          /* all-zero block: d16 = +0, qs = 0, ssum = 0 */
    float d = amax / 127.0f;
    int32_t ssum = 0;
    for (int i = 0; i < 32; ++i) {
        float v = x[i] / d;
        int q = (int)roundf(v);          /* half away from zero */
        if (q > 127) q = 127;
        if (q < -127) q = -127;
        blk[OR_Q8_QS + i] = (uint8_t)(int8_t)q;
        ssum += q;
    }
    uint16_t h = f32_to_f16_bits(d);
    blk[0] = (uint8_t)(h & 0xFF);
    blk[1] = (uint8_t)(h >> 8);
    uint32_t u = (uint32_t)ssum;
    blk[OR_Q8_SSUM + 0] = (uint8_t)(u);
    blk[OR_Q8_SSUM + 1] = (uint8_t)(u >> 8);
    blk[OR_Q8_SSUM + 2] = (uint8_t)(u >> 16);
    blk[OR_Q8_SSUM + 3] = (uint8_t)(u >> 24);
    return 0;
}

/* X: nt x id fp32 row-major.  Q: nt x (id/32) blocks of 40 B, block (t, c)
 * at byte (t*nb32 + c)*40 [P-r20 §2.3].  Returns 0, -1 on bad shape, -2 on a
 * non-finite input. */
int mmq_oracle_quantize_q8_0(const float *X, int64_t nt, int64_t id, uint8_t *Q) {
    if (nt < 0 || id <= 0 || id % 32 != 0) return -1;
    int64_t nb32 = id / 32;
    for (int64_t t = 0; t < nt; ++t)
        for (int64_t c = 0; c < nb32; ++c)
            if (quantize_chunk(X + t * id + c * 32, Q + (t * nb32 + c) * OR_Q8_PITCH))
                return -2;
    return 0;
}

/* x_hat[t][k] = d16(t, k/32) * qs[t][k] in fp64. */
void mmq_oracle_dequant_act(const uint8_t *Q, int64_t nt, int64_t id, double *Xh) {
    int64_t nb32 = id / 32;
    for (int64_t t = 0; t < nt; ++t)
        for (int64_t c = 0; c < nb32; ++c) {
            const uint8_t *b = Q + (t * nb32 + c) * OR_Q8_PITCH;
            double d = f16_bits_to_f64(rd_u16(b));
            for (int i = 0; i < 32; ++i)
                Xh[t * id + c * 32 + i] = d * (double)(int8_t)b[OR_Q8_QS + i];
        }
}

/* ====================================================================== */
/* q6_K                                                                     */
/* ====================================================================== */

/* Centered 6-bit value (q - 32) of element e in [0,256) of one block.
 * [P-r44 §3.2]: the block splits into two 128-element halves; inside a half,
 * element r takes the nibble of ql[half*64 + r%64] selected by r/64 (low,
 * then high), and the 2-bit field of qh[half*32 + r%32] selected by r/32. */
int mmq_oracle_q6k_centered(const uint8_t *blk, int e) {
    int half = e / 128;
    int r = e % 128;
    int ql = blk[OR_Q6_QL + half * 64 + r % 64];
    int qh = blk[OR_Q6_QH + half * 32 + r % 32];
    int lo4 = (ql >> (4 * (r / 64))) & 0xF;
    int hi2 = (qh >> (2 * (r / 32))) & 0x3;
    return (lo4 | (hi2 << 4)) - 32;
}

/* int8 scale of the 16-element sub-block holding element e [P-r44 §2.2]. */
static int q6k_scale(const uint8_t *blk, int e) { return (int8_t)blk[OR_Q6_SC + e / 16]; }

static double q6k_weight(const uint8_t *blk, int e) {
    double d = f16_bits_to_f64(rd_u16(blk + OR_Q6_D));
    return d * (double)q6k_scale(blk, e) * (double)mmq_oracle_q6k_centered(blk, e);
}

/* Dense centered-int8 plane [P-r43 §3.2]: out[j*id + sb*256 + e] = q - 32.
 * Input: packed rows of nsb = id/256 blocks of 210 B (row pitch nsb*210). */
int mmq_oracle_expand_q6k_dense(const uint8_t *W, int64_t od, int64_t id, int8_t *out) {
    if (od < 0 || id <= 0 || id % 256 != 0) return -1;
    int64_t nsb = id / 256;
    for (int64_t j = 0; j < od; ++j)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = W + (j * nsb + sb) * OR_Q6_BYTES;
            for (int e = 0; e < 256; ++e)
                out[j * id + sb * 256 + e] = (int8_t)mmq_oracle_q6k_centered(blk, e);
        }
    return 0;
}

/* ====================================================================== */
/* q4_K (reading: ggml block_q4_K)                                          */
/* ====================================================================== */

/* 6-bit (scale, min) of sub-block j in [0,8).  Sub-blocks 0..3 keep both in
 * the low 6 bits of bytes j and j+4; sub-blocks 4..7 keep their low 4 bits
 * in the nibbles of byte j+4 and their top 2 bits in the top bits of bytes
 * j-4 (scale) and j (min). */
void mmq_oracle_q4k_scale_min(const uint8_t *blk, int j, int *sc, int *m) {
    const uint8_t *s = blk + OR_Q4_SC;
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 0xF) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* 4-bit value of element e: sub-block j = e/32; the pair of sub-blocks
 * (2i, 2i+1) shares qs[32i .. 32i+31], low nibbles for 2i, high for 2i+1. */
int mmq_oracle_q4k_quant(const uint8_t *blk, int e) {
    int j = e / 32;
    int b = blk[OR_Q4_QS + 32 * (j / 2) + e % 32];
    return (j % 2 == 0) ? (b & 0xF) : (b >> 4);
}

/* Dense q4_K code plane (the W_exp idea carried to q4_K): element (j, k) of
 * the od x id plane is the 4-bit code q of weight (j, k), row pitch id,
 * super-block pitch 256, as for the q6_K plane. */
int mmq_oracle_expand_q4k_dense(const uint8_t *W, int64_t od, int64_t id, int8_t *out) {
    if (od < 0 || id <= 0 || id % 256 != 0) return -1;
    int64_t nsb = id / 256;
    for (int64_t j = 0; j < od; ++j)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = W + (j * nsb + sb) * OR_Q4_BYTES;
            for (int e = 0; e < 256; ++e)
                out[j * id + sb * 256 + e] = (int8_t)mmq_oracle_q4k_quant(blk, e);
        }
    return 0;
}

static double q4k_weight(const uint8_t *blk, int e) {
    int sc, m;
    mmq_oracle_q4k_scale_min(blk, e / 32, &sc, &m);
    double d = f16_bits_to_f64(rd_u16(blk + OR_Q4_D));
    double dmin = f16_bits_to_f64(rd_u16(blk + OR_Q4_DMIN));
    return d * (double)sc * (double)mmq_oracle_q4k_quant(blk, e) - dmin * (double)m;
}

/* ====================================================================== */
/* weights, both types                                                      */
/* ====================================================================== */

double mmq_oracle_weight(int type, const uint8_t *blk, int e) {
    return type == OR_Q6_K ? q6k_weight(blk, e) : q4k_weight(blk, e);
}

/* Rows o0..o1-1 of the dequantized weight matrix, fp64, row pitch id. */
int mmq_oracle_dequant_weights(int type, const uint8_t *W, int64_t od, int64_t id, int64_t o0,
                               int64_t o1, double *out) {
    int bb = block_bytes(type);
    if (bb < 0 || id <= 0 || id % 256 != 0 || o0 < 0 || o1 > od || o0 > o1) return -1;
    int64_t nsb = id / 256;
    for (int64_t o = o0; o < o1; ++o)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = W + (o * nsb + sb) * bb;
            for (int e = 0; e < 256; ++e)
                out[(o - o0) * id + sb * 256 + e] = mmq_oracle_weight(type, blk, e);
        }
    return 0;
}

/* ====================================================================== */
/* GEMM                                                                     */
/* ====================================================================== */

/* Formulation A: y = sum_k w[o][k] * x_hat[t][k], fp64, for the listed
 * (t, o) pairs. */
int mmq_oracle_gemm_entries(int type, const uint8_t *W, int64_t od, int64_t id, const uint8_t *Q,
                            int64_t nt, const int64_t *ts, const int64_t *os, int64_t n,
                            double *y) {
    int bb = block_bytes(type);
    if (bb < 0 || id <= 0 || id % 256 != 0) return -1;
    int64_t nsb = id / 256, nb32 = id / 32;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = ts[i], o = os[i];
        if (t < 0 || t >= nt || o < 0 || o >= od) return -1;
        double acc = 0.0;
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = W + (o * nsb + sb) * bb;
            for (int e = 0; e < 256; ++e) {
                int64_t k = sb * 256 + e;
                const uint8_t *qb = Q + (t * nb32 + k / 32) * OR_Q8_PITCH;
                double xh = f16_bits_to_f64(rd_u16(qb)) * (double)(int8_t)qb[OR_Q8_QS + k % 32];
                acc += mmq_oracle_weight(type, blk, e) * xh;
            }
        }
        y[i] = acc;
    }
    return 0;
}

/* Formulation B: exact integer sub-block dot products first, then scales.
 *   q6_K:  y = sum_sb d * sum_c da_c * sum_{j in c} sc_j * P_j,
 *          P_j = sum_{k in j} (q-32)*qs  (16-element sub-blocks, int64)
 *   q4_K:  y = sum_sb sum_c da_c * (d*sc_c*P_c - dmin*m_c*ssum_c),
 *          P_c = sum_{k in c} q*qs       (32-element sub-blocks, int64)
 * ssum is the value stored in the activation block. */
int mmq_oracle_gemm_entries_int(int type, const uint8_t *W, int64_t od, int64_t id,
                                const uint8_t *Q, int64_t nt, const int64_t *ts,
                                const int64_t *os, int64_t n, double *y) {
    int bb = block_bytes(type);
    if (bb < 0 || id <= 0 || id % 256 != 0) return -1;
    int64_t nsb = id / 256, nb32 = id / 32;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = ts[i], o = os[i];
        if (t < 0 || t >= nt || o < 0 || o >= od) return -1;
        double acc = 0.0;
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = W + (o * nsb + sb) * bb;
            double sb_sum = 0.0;
            for (int cc = 0; cc < 8; ++cc) {
                const uint8_t *qb = Q + (t * nb32 + sb * 8 + cc) * OR_Q8_PITCH;
                double da = f16_bits_to_f64(rd_u16(qb));
                const int8_t *qs = (const int8_t *)(qb + OR_Q8_QS);
                if (type == OR_Q6_K) {
                    int64_t s = 0;
                    for (int half = 0; half < 2; ++half) {
                        int e0 = cc * 32 + half * 16;
                        int64_t p = 0;
                        for (int i2 = 0; i2 < 16; ++i2)
                            p += (int64_t)mmq_oracle_q6k_centered(blk, e0 + i2) * qs[half * 16 + i2];
                        s += (int64_t)q6k_scale(blk, e0) * p;
                    }
                    sb_sum += da * (double)s;
                } else {
                    int sc, m;
                    mmq_oracle_q4k_scale_min(blk, cc, &sc, &m);
                    int64_t p = 0;
                    for (int i2 = 0; i2 < 32; ++i2)
                        p += (int64_t)mmq_oracle_q4k_quant(blk, cc * 32 + i2) * qs[i2];
                    double d = f16_bits_to_f64(rd_u16(blk + OR_Q4_D));
                    double dmin = f16_bits_to_f64(rd_u16(blk + OR_Q4_DMIN));
                    sb_sum += da * (d * (double)sc * (double)p -
                                    dmin * (double)m * (double)rd_i32(qb + OR_Q8_SSUM));
                }
            }
            if (type == OR_Q6_K) sb_sum *= f16_bits_to_f64(rd_u16(blk + OR_Q6_D));
            acc += sb_sum;
        }
        y[i] = acc;
    }
    return 0;
}

/* The exact integer partial of each 32-element chunk c, with the weight's
 * sub-block scales applied but not d or the activation scale -- the sum the
 * pages' integer MMA produces per chunk before its float rescale:
 *   q6_K:  S[t][c][o] = sum_{j in c} sc_j * P_j,  P_j over 16 elements
 *   q4_K:  S[t][c][o] = sc_c * P_c,               P_c over 32 elements
 * (P as in formulation B).  S row-major nt x nb32 x od, int64. */
int mmq_oracle_chunk_partials(int type, const uint8_t *W, int64_t od, int64_t id,
                              const uint8_t *Q, int64_t nt, int64_t *S) {
    int bb = block_bytes(type);
    if (bb < 0 || id <= 0 || id % 256 != 0 || nt < 0 || od < 0) return -1;
    int64_t nsb = id / 256, nb32 = id / 32;
    for (int64_t t = 0; t < nt; ++t)
        for (int64_t c = 0; c < nb32; ++c) {
            const int8_t *qs = (const int8_t *)(Q + (t * nb32 + c) * OR_Q8_PITCH + OR_Q8_QS);
            int64_t sb = c / 8;
            int cc = (int)(c % 8);
            for (int64_t o = 0; o < od; ++o) {
                const uint8_t *blk = W + (o * nsb + sb) * bb;
                int64_t s = 0;
                if (type == OR_Q6_K) {
                    for (int half = 0; half < 2; ++half) {
                        int e0 = cc * 32 + half * 16;
                        int64_t p = 0;
                        for (int i2 = 0; i2 < 16; ++i2)
                            p += (int64_t)mmq_oracle_q6k_centered(blk, e0 + i2) * qs[half * 16 + i2];
                        s += (int64_t)q6k_scale(blk, e0) * p;
                    }
                } else {
                    int sc, m;
                    mmq_oracle_q4k_scale_min(blk, cc, &sc, &m);
                    int64_t p = 0;
                    for (int i2 = 0; i2 < 32; ++i2)
                        p += (int64_t)mmq_oracle_q4k_quant(blk, cc * 32 + i2) * qs[i2];
                    s = (int64_t)sc * p;
                }
                S[(t * nb32 + c) * od + o] = s;
            }
        }
    return 0;
}

/* Full nt x od output (formulation A) for small problems: dequantizes the
 * activations once and one weight row at a time.  Y row-major nt x od. */
int mmq_oracle_gemm(int type, const uint8_t *W, int64_t od, int64_t id, const uint8_t *Q,
                    int64_t nt, double *Y) {
    if (block_bytes(type) < 0 || id <= 0 || id % 256 != 0 || nt < 0 || od < 0) return -1;
    double *xh = (double *)malloc(sizeof(double) * (size_t)(nt > 0 ? nt : 1) * (size_t)id);
    double *wr = (double *)malloc(sizeof(double) * (size_t)id);
    if (!xh || !wr) {
        free(xh);
        free(wr);
        return -3;
    }
    mmq_oracle_dequant_act(Q, nt, id, xh);
    for (int64_t o = 0; o < od; ++o) {
        mmq_oracle_dequant_weights(type, W, od, id, o, o + 1, wr);
        for (int64_t t = 0; t < nt; ++t) {
            const double *x = xh + t * id;
            double acc = 0.0;
            for (int64_t k = 0; k < id; ++k) acc += wr[k] * x[k];
            Y[t * od + o] = acc;
        }
    }
    free(xh);
    free(wr);
    return 0;
}

/* The same output as mmq_oracle_gemm, with the weight rows shared out over
 * nthreads POSIX threads (contiguous row ranges).  Each output is the same
 * fp64 sum in the same order as there, so Y is identical bit for bit; only
 * the timing changes (the bench's CPU baseline runs on every host core). */
struct or_gemm_job {
    int type;
    const uint8_t *W;
    int64_t od, id, nt, o0, o1;
    const double *xh;
    double *Y;
    int rc;
};

static void *or_gemm_rows(void *arg) {
    struct or_gemm_job *j = (struct or_gemm_job *)arg;
    double *wr = (double *)malloc(sizeof(double) * (size_t)j->id);
    if (!wr) {
        j->rc = -3;
        return NULL;
    }
    for (int64_t o = j->o0; o < j->o1; ++o) {
        mmq_oracle_dequant_weights(j->type, j->W, j->od, j->id, o, o + 1, wr);
        for (int64_t t = 0; t < j->nt; ++t) {
            const double *x = j->xh + t * j->id;
            double acc = 0.0;
            for (int64_t k = 0; k < j->id; ++k) acc += wr[k] * x[k];
            j->Y[t * j->od + o] = acc;
        }
    }
    free(wr);
    j->rc = 0;
    return NULL;
}

int mmq_oracle_gemm_mt(int type, const uint8_t *W, int64_t od, int64_t id, const uint8_t *Q,
                       int64_t nt, double *Y, int nthreads) {
    if (block_bytes(type) < 0 || id <= 0 || id % 256 != 0 || nt < 0 || od < 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > od && od > 0) nthreads = (int)od;
    double *xh = (double *)malloc(sizeof(double) * (size_t)(nt > 0 ? nt : 1) * (size_t)id);
    struct or_gemm_job *jobs = (struct or_gemm_job *)calloc((size_t)nthreads, sizeof(*jobs));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int *started = (int *)calloc((size_t)nthreads, sizeof(int));
    if (!xh || !jobs || !th || !started) {
        free(xh);
        free(jobs);
        free(th);
        free(started);
        return -3;
    }
    mmq_oracle_dequant_act(Q, nt, id, xh);
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].type = type;
        jobs[i].W = W;
        jobs[i].od = od;
        jobs[i].id = id;
        jobs[i].nt = nt;
        jobs[i].o0 = od * i / nthreads;
        jobs[i].o1 = od * (i + 1) / nthreads;
        jobs[i].xh = xh;
        jobs[i].Y = Y;
        jobs[i].rc = -3;
        started[i] = pthread_create(&th[i], NULL, or_gemm_rows, &jobs[i]) == 0;
        if (!started[i]) or_gemm_rows(&jobs[i]); /* no thread: run the range here */
    }
    for (int i = 0; i < nthreads; ++i) {
        if (started[i]) pthread_join(th[i], NULL);
        if (jobs[i].rc != 0) rc = jobs[i].rc;
    }
    free(xh);
    free(jobs);
    free(th);
    free(started);
    return rc;
}
