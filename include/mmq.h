/*
 * mmq.h -- C ABI of the GB300 (sm_103a) k-quant x q8_0 prefill GEMM library
 * (libmmq.so).
 *
 * The operation is the prefill "MMQ" GEMM of the minfer CUDA optimisation
 * log:   Y[t][o] = sum_k W[o][k] * X[t][k]
 * with W stored as q6_K or q4_K super-blocks and X quantized per token into
 * q8_0 "pad40" blocks.  Three steps, one entry point each:
 *   mmq_quantize_act     X (fp32)            -> Q (q8_0 pad40 blocks)
 *   mmq_register_weights W (packed k-quant)  -> handle (internal planes,
 *                                               optional dense W_exp plane)
 *   mmq_gemm             handle, Q           -> Y (fp32)
 * and mmq_gemm_f32 (handle, X -> Y) for the two steps fused.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device pointers on the current device;
 *     the caller owns them.  Nothing is freed or retained by the library
 *     except inside an mmq_weights_t handle.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) unless stated otherwise.
 *   - Return value: MMQ_OK (0) or a negative MMQ_ERR_* code.  Argument
 *     checks happen on the host before anything is enqueued; no C++
 *     exception crosses this boundary.
 *   - A device-side bounded wait that expires records a status word read by
 *     mmq_last_device_error(); the kernel then returns instead of hanging.
 */
#ifndef MMQ_H
#define MMQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mmq_stream_t;   /* same type as cudaStream_t */
typedef struct mmq_weights_s *mmq_weights_t;

/* ---- status codes ------------------------------------------------------ */
#define MMQ_OK 0
#define MMQ_ERR_ARG -1             /* null pointer, bad size, id % 256 != 0, ... */
#define MMQ_ERR_ALIGN -2           /* a pointer misses the alignment stated below */
#define MMQ_ERR_TYPE -3            /* unknown weight type */
#define MMQ_ERR_CUDA -4            /* a CUDA runtime call failed */
#define MMQ_ERR_DEVICE_TIMEOUT -5  /* a bounded device wait expired (see above) */
#define MMQ_ERR_OOM -6             /* device allocation failed */
#define MMQ_ERR_UNSUPPORTED -7     /* valid input this build does not handle */
#define MMQ_ERR_NO_DEVICE -8       /* current device is not a GB300 (sm_103) */
#define MMQ_ERR_SCRATCH_LIMIT -9   /* problem exceeds mmq_gemm_noalloc's fixed scratch */

/* ---- weight types (ggml numbering) ------------------------------------- */
#define MMQ_Q4_K 12
#define MMQ_Q6_K 14

/* ---- byte layouts (defined once; the library's kernels use these) ------
 * q8_0 pad40 activation block, one per token t per 32-element chunk c of K,
 * block (t, c) at byte (t*nb32 + c)*40, nb32 = id/32.
 * Source: "26 · r21 — Coalesced block-linear A staging", §2.1, and
 * "25 · r20: Split-phase A staging", §3.2.
 *   [0,2)  d    fp16, little-endian;  [2,4) zero
 *   [4,36) qs   32 x int8;            [36,40) ssum int32 = sum of qs        */
#define MMQ_Q8_BLOCK_BYTES 40
#define MMQ_Q8_D_OFF 0
#define MMQ_Q8_QS_OFF 4
#define MMQ_Q8_SSUM_OFF 36
/* block_q6_K, 256 weights in 16 sub-blocks of 16, w = d*sc[e/16]*(q-32).
 * Source: "47 · r44 — W_exp stride mismatch root cause", §2.2; scale bytes
 * at 192: "46 · r43 — PC-sampling attribution", §3.1.                      */
#define MMQ_Q6K_BLOCK_BYTES 210
#define MMQ_Q6K_QL_OFF 0
#define MMQ_Q6K_QH_OFF 128
#define MMQ_Q6K_SC_OFF 192
#define MMQ_Q6K_D_OFF 208
/* block_q4_K, 256 weights in 8 sub-blocks of 32, w = d*sc*q - dmin*m.  Not
 * printed on the pages; the ggml layout is the reading taken.              */
#define MMQ_Q4K_BLOCK_BYTES 144
#define MMQ_Q4K_D_OFF 0
#define MMQ_Q4K_DMIN_OFF 2
#define MMQ_Q4K_SC_OFF 4
#define MMQ_Q4K_QS_OFF 16
/* every GEMM entry point requires id % MMQ_QK == 0 ("the NB-BT launch gate",
 * "47 · r44 — W_exp stride mismatch root cause", §3.1)                     */
#define MMQ_QK 256

/* ---- registration flags ------------------------------------------------ */
#define MMQ_REG_WEXP 0x1u  /* also build the dense int8 W_exp code plane */
#define MMQ_REG_RAW 0x2u   /* also keep the packed bytes, regrouped, for MMQ_ARM_RAW */

/* ---- GEMM arms (flags of mmq_gemm select one; arm_used reports it) ----- */
#define MMQ_ARM_AUTO 0     /* library choice: MMQ_ARM_PAIR above 128 tokens for one-plane
                              operands (q4_K, and q6_K with every |sc| <= 64), except
                              q6_K problems whose 256-row split tiles fill two or more
                              waves of SMs to 85 %; otherwise MMQ_ARM_SPLIT for one-plane
                              q6_K, and for q4_K when the split arm runs 256-row weight
                              tiles (problems with more 128 x 128 output tiles than SMs)
                              or pieces of tiles (problems with at most half as many tiles
                              as SMs); else MMQ_ARM_F16 */
#define MMQ_ARM_F16 1      /* operands from the registered fp16 operand plane (bulk copies) */
#define MMQ_ARM_RAW 2      /* packed weight bytes streamed and unpacked to fp16 in shared
                              memory inside the GEMM ("47 · r44 — W_exp stride mismatch
                              root cause", §3.2: the in-kernel recombination); needs a
                              handle registered with MMQ_REG_RAW whose operand is one
                              plane (q4_K, or q6_K with every |sc| <= 64; otherwise
                              MMQ_ERR_UNSUPPORTED); bit-identical to F16 */
#define MMQ_ARM_SPLIT 3    /* the activation scale folded into the A operand as an exact
                              fp16 pair (hi = rn(da'*qs), lo = rn(da'*qs - hi)), so the
                              tensor core sums a whole 256-K super-block and the scales
                              apply once per super-block: every product exact, fp32
                              summation (results within the GEMM tolerance, not
                              bit-identical to F16); whole tiles of 128 or 256 weight
                              rows per CTA, or -- with at most half as many 128 x 128
                              tiles as SMs -- each tile's super-blocks cut into pieces
                              over several CTAs whose partial sums are added in a fixed
                              order (repeat calls bit-identical) */
#define MMQ_ARM_PAIR 4     /* MMQ_ARM_SPLIT's operands and arithmetic on pairs of SMs: 2-CTA
                              clusters run cta_group::2 UMMAs of 256 weight rows x 128 (112,
                              96) tokens, each SM staging its own 128 weight rows and half
                              of the token rows, so a 64-K stage of the operand ring holds a
                              third less and takes two bulk copies; whole tiles; results
                              within fp32 summation of MMQ_ARM_SPLIT's (the tensor core sums
                              the transposed tile in its own order); handles whose operand
                              is one plane (otherwise MMQ_ERR_UNSUPPORTED) */

/*
 * mmq_quantize_act -- q8_0 quantization of activations.
 * Source: the pad40 block of "26 · r21 — Coalesced block-linear A staging",
 * §2.1; the quantizer itself (d = amax/127, q = round-half-away(x/d)) is the
 * task's workload definition, computed in fp32 with IEEE division.
 *   X   device, fp32, nt x id row-major, 16-byte aligned.
 *   nt  tokens (>= 0; 0 is a no-op).   id  K, a positive multiple of 32.
 *   Q   device, caller-allocated nt*(id/32)*40 bytes, 16-byte aligned;
 *       fully overwritten (pad bytes [2,4) of each block are written as 0).
 * Non-finite X, or |X| large enough that amax/127 overflows fp16, is out of
 * contract (no error is raised; the bytes written are unspecified).
 * Errors: MMQ_ERR_ARG, MMQ_ERR_ALIGN, MMQ_ERR_NO_DEVICE, MMQ_ERR_CUDA.
 */
int mmq_quantize_act(const float *X, int64_t nt, int64_t id, void *Q, mmq_stream_t stream);

/*
 * mmq_register_weights -- one-time expansion of a packed k-quant weight.
 * Source: registration-time expansion and the dense W_exp plane of
 * "46 · r43 — PC-sampling attribution", §3.2, and "47 · r44 — W_exp stride
 * mismatch root cause", §2.1-2.2 (out[j*id + sb*256 + e] = q - 32, row pitch
 * id, super-block pitch 256).
 *   type  MMQ_Q6_K or MMQ_Q4_K.
 *   W     device, od rows of id/256 packed blocks (210 B q6_K, 144 B q4_K),
 *         row pitch (id/256)*block bytes, no alignment requirement.  Read
 *         only during this call; the caller keeps ownership.
 *   od    output rows (> 0).   id  K, a positive multiple of 256.
 *   flags MMQ_REG_WEXP: also keep the dense int8 W_exp code plane (od*id
 *         bytes): q6_K the centered code q - 32, q4_K the code q (the same
 *         plane carried to q4_K); the operand plane is then built by reading
 *         W_exp back with its dense strides.
 *         MMQ_REG_RAW: also keep the packed bytes regrouped for MMQ_ARM_RAW
 *         (od_pad*id*0.56 B q4_K, *0.88 B q6_K).
 *   out   receives a handle owning the internal planes (fp16 operand plane
 *         with sub-block scales folded in, fp32 scale planes, optional
 *         W_exp) until mmq_release_weights.
 * Synchronizes `stream` before returning (registration is a one-time cost).
 * q6_K sub-block scales take the whole int8 range.  While every |sc| <= 64
 * the folded operand sc*(q-32) (|.| <= 2048) is one exact fp16 plane; if any
 * |sc| > 64 (up to 4096, not always exact in fp16) the handle holds two
 * planes, B1 = 2*sc*((q-32) >> 1) and B0 = sc*((q-32) & 1), each exact, whose
 * sum the GEMM forms on the tensor core (twice the operand bytes; see
 * mmq_weights_info).  Errors: MMQ_ERR_ARG, MMQ_ERR_TYPE, MMQ_ERR_OOM,
 * MMQ_ERR_NO_DEVICE, MMQ_ERR_CUDA.
 */
int mmq_register_weights(int type, const void *W, int64_t od, int64_t id, uint32_t flags,
                         mmq_stream_t stream, mmq_weights_t *out);

/* Frees a handle and its device planes (synchronizes the device). NULL is
 * accepted.  Returns MMQ_OK or MMQ_ERR_CUDA. */
int mmq_release_weights(mmq_weights_t h);

/*
 * mmq_weights_wexp -- the dense int8 W_exp plane of a handle registered with
 * MMQ_REG_WEXP ("46 · r43 — PC-sampling attribution", §3.2; q6_K q - 32, q4_K q):
 * element (o, k) at plane[o*row_pitch + k], row_pitch == id, super-block
 * pitch 256.  The pointer is device memory owned by the handle.
 * Errors: MMQ_ERR_ARG (null argument), MMQ_ERR_UNSUPPORTED (no plane).
 */
int mmq_weights_wexp(mmq_weights_t h, const int8_t **plane, int64_t *row_pitch);

/*
 * mmq_dequantize_weights -- the dequantization fallback: packed k-quant rows
 * to a dense od x id plane of real weights, for consumers that do not run
 * the MMQ contraction ("47 · r44 — W_exp stride mismatch root cause", §2.2:
 * the dequant/embedding paths read the raw blocks).  Each weight
 * (q6_K d*sc*(q-32), q4_K d*sc*q - dmin*m) is formed exactly in fp64 and
 * rounded once, to nearest even, to the output type.
 *   type   MMQ_Q6_K or MMQ_Q4_K.   W  device, packed rows as for
 *          mmq_register_weights.   od, id  as there.
 *   out    device, od*id elements of out_type, row-major (row pitch id),
 *          16-byte aligned.
 *   out_type MMQ_OUT_F16 or MMQ_OUT_F32.
 * Errors: MMQ_ERR_ARG, MMQ_ERR_ALIGN, MMQ_ERR_TYPE, MMQ_ERR_NO_DEVICE,
 * MMQ_ERR_CUDA.
 */
#define MMQ_OUT_F16 1
#define MMQ_OUT_F32 2
int mmq_dequantize_weights(int type, const void *W, int64_t od, int64_t id, void *out,
                           int out_type, mmq_stream_t stream);

/* Sizes of a handle's device planes, in bytes (the VRAM side of the
 * registration trade-off, "47 · r44 — W_exp stride mismatch root cause",
 * §2.4).  Any out pointer may be NULL. */
int mmq_weights_info(mmq_weights_t h, int *type, int64_t *od, int64_t *id,
                     int64_t *operand_bytes, int64_t *scale_bytes, int64_t *wexp_bytes);

/*
 * mmq_gemm -- Y = dequant(Q) . dequant(W)^T for a registered weight.
 * Source: the MMQ contraction with per-sub-block integer dot products
 * rescaled by d*sc (q6_K: "47 · r44 — W_exp stride mismatch root cause",
 * §1.1 and §2.1) and the q4_K min correction through ssum.
 *   h     handle from mmq_register_weights (same device).
 *   Q     device, nt*(id/32)*40 bytes of pad40 blocks, 16-byte aligned.
 *   nt    tokens (>= 0; 0 is a no-op).
 *   Y     device, fp32, nt x od row-major, 16-byte aligned; overwritten.
 *   flags MMQ_ARM_AUTO or one MMQ_ARM_*; arm_used (may be NULL) receives
 *         the arm that ran.
 * Allocates its scratch -- the activation operand plane for tokens padded to
 * a multiple of 128 (nt_pad*id*2 bytes for MMQ_ARM_F16 and MMQ_ARM_RAW, plus
 * nt_pad*(id/32)*8 of per-block scales; nt_pad*id*4 of hi + lo images for
 * MMQ_ARM_SPLIT; about 1/16 more for q4_K's min images), and for a stream-K
 * launch of the fp16-plane arm one 64 KB partial tile per CTA (for the split
 * arm's pieces one 64 KB partial per piece and a counter per tile) -- stream-ordered from a
 * library-private memory pool and frees it stream-ordered; while `stream` is
 * being captured into a CUDA graph the scratch becomes a graph memory node
 * (cudaMallocAsync), so the call can be captured and replayed.
 * Errors: MMQ_ERR_ARG, MMQ_ERR_ALIGN, MMQ_ERR_UNSUPPORTED, MMQ_ERR_OOM,
 * MMQ_ERR_NO_DEVICE, MMQ_ERR_CUDA.  A device timeout is reported later by
 * mmq_last_device_error().
 */
int mmq_gemm(mmq_weights_t h, const void *Q, int64_t nt, float *Y, mmq_stream_t stream,
             uint32_t flags, int *arm_used);

/*
 * mmq_gemm_f32 -- the GEMM straight from fp32 activations: each token is
 * quantized to q8_0 exactly as mmq_quantize_act does and fed to the
 * contraction without the pad40 plane being written: the producer emits the
 * quantized operand plane directly, the step after the separate
 * quantize-transpose prepass in "26 · r21 — Coalesced block-linear A
 * staging", §5.  Y is bit-identical to mmq_quantize_act followed by
 * mmq_gemm on the same X.
 *   X     device, fp32, nt x id row-major, 16-byte aligned.
 *   Other arguments, scratch, the out-of-contract inputs of mmq_quantize_act
 *   and the errors as mmq_gemm.
 */
int mmq_gemm_f32(mmq_weights_t h, const float *X, int64_t nt, float *Y, mmq_stream_t stream,
                 uint32_t flags, int *arm_used);

/*
 * mmq_gemm_profiled -- mmq_gemm that also records two caller-created CUDA
 * events (cudaEvent_t, either may be NULL) on `stream` immediately before
 * and after the main GEMM kernel, so the caller can time that kernel alone.
 * Arguments and errors otherwise as mmq_gemm.
 */
int mmq_gemm_profiled(mmq_weights_t h, const void *Q, int64_t nt, float *Y, mmq_stream_t stream,
                      uint32_t flags, int *arm_used, void *ev_start, void *ev_stop);

/* mmq_gemm_f32 with the same two events around its main GEMM kernel. */
int mmq_gemm_f32_profiled(mmq_weights_t h, const float *X, int64_t nt, float *Y,
                          mmq_stream_t stream, uint32_t flags, int *arm_used, void *ev_start,
                          void *ev_stop);

/*
 * mmq_gemm_noalloc -- mmq_gemm for callers that cannot allocate device
 * memory: a caller whose GPU memory is entirely owned by another allocator
 * (for example a framework's caching allocator that reserved the device),
 * or one on a path where cudaMalloc's implicit device synchronization is not
 * acceptable.  The log pages have no counterpart to this entry point.
 * It allocates nothing: its scratch is a fixed 16 MiB device array compiled
 * into the library, which every device that loads the library holds until
 * the process exits.  The caller still passes Q and Y (as for mmq_gemm) and
 * a handle from mmq_register_weights, which must have run on the current
 * device first.
 *   - Problems whose scratch exceeds 16 MiB are rejected with
 *     MMQ_ERR_SCRATCH_LIMIT.  Scratch per token, with nt rounded up to a
 *     multiple of 128: id*2 + (id/32)*4 + 4 bytes, plus (id/256)*32 for q4_K;
 *     e.g. id = 3584 allows up to 2048 (q4_K) or 2176 (q6_K) tokens.
 *   - mmq_register_weights prepares what this entry point launches: it
 *     looks up the array's device address on its device and loads the
 *     GEMM's module and kernels there.  Without that, CUDA's lazy module
 *     loading (the default since CUDA 12.2) would load them -- allocating
 *     the array and the kernels' code -- inside the first call here.  So,
 *     after a registration on the device, no call allocates; the first call
 *     on a device still looks the address up in a host-side table, so make
 *     it before any stream capture.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents; each call rewrites or clears everything it reads.  Calls
 *     that can overlap on the GPU (different streams, no ordering) race on
 *     the array: order them on one stream or with events.
 * Always runs the MMQ_ARM_F16 arm.  Errors: MMQ_ERR_ARG, MMQ_ERR_ALIGN,
 * MMQ_ERR_SCRATCH_LIMIT, MMQ_ERR_NO_DEVICE, MMQ_ERR_CUDA; a device timeout is
 * reported by mmq_last_device_error().
 */
int mmq_gemm_noalloc(mmq_weights_t h, const void *Q, int64_t nt, float *Y, mmq_stream_t stream);

/*
 * mmq_debug_chunk_partials -- test hook for the integer exactness of the
 * fp16-plane arm: runs its GEMM (whole tiles) on Q and writes, for every
 * token t, 32-element chunk c and output row o, the raw partial the tensor
 * core left in TMEM before any float scale was applied:
 *   P[t][c][o] = sum_{k in chunk c} qs[t][k] * B[o][k],
 * B the registered operand (sc*(q-32) for q6_K, sc*q for q4_K; for a
 * two-plane q6_K handle the sum of both planes' UMMAs).  Each is an integer
 * below 2^24 in magnitude, stored exactly in fp32 (the per-sub-block integer
 * dot products of "47 · r44 — W_exp stride mismatch root cause", §1.1,
 * rescaled by sc).
 *   Q   device pad40 blocks as for mmq_gemm, 16-byte aligned.
 *   P   device, fp32, nt x (id/32) x od, 16-byte aligned; overwritten.
 * Takes nt_pad*(id/32)*od_pad*4 bytes of scratch beside the GEMM's (meant
 * for small problems).  Errors as mmq_gemm.
 */
int mmq_debug_chunk_partials(mmq_weights_t h, const void *Q, int64_t nt, float *P, mmq_stream_t stream);

/* Synchronizes the current device, then returns and clears the device status
 * word: MMQ_OK, or MMQ_ERR_DEVICE_TIMEOUT if a bounded wait expired since
 * the last call. */
int mmq_last_device_error(void);

/* Limit of every device-side wait, in ns (default 2e9).  Host-global. */
void mmq_set_wait_timeout_ns(uint64_t ns);

/* Failure-detection self test: launches one CTA that waits on a barrier
 * nothing arrives at, bounded by timeout_ns, then synchronizes and returns
 * mmq_last_device_error() -- MMQ_ERR_DEVICE_TIMEOUT when the bound works. */
int mmq_selftest_wait_timeout(uint64_t timeout_ns, mmq_stream_t stream);

/*
 * mmq_probe_engine_rates -- measurement hook, not part of the method: the
 * rates of the exact-integer-capable tensor engines on the current device,
 * the numbers behind the choice of tcgen05 kind::f16 for the integer
 * contraction and of the fp16/bf16 peak as the roofline's denominator (the
 * log pages run int8 IMMA; sm_103a has no tcgen05 kind::i8).  Writes
 *   out[0..2]  tcgen05.mma kind::f16, M = 128, K = 16, N = 64 / 128 / 256:
 *              MACs per clock per SM (one issuing warp per SM, back to back)
 *   out[3]     mma.sync m16n8k32 s8 -> s32 over the whole GPU, TOPS (2 ops per MAC)
 *   out[4]     mma.sync m16n8k16 f16 -> f32 over the whole GPU, TFLOP/s
 *   out[5..6]  as out[0..2], N = 96 / 112
 *   out[7..11] tcgen05.mma.cta_group::2 kind::f16 on 2-CTA clusters, M = 256,
 *              K = 16, N = 64 / 96 / 112 / 128 / 256: MACs per clock per SM
 *              of the pair (the pair arm's UMMA shape)
 * (12 doubles.)
 * Synchronizes `stream`; takes well under a second.  Errors: MMQ_ERR_ARG,
 * MMQ_ERR_NO_DEVICE, MMQ_ERR_CUDA, MMQ_ERR_DEVICE_TIMEOUT.
 */
int mmq_probe_engine_rates(double *out, mmq_stream_t stream);

/* Static text for a status code. */
const char *mmq_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* MMQ_H */
