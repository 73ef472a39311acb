// gemm.cu -- the k-quant x q8_0 MMQ GEMM on sm_103a tensor cores.
//
// The contraction the pages run on int8 IMMA ("25 · r20: Split-phase A
// staging", §2.2: one m16n8k32 per 4096 MACs) runs here on tcgen05 UMMA of
// kind::f16.  sm_103a has no kind::i8, so the integers travel as fp16:
//   A = qs in [-127, 127]                              exact in fp16
//   B = sc*(q-32) (q6_K, |sc| <= 64) or sc*q (q4_K)    |B| <= 2048, exact
// Every product is exact in the fp32 accumulator and a 32-element chunk sums
// to at most 32 * 127 * 2048 < 2^24, so each per-chunk partial
//   S[t][o][c] = sum_{k in c} qs[t][k] * B[o][k]
// lands in TMEM exactly: the pages' integer sub-block dot product with the
// sub-block scale already applied.  The epilogue rescales in two levels:
//   acc[t][o]  = sum_{c in sb} da'[t][c] * S[t][o][c]          (per chunk)
//   Y'[t][o] += d[o][sb] * acc[t][o]  -  dmin[o][sb] * MIN[t][o][sb]   (per super-block)
//   Y[t][o]   = Y'[t][o] * 2^-s_t                                (per tile)
// The q4_K min term  sum_c da*ssum * dmin*m  runs on the tensor core: per
// super-block one K=16 UMMA of  g' = da*ssum*2^s_t  split into fp16 hi + lo
// against the integer mins m  (MIN above).  g' carries up to 23 significant
// bits and hi + lo 22, so the split is exact for most chunks and otherwise
// off by one unit of about 2^-22 of the token's largest g'; s_t is a per-token power
// of two that keeps g' in fp16 range, and da' = da*2^s_t carries the same
// factor so the final scaling by 2^-s_t is exact.
//
// Data movement: operands arrive pre-tiled and pre-swizzled (tiling.h), two
// bulk copies per 128-K stage (activation block, weight block) into a
// 3-stage ring that only the tensor core releases, plus one small copy per
// super-block of the weight scales (d, dmin) into a 4-entry scale ring that
// the epilogue releases.
//
// Kernel shape: persistent, one CTA of 384 threads per SM (512 for the raw
// arm), 128 x 128 tiles, token tiles fastest so concurrently running CTAs
// share weight tiles in L2; whole tiles per CTA, or (few tiles, many
// super-blocks) the stream-K split below.
//   warps 0..7  epilogue: warp w reads TMEM lanes 32*(w%4).. and columns
//               64*(w/4)..: TMEM -> registers in 32-column halves,
//               software-pipelined with packed fp32x2 FMAs; one barrier wait
//               per pair of chunks
//   warp 8      producer: lane 0 the activation block, lane 1 the weight
//               block, lane 2 the scale block
//   warps 9-10  UMMA issuers (one elected lane of a warp-uniform loop each);
//               warp 9 also owns TMEM.  The eight 32-K chunks of a super-block
//               go in pairs, (0,1) and (4,5) to issuer 0, (2,3) and (6,7) to
//               issuer 1; each issuer has two of the four 128-column TMEM chunk
//               slots and commits every chunk on its slot's barrier (a commit
//               covers all earlier UMMAs of its thread, so a pair's second
//               barrier covers the pair); issuer 0 also issues the q4_K
//               min-term UMMA per super-block
//   warp 11     pulls the first weight blocks into L2 at launch
//   warps 12-15 (raw arm) converters: packed weight bytes -> fp16 operand
// The launch is programmatic: the producer and the epilogue wait for the
// prepass kernel just before their first read of its output.
// Every wait is bounded (ptx.cuh); a CTA that gives up drains its own copies
// and UMMAs, frees TMEM and returns.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "q8.cuh"
#include "tiling.h"

namespace mmq {
namespace {

using namespace tiling;

constexpr int SLOTS = 4;          // TMEM chunk slots of kTileN columns (512 columns)
constexpr int SRING = 4;          // per-super-block scale ring entries
constexpr int RRING = 4;          // raw arm: raw weight block ring entries
constexpr int EPI_WARPS = 8;      // warpgroups 0 and 1
constexpr int PRODUCER_WARP = 8;  // warpgroup 2: producer, two UMMA issuers, one idle warp
constexpr int PRODUCER2_WARP = 10;  // the pair arm's second producer
constexpr int ISSUER_WARP = 9;    // issuers 9 and 10; issuer i owns TMEM slots 2i and 2i+1
constexpr int ISSUERS = 2;
constexpr int CONVERTER_WARP = 12;  // raw arm: warpgroup 3 unpacks the weight blocks
constexpr int CONVERTERS = 4;
constexpr int TMEM_COLS = SLOTS * kTileN;  // 512

// Launch shape of the two arms.  Register split: the CTA is launched at
// kRegsLaunch per thread; warpgroup 2 (and the raw arm's converter
// warpgroup 3) drop to kRegsCtl and the two epilogue warpgroups rise to
// kRegsEpi, using the whole register file the launch holds.
template <bool kRaw, bool kB0 = false>
struct Shape {
  static constexpr int kStages = kB0 ? 4 : kRaw ? 2 : 3;
  static constexpr int kThreads = kRaw ? 512 : 384;
  static constexpr int kRegsLaunch = kRaw ? 128 : 168;
  static constexpr int kRegsEpi = kRaw ? 208 : 224;
  static constexpr int kRegsCtl = kRaw ? 48 : 56;
  static_assert(kThreads * kRegsLaunch <= 65536, "register file");
  static_assert(256 * kRegsEpi + (kThreads - 256) * kRegsCtl == kThreads * kRegsLaunch,
                "the register split must add up to what the launch holds");
};

// kB0 (q6_K with |sc| > 64): stages of 64 K (one K-block of A, B1 and B0,
// 16 KB each; four in the ring), each taken by one issuer; otherwise stages
// of 128 K (a half super-block).
template <bool kQ4, bool kRaw, bool kB0 = false>
struct Smem {
  using S = Shape<kRaw, kB0>;
  static constexpr int kKB = kTileM * 64 * 2;  // one 64-K block of a tile: 16384
  static constexpr int kA = kB0 ? kKB : a_odd_bytes(kQ4);                                // A region per stage
  static constexpr int kB = kB0 ? 2 * kKB : ((b_odd_bytes(kQ4) + 1023) / 1024) * 1024;  // B region per stage
  static constexpr int kB0Off = kKB;  // the B0 K-block after the B1 one
  static constexpr int kStage = kA + kB;
  static constexpr int kRaw_ = ((raw_block_bytes(kQ4) + 127) / 128) * 128;  // one raw ring entry
  static constexpr int kRawRing = S::kStages * kStage;
  static constexpr int kScale = scale_block_bytes(kQ4);                // one scale ring entry
  static constexpr int kScaleRing = kRawRing + (kRaw ? RRING * kRaw_ : 0);
  static constexpr int kBar = kScaleRing + SRING * kScale;
  // full, empty, conv per stage; rfull, rempty per slot; sfull, sempty per
  // scale entry; rawfull, rawempty per raw entry; done
  static constexpr int kNumBars = 3 * S::kStages + 2 * SLOTS + 2 * SRING + 2 * RRING + 1;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kUsed = kSlot + 16;
  static constexpr int kBytes = kUsed + 1024;  // slack for 1024-byte alignment
  static_assert(kA % 1024 == 0 && kStage % 1024 == 0, "stage buffers must keep 1 KB alignment");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

// ---------------------------------------------------------------- raw unpack
// 4 values of 4-bit or 6-bit codes (one per byte of x) -> 2 x half2 of
// 1024 + code (the 0x64 exponent byte above each code byte).
__device__ __forceinline__ uint32_t bytes01_to_h2(uint32_t x) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(d) : "r"(x), "r"(0x64646464u));
  return d;
}
__device__ __forceinline__ uint32_t bytes23_to_h2(uint32_t x) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(d) : "r"(x), "r"(0x64646464u));
  return d;
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, __half2 b, __half2 c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&a), b, c);
  return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t h2_sub(uint32_t a, __half2 b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&a), b);
  return *reinterpret_cast<const uint32_t *>(&r);
}

// One stage (half super-block, 128 rows x 128 K) of raw weight bytes ->
// the fp16 operand image, byte-identical to the registered operand plane:
// q4_K sc*q (as (1024+q)*sc - 1024*sc, one exact fp16 FMA), q6_K sc*(q-32)
// (as ((1024+q) - 1056) * sc + 0, exact, +0 for zero).  Thread t of the
// converter warpgroup handles row t.
template <bool kQ4>
__device__ __forceinline__ void unpack_stage(const uint8_t *__restrict__ raw, uint8_t *__restrict__ bop,
                                             int r) {
  if constexpr (kQ4) {
    const uint2 *qs = reinterpret_cast<const uint2 *>(raw + kRawQ4Qs);
    const __half *sc = reinterpret_cast<const __half *>(raw + kRawQ4Sc);
    __half2 s2[4], n2[4];
#pragma unroll
    for (int sub = 0; sub < 4; ++sub) {
      s2[sub] = __half2half2(sc[sub * 128 + r]);
      n2[sub] = __hmul2(s2[sub], __float2half2_rn(-1024.0f));  // exact: 1024 * sc <= 64512
    }
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint2 w = qs[(kb * 4 + j) * 128 + r];
        const uint32_t l0 = w.x & 0x0F0F0F0Fu, l1 = w.y & 0x0F0F0F0Fu;
        const uint32_t h0 = (w.x >> 4) & 0x0F0F0F0Fu, h1 = (w.y >> 4) & 0x0F0F0F0Fu;
        const int sl = 2 * kb, sh = 2 * kb + 1;
        const uint4 lo = make_uint4(h2_fma(bytes01_to_h2(l0), s2[sl], n2[sl]),
                                    h2_fma(bytes23_to_h2(l0), s2[sl], n2[sl]),
                                    h2_fma(bytes01_to_h2(l1), s2[sl], n2[sl]),
                                    h2_fma(bytes23_to_h2(l1), s2[sl], n2[sl]));
        const uint4 hi = make_uint4(h2_fma(bytes01_to_h2(h0), s2[sh], n2[sh]),
                                    h2_fma(bytes23_to_h2(h0), s2[sh], n2[sh]),
                                    h2_fma(bytes01_to_h2(h1), s2[sh], n2[sh]),
                                    h2_fma(bytes23_to_h2(h1), s2[sh], n2[sh]));
        *reinterpret_cast<uint4 *>(bop + operand_off(r, 64 * kb + 8 * j)) = lo;
        *reinterpret_cast<uint4 *>(bop + operand_off(r, 64 * kb + 8 * (j + 4))) = hi;
      }
  } else {
    const uint2 *ql = reinterpret_cast<const uint2 *>(raw + kRawQ6Ql);
    const uint2 *qh = reinterpret_cast<const uint2 *>(raw + kRawQ6Qh);
    const __half *sc = reinterpret_cast<const __half *>(raw + kRawQ6Sc);
    const __half2 off2 = __float2half2_rn(1056.0f), zero2 = __float2half2_rn(0.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 a = ql[j * 128 + r], b = ql[(j + 4) * 128 + r], h = qh[j * 128 + r];
      // chunk (kb, jj): low bits from ql nibble kb, high bits from qh pair 2*kb + (jj >= 4)
      auto chunk = [&](uint2 q, int nib, int pair, int kb, int jj) {
        const uint32_t lo0 = (q.x >> (4 * nib)) & 0x0F0F0F0Fu, lo1 = (q.y >> (4 * nib)) & 0x0F0F0F0Fu;
        const uint32_t v0 = lo0 | (((h.x >> (2 * pair)) & 0x03030303u) << 4);
        const uint32_t v1 = lo1 | (((h.y >> (2 * pair)) & 0x03030303u) << 4);
        const __half2 s2 = __half2half2(sc[(4 * kb + (jj >> 1)) * 128 + r]);
        const uint4 o = make_uint4(h2_fma(h2_sub(bytes01_to_h2(v0), off2), s2, zero2),
                                   h2_fma(h2_sub(bytes23_to_h2(v0), off2), s2, zero2),
                                   h2_fma(h2_sub(bytes01_to_h2(v1), off2), s2, zero2),
                                   h2_fma(h2_sub(bytes23_to_h2(v1), off2), s2, zero2));
        *reinterpret_cast<uint4 *>(bop + operand_off(r, 64 * kb + 8 * jj)) = o;
      };
      chunk(a, 0, 0, 0, j);
      chunk(b, 0, 1, 0, j + 4);
      chunk(a, 1, 2, 1, j);
      chunk(b, 1, 3, 1, j + 4);
    }
  }
}

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared-memory descriptor for the 32-byte-swizzled K=16 min-term images:
// rows of 32 B, 8-row groups 256 B apart, swizzle mode 6 (32 B).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw32(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(256 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(6) << 61;
  return d;
}

// ---------------------------------------------------------------- activation prepass
// One CTA of 128 threads per token t < nt: pad40 blocks -> the token's row of
// every activation block (fp16 qs, swizzled), da' = da*2^s_t, inv = 2^-s_t,
// and for q4_K the min-term image slots hi/lo of g' = da*ssum*2^s_t.
template <bool kQ4>
__global__ void __launch_bounds__(128) gemm_prepass_kernel(const uint8_t *__restrict__ Q,
                                                           int64_t nt, int64_t nb32,
                                                           uint8_t *__restrict__ aplane,
                                                           float *__restrict__ dap,
                                                           float *__restrict__ invp,
                                                           uint64_t *__restrict__ flags, int nflags) {
  griddep_launch_dependents();
  if (blockIdx.x == 0)  // the GEMM's stream-K hand-off flags start clear (a graph replays its tags)
    for (int i = threadIdx.x; i < nflags; i += blockDim.x) flags[i] = 0;
  const int64_t t = blockIdx.x;
  const bool live = t < nt;  // rows nt .. nt_pad - 1 of the last tile: a zero activation row
  const int tid = threadIdx.x;
  const uint8_t *qrow = Q + (live ? t : 0) * nb32 * MMQ_Q8_BLOCK_BYTES;
  const int64_t nsb = nb32 / 8;
  int s = 0;
  if (kQ4) {  // s_t: the token's largest |g| lands in [2^14, 2^15)
    __shared__ float wmax[4];
    float gmax = 0.f;
    for (int64_t c = tid; c < nb32 && live; c += 128) {
      const uint8_t *b = qrow + c * MMQ_Q8_BLOCK_BYTES;
      const float da = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short *>(b)));
      const int ssum = *reinterpret_cast<const int *>(b + MMQ_Q8_SSUM_OFF);
      gmax = fmaxf(gmax, fabsf(da * static_cast<float>(ssum)));
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, m));
    if ((tid & 31) == 0) wmax[tid >> 5] = gmax;
    __syncthreads();
    gmax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    if (gmax > 0.f) {
      const int e = static_cast<int>((__float_as_uint(gmax) >> 23) & 0xFF) - 127;
      s = min(30, max(-30, 14 - e));
    }
  }
  const float scale = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
  const int r = static_cast<int>(t & (kTileM - 1));
  const int64_t tile = t / kTileM;
  if (tid == 0) invp[t] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  for (int64_t c = tid; c < nb32; c += 128) {
    const uint2 *src = reinterpret_cast<const uint2 *>(qrow + c * MMQ_Q8_BLOCK_BYTES);
    const uint2 z = make_uint2(0u, 0u);
    const uint2 w0 = live ? __ldg(src + 0) : z, w1 = live ? __ldg(src + 1) : z, w2 = live ? __ldg(src + 2) : z,
                w3 = live ? __ldg(src + 3) : z, w4 = live ? __ldg(src + 4) : z;
    const uint32_t qw[8] = {w0.y, w1.x, w1.y, w2.x, w2.y, w3.x, w3.y, w4.x};
    const int64_t sb = c >> 3;
    const int half = static_cast<int>((c >> 2) & 1);
    uint8_t *blk = aplane + a_block(tile, sb, half, nsb, kQ4);
    const int k0 = static_cast<int>(c & 3) * 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __half h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w = qw[2 * q + (j >> 2)];
        h[j] = __int2half_rn(static_cast<int8_t>((w >> (8 * (j & 3))) & 0xFF));
      }
      *reinterpret_cast<uint4 *>(blk + operand_off(r, k0 + 8 * q)) =
          *reinterpret_cast<const uint4 *>(h);
    }
    const float da = __half2float(__ushort_as_half(static_cast<unsigned short>(w0.x & 0xFFFFu)));
    dap[t * nb32 + c] = da * scale;
    if (kQ4) {
      const float g = da * static_cast<float>(static_cast<int>(w4.y)) * scale;  // exact
      const __half hi = __float2half_rn(g);
      const __half lo = __float2half_rn(g - __half2float(hi));
      uint8_t *mblk = aplane + a_block(tile, sb, 1, nsb, true) + kAMin;
      const uint32_t pair = static_cast<uint32_t>(__half_as_ushort(hi)) |
                            (static_cast<uint32_t>(__half_as_ushort(lo)) << 16);
      *reinterpret_cast<uint32_t *>(mblk + min_off(r, 2 * static_cast<int>(c & 7))) = pair;
    }
  }
}

// ---------------------------------------------------------------- fused quantization
// The same per-token result as mmq_quantize_act followed by the prepass
// above, straight from fp32 activations: one CTA of 128 threads per token,
// eight lanes per 32-value block (one float4 each).  The quantization is the
// q8_0 rule of quantize.cu (d = amax/127 by IEEE division, q = round half
// away from zero of x/d, d16 = fp16_rn(d)), so the operand plane, da' and the
// min slots are bit-identical to the two-kernel path.  For q4_K the token's
// scale exponent s_t needs every block first: a first pass computes it, the
// second (reading X again, from L2) writes the planes.
// the q8_0 rule of quantize.cu (q8.cuh) on one lane's float4 of a block: the
// block's d16 (as fp32), its code sum and the lane's codes as two half2 words
__device__ __forceinline__ void quant_block8(float4 v, float &d16f, uint32_t &h01, uint32_t &h23, int &ssum) {
  float q[4];
  q8_lane(v, d16f, q);
  ssum = static_cast<int>(q8_ssum(q));
  h01 = q8_h2(q[0], q[1]);
  h23 = q8_h2(q[2], q[3]);
}

// One 32-value block's fp16 operand words in the token's operand row; lane
// `part` of the block's eight writes its 4 values.
template <bool kQ4>
__device__ __forceinline__ void emit_operand(uint8_t *__restrict__ aplane, int64_t t, int64_t c,
                                             int64_t nb32, int part, uint32_t h01, uint32_t h23) {
  const int64_t nsb = nb32 / 8;
  const int r = static_cast<int>(t & (kTileM - 1));
  uint8_t *blk = aplane + a_block(t / kTileM, c >> 3, static_cast<int>((c >> 2) & 1), nsb, kQ4);
  const int k0 = static_cast<int>(c & 3) * 32;
  *reinterpret_cast<uint2 *>(blk + operand_off(r, k0 + 4 * part)) = make_uint2(h01, h23);
}

// One block's da' and (q4_K) min-term slots, written by one thread.
template <bool kQ4>
__device__ __forceinline__ void emit_scales(uint8_t *__restrict__ aplane, float *__restrict__ dap,
                                            int64_t t, int64_t c, int64_t nb32, float d16f, int ssum,
                                            float scale) {
  dap[t * nb32 + c] = d16f * scale;
  if (kQ4) {
    const int64_t nsb = nb32 / 8;
    const int r = static_cast<int>(t & (kTileM - 1));
    const float g = d16f * static_cast<float>(ssum) * scale;  // exact
    const __half hi = __float2half_rn(g);
    const __half lo = __float2half_rn(g - __half2float(hi));
    uint8_t *mblk = aplane + a_block(t / kTileM, c >> 3, 1, nsb, true) + kAMin;
    const uint32_t pair = static_cast<uint32_t>(__half_as_ushort(hi)) |
                          (static_cast<uint32_t>(__half_as_ushort(lo)) << 16);
    *reinterpret_cast<uint32_t *>(mblk + min_off(r, 2 * static_cast<int>(c & 7))) = pair;
  }
}

// The operand words do not depend on the token scale s_t, so the first pass
// writes them; q4_K's da' and min-term slots wait for s_t.  kStash (q4_K):
// the first pass keeps every block's d16 and ssum in shared memory (8 B per
// block) for the second; otherwise the second pass re-reads X and quantizes
// again.  Each warp takes 16 blocks per step, four loads in flight per lane.
constexpr int kStashBytesPerBlock = 8;
constexpr int kStashMaxBytes = 48 * 1024;

constexpr int kQuantWarps = 8;  // one step of 16 blocks per warp covers id <= 4096

template <bool kQ4, bool kStash>
__global__ void __launch_bounds__(32 * kQuantWarps) quantize_prepass_kernel(const float *__restrict__ X,
                                                               int64_t nt, int64_t nb32,
                                                               uint8_t *__restrict__ aplane,
                                                               float *__restrict__ dap,
                                                               float *__restrict__ invp,
                                                               uint64_t *__restrict__ flags, int nflags) {
  extern __shared__ float stash[];  // [nb32] d16, then [nb32] ssum
  griddep_launch_dependents();
  if (blockIdx.x == 0)  // the GEMM's stream-K hand-off flags start clear (a graph replays its tags)
    for (int i = threadIdx.x; i < nflags; i += blockDim.x) flags[i] = 0;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = lane & 7, grp = lane >> 3;
  const bool live = t < nt;  // rows nt .. nt_pad - 1 of the last tile: a zero activation row
  const float4 *xrow = reinterpret_cast<const float4 *>(X + (live ? t : 0) * nb32 * 32);
  float *sd16 = stash;
  int *sssum = reinterpret_cast<int *>(stash + nb32);
  float gmax = 0.f;
  // pass 1: operand words (and, for q6_K, whose operands need no token scale, everything)
  for (int64_t base = warp * 16; base < nb32; base += 16 * kQuantWarps) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = base + u * 4 + grp;
      v[u] = c < nb32 && live ? __ldg(xrow + c * 8 + part) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = base + u * 4 + grp;
      float d16f;
      uint32_t h01, h23;
      int ssum;
      quant_block8(v[u], d16f, h01, h23, ssum);
      if (c >= nb32) continue;
      emit_operand<kQ4>(aplane, t, c, nb32, part, h01, h23);
      if (!kQ4) {
        if (part == 0) emit_scales<false>(aplane, dap, t, c, nb32, d16f, ssum, 1.0f);
      } else {
        gmax = fmaxf(gmax, fabsf(d16f * static_cast<float>(ssum)));
        if (kStash && part == 0) {
          sd16[c] = d16f;
          sssum[c] = ssum;
        }
      }
    }
  }
  if constexpr (!kQ4) {
    if (tid == 0) invp[t] = 1.0f;
  } else {
  // s_t: the token's largest |d16 * ssum| lands in [2^14, 2^15)
  __shared__ float wmax[kQuantWarps];
#pragma unroll
  for (int m = 16; m; m >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, m));
  if (lane == 0) wmax[warp] = gmax;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kQuantWarps; ++w) gmax = fmaxf(gmax, wmax[w]);
  int s = 0;
  if (gmax > 0.f) {
    const int e = static_cast<int>((__float_as_uint(gmax) >> 23) & 0xFF) - 127;
    s = min(30, max(-30, 14 - e));
  }
  const float scale = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
  if (tid == 0) invp[t] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  // pass 2: da' and the min-term slots
  if (kStash) {
    for (int64_t c = tid; c < nb32; c += 32 * kQuantWarps)
      emit_scales<true>(aplane, dap, t, c, nb32, sd16[c], sssum[c], scale);
  } else {
    for (int64_t base = warp * 16; base < nb32; base += 16 * kQuantWarps) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t c = base + u * 4 + grp;
        v[u] = c < nb32 && live ? __ldg(xrow + c * 8 + part) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t c = base + u * 4 + grp;
        float d16f;
        uint32_t h01, h23;
        int ssum;
        quant_block8(v[u], d16f, h01, h23, ssum);
        if (c < nb32 && part == 0) emit_scales<true>(aplane, dap, t, c, nb32, d16f, ssum, scale);
      }
    }
  }
  }
}

// ---------------------------------------------------------------- split-arm prepass
// The split arm's activation blocks (tiling.h): a = d16 * 2^s_t * q, exact in
// fp32 (11 x 7 significant bits), travels as fp16 hi = rn(a), lo = rn(a - hi).
// The pair is exact while |a| >= 2^-7 (lo keeps its bits above the fp16
// subnormal step), i.e. for every block within 2^22 of the token's largest.
// s_t puts the token's largest |d16 * 127| and (q4_K) |d16 * ssum| in
// [2^14, 2^15), so hi, lo and the min-term g' stay in fp16 range; inv = 2^-s_t.
__device__ __forceinline__ int split_scale_exp(float m) {
  if (!(m > 0.f)) return 0;
  const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127;
  return min(30, max(-30, 14 - e));
}

// two integer codes (as fp32) times da_s -> hi word and lo word, both lanes
// of the pair at once (packed fp32x2 arithmetic, paired fp16 conversions)
__device__ __forceinline__ void split_pair(float2 q, float da_s, uint32_t &hi, uint32_t &lo) {
  const float2 a = __fmul2_rn(make_float2(da_s, da_s), q);
  const __half2 h = __float22half2_rn(a);  // a is exact; h = rn(a) per lane
  // a - h is exact in fp32; fma(h, -1, a) forms it in one packed instruction
  const __half2 l = __float22half2_rn(__ffma2_rn(__half22float2(h), make_float2(-1.0f, -1.0f), a));
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Lane `part` of block c's eight: its 4 values into the hi and lo images, and
// (part 0, q4_K) the block's min-term slots.
// kPair: the pair arm's block layout (tiling.h) with token tiles of tp rows,
// else the split arm's.
template <bool kQ4, bool kPair>
__device__ __forceinline__ void emit_split(uint8_t *__restrict__ aplane, int64_t t, int64_t c, int64_t nb32,
                                           int part, float2 q01, float2 q23, float d16f, int ssum,
                                           float scale, int tp) {
  const int64_t nsb = nb32 / 8;
  const int64_t tile = kPair ? t / tp : t / kTileM;
  const int r = static_cast<int>(kPair ? t % tp : t & (kTileM - 1)), h = tp / 2;
  const int half = static_cast<int>((c >> 2) & 1), k = static_cast<int>(c & 3) * 32 + 4 * part;
  uint8_t *blk = aplane + (kPair ? pair_block(tile, c >> 3, half, nsb, kQ4, h) : as_block(tile, c >> 3, half, nsb, kQ4));
  const uint32_t off = kPair ? pair_off(r, k, kQ4, half, h) : split_off(r, k);
  const float da_s = d16f * scale;
  uint32_t hi0, lo0, hi1, lo1;
  split_pair(q01, da_s, hi0, lo0);
  split_pair(q23, da_s, hi1, lo1);
  *reinterpret_cast<uint2 *>(blk + off) = make_uint2(hi0, hi1);
  *reinterpret_cast<uint2 *>(blk + (kPair ? pair_kb_bytes(h) : kSplitLo) + off) = make_uint2(lo0, lo1);
  if (kQ4 && part == 0) {
    const float g = d16f * static_cast<float>(ssum) * scale;  // exact to fp32
    const __half hi = __float2half_rn(g);
    const __half lo = __float2half_rn(g - __half2float(hi));
    uint8_t *mblk = aplane + (kPair ? pair_block(tile, c >> 3, 1, nsb, true, h) : as_block(tile, c >> 3, 1, nsb, true));
    const int j = 2 * static_cast<int>(c & 7);
    *reinterpret_cast<uint32_t *>(mblk + (kPair ? pair_min_off(r, j, h) : kSplitMin + min_off(r, j))) =
        static_cast<uint32_t>(__half_as_ushort(hi)) | (static_cast<uint32_t>(__half_as_ushort(lo)) << 16);
  }
}

// the largest value the token's scale has to keep in range, for one block
template <bool kQ4>
__device__ __forceinline__ float split_range(float d16f, int ssum) {
  const float m = d16f * 127.0f;
  return kQ4 ? fmaxf(m, fabsf(d16f * static_cast<float>(ssum))) : m;
}

constexpr int kSplitStashBytesPerBlock = 72;  // 32 fp16 codes, d16, ssum

// the four int8 codes of one word as two fp32 pairs (low byte first)
__device__ __forceinline__ void codes_of_word(uint32_t w, float2 &q01, float2 &q23) {
  q01 = make_float2(static_cast<float>(static_cast<int8_t>(w & 0xFF)),
                    static_cast<float>(static_cast<int8_t>((w >> 8) & 0xFF)));
  q23 = make_float2(static_cast<float>(static_cast<int8_t>((w >> 16) & 0xFF)),
                    static_cast<float>(static_cast<int8_t>(w >> 24)));
}

// Eight consecutive codes (four half2 words, fp16 integers) times da_s ->
// 16 bytes of the hi image and 16 of the lo image (split_pair per pair).
__device__ __forceinline__ void split_chunk(uint4 codes, float da_s, uint4 &hi, uint4 &lo) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    split_pair(__half22float2(*reinterpret_cast<const __half2 *>(&w[i])), da_s, h[i], l[i]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// From fp32 X: one CTA of eight warps per token.  Pass one, eight lanes per
// 32-value block: the q8_0 rule (q8.cuh); each block's codes (fp16), d16 and
// code sum go to shared memory (kStash), and the token's scale exponent s_t
// is reduced over its blocks.  Pass two, one thread per 8-value chunk: the
// chunk's hi and lo words, one 16-byte store each, and (q4_K, first chunk of
// a block) the block's min-term slots.  Without kStash (tokens too long for
// shared memory) pass two quantizes X again, per block as in pass one.
// kPair: the pair arm's block layout, token tiles of tp rows.
template <bool kQ4, bool kStash, bool kPair = false>
__global__ void __launch_bounds__(32 * kQuantWarps, kStash ? 5 : 4) split_prepass_f32_kernel(const float *__restrict__ X,
                                                                   int64_t nt, int64_t nb32,
                                                                   uint8_t *__restrict__ aplane,
                                                                   float *__restrict__ invp,
                                                                   int *__restrict__ cnt, int ncnt, int tp) {
  extern __shared__ uint4 sstash4[];  // [nb32][4] 16-byte code chunks, then [nb32] d16, [nb32] ssum
  griddep_launch_dependents();
  if (blockIdx.x == 0)  // the GEMM's per-tile piece counters start at zero
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = lane & 7, grp = lane >> 3;
  const bool live = t < nt;  // rows nt .. nt_pad - 1 of the last tile: a zero activation row
  const float4 *xrow = reinterpret_cast<const float4 *>(X + (live ? t : 0) * nb32 * 32);
  uint2 *scodes = reinterpret_cast<uint2 *>(sstash4);  // 8 bytes (four codes) per lane of a block
  float *sd16 = reinterpret_cast<float *>(sstash4 + nb32 * 4);
  float *sssum = sd16 + nb32;
  float gmax = 0.f;
  for (int64_t base = warp * 16; base < nb32; base += 16 * kQuantWarps) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = base + u * 4 + grp;
      v[u] = c < nb32 && live ? __ldg(xrow + c * 8 + part) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = base + u * 4 + grp;
      float d16f, q[4];
      q8_lane(v[u], d16f, q);
      const float ssum = kQ4 ? q8_ssum(q) : 0.f;
      if (c >= nb32) continue;
      gmax = fmaxf(gmax, kQ4 ? fmaxf(d16f * 127.0f, fabsf(d16f * ssum)) : d16f * 127.0f);
      if (kStash) {
        scodes[c * 8 + part] = make_uint2(q8_h2(q[0], q[1]), q8_h2(q[2], q[3]));
        if (part == 0) {
          sd16[c] = d16f;
          sssum[c] = ssum;
        }
      }
    }
  }
  __shared__ float wmax[kQuantWarps];
#pragma unroll
  for (int m = 16; m; m >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, m));
  if (lane == 0) wmax[warp] = gmax;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kQuantWarps; ++w) gmax = fmaxf(gmax, wmax[w]);
  const int s = split_scale_exp(gmax);
  const float scale = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
  if (tid == 0) invp[t] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  const int64_t nsb = nb32 / 8;
  const int r = static_cast<int>(kPair ? t % tp : t & (kTileM - 1)), h = tp / 2;
  const int64_t tile = kPair ? t / tp : t / kTileM;
  if (kStash) {
    // chunk g: k = 8g .. 8g + 7, block c = g / 4; within its half super-block
    // (sb, half) the chunk sits at K offset kk = 8 * (g % 16)
    const uint32_t row_off = static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128);
    for (int64_t g = tid; g < nb32 * 4; g += 32 * kQuantWarps) {
      const int64_t c = g >> 2;
      const int kk = static_cast<int>(g & 15) * 8;
      const int half = static_cast<int>((c >> 2) & 1);
      uint8_t *blk = aplane + (kPair ? pair_block(tile, c >> 3, half, nsb, kQ4, h) : as_block(tile, c >> 3, half, nsb, kQ4));
      const uint32_t off = kPair ? pair_off(r, kk, kQ4, half, h)
                                 : static_cast<uint32_t>(kk >> 6) * kSplitQuarter + row_off +
                                       ((((kk & 63) >> 3) ^ (r & 7)) << 4);
      const float d16f = sd16[c];
      uint4 hi, lo;
      split_chunk(sstash4[g], d16f * scale, hi, lo);
      *reinterpret_cast<uint4 *>(blk + off) = hi;
      *reinterpret_cast<uint4 *>(blk + (kPair ? pair_kb_bytes(h) : kSplitLo) + off) = lo;
      if (kQ4 && (g & 3) == 0) {
        const float gv = d16f * sssum[c] * scale;  // exact to fp32
        const __half ghi = __float2half_rn(gv);
        const __half glo = __float2half_rn(gv - __half2float(ghi));
        uint8_t *mblk = aplane + (kPair ? pair_block(tile, c >> 3, 1, nsb, true, h) : as_block(tile, c >> 3, 1, nsb, true));
        const int j = 2 * static_cast<int>(c & 7);
        *reinterpret_cast<uint32_t *>(mblk + (kPair ? pair_min_off(r, j, h) : kSplitMin + min_off(r, j))) =
            static_cast<uint32_t>(__half_as_ushort(ghi)) | (static_cast<uint32_t>(__half_as_ushort(glo)) << 16);
      }
    }
  } else {
    for (int64_t base = warp * 16; base < nb32; base += 16 * kQuantWarps) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t c = base + u * 4 + grp;
        v[u] = c < nb32 && live ? __ldg(xrow + c * 8 + part) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t c = base + u * 4 + grp;
        float d16f, q[4];
        q8_lane(v[u], d16f, q);
        const float ssum = kQ4 ? q8_ssum(q) : 0.f;
        if (c < nb32)
          emit_split<kQ4, kPair>(aplane, t, c, nb32, part, make_float2(q[0], q[1]), make_float2(q[2], q[3]), d16f,
                                 static_cast<int>(ssum), scale, tp);
      }
    }
  }
}

// From pad40 q8_0 blocks: one CTA of 128 threads per token.  kPair: the pair
// arm's block layout.
template <bool kQ4, bool kPair = false>
__global__ void __launch_bounds__(128) split_prepass_q_kernel(const uint8_t *__restrict__ Q, int64_t nt,
                                                              int64_t nb32, uint8_t *__restrict__ aplane,
                                                              float *__restrict__ invp, int *__restrict__ cnt,
                                                              int ncnt, int tp) {
  griddep_launch_dependents();
  if (blockIdx.x == 0)  // the GEMM's per-tile piece counters start at zero
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool live = t < nt;  // rows nt .. nt_pad - 1 of the last tile: a zero activation row
  const uint8_t *qrow = Q + (live ? t : 0) * nb32 * 40;
  float gmax = 0.f;
  for (int64_t c = tid; c < nb32 && live; c += 128) {
    const uint8_t *b = qrow + c * 40;
    const float d16f = __half2float(*reinterpret_cast<const __half *>(b));
    gmax = fmaxf(gmax, split_range<kQ4>(d16f, *reinterpret_cast<const int *>(b + 36)));
  }
  __shared__ float wmax[4];
#pragma unroll
  for (int m = 16; m; m >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, m));
  if (lane == 0) wmax[warp] = gmax;
  __syncthreads();
  gmax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  const int s = split_scale_exp(gmax);
  const float scale = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
  if (tid == 0) invp[t] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  const int part = tid & 7;
  for (int64_t c = tid >> 3; c < nb32; c += 16) {
    const uint8_t *b = qrow + c * 40;
    const float d16f = live ? __half2float(*reinterpret_cast<const __half *>(b)) : 0.f;
    const int ssum = live ? *reinterpret_cast<const int *>(b + 36) : 0;
    const uint32_t q4b = live ? *reinterpret_cast<const uint32_t *>(b + 4 + 4 * part) : 0u;
    float2 q01, q23;
    codes_of_word(q4b, q01, q23);
    emit_split<kQ4, kPair>(aplane, t, c, nb32, part, q01, q23, d16f, ssum, scale, tp);
  }
}

// ---------------------------------------------------------------- the GEMM
// acc[h*16 ..] = da * S (first chunk of a super-block) or += da * S, on one
// 32-column half h of a chunk.
__device__ __forceinline__ void fold_half(float2 (&acc)[32], int h, const uint32_t (&r)[32], float da,
                                          bool first) {
  const float2 da2 = make_float2(da, da);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 x = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    acc[h * 16 + j] = first ? __fmul2_rn(da2, x) : __ffma2_rn(da2, x, acc[h * 16 + j]);
  }
}

// Makes the compiler treat r as written here, so code that reads r is not
// moved above this point.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// The work of one CTA as segments (tile, super-blocks [sb0, sb1)); tile =
// token tile + n_tt * weight tile.
// Tile mode: whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// Stream-K mode: the grid is gridDim.x / n_tt groups of n_tt CTAs.  Member m
// of a group takes token tile m, and each group an equal contiguous share of
// the (weight tile, super-block) units, so the CTAs of a group read the same
// weight blocks at the same time.  A tile cut between groups is finished by
// the CTA that holds its first super-block (its owner).
struct Work {
  int64_t u, u_end;  // stream-K: current and end unit of the group
  int tile;          // tile mode: next tile
  int member;        // stream-K: token tile
  bool sk;
};
__device__ __forceinline__ int64_t sk_begin(int64_t gunits, int group, int groups) {
  return gunits * group / groups;
}
__device__ __forceinline__ Work work_begin(bool sk, int n_tt, int n_ot, int64_t nsb) {
  Work w;
  w.sk = sk;
  const int groups = static_cast<int>(gridDim.x) / n_tt, g = static_cast<int>(blockIdx.x) / n_tt;
  const int64_t gunits = static_cast<int64_t>(n_ot) * nsb;
  w.u = sk_begin(gunits, g, groups);
  w.u_end = sk_begin(gunits, g + 1, groups);
  w.member = static_cast<int>(blockIdx.x) % n_tt;
  w.tile = blockIdx.x;
  return w;
}
__device__ __forceinline__ bool work_next(Work &w, int n_tiles, int n_tt, int64_t nsb, int &tile, int64_t &sb0,
                                          int64_t &sb1) {
  if (w.sk) {
    if (w.u >= w.u_end) return false;
    tile = w.member + n_tt * static_cast<int>(w.u / nsb);
    sb0 = w.u % nsb;
    sb1 = min(nsb, sb0 + (w.u_end - w.u));
    w.u += sb1 - sb0;
    return true;
  }
  if (w.tile >= n_tiles) return false;
  tile = w.tile;
  sb0 = 0;
  sb1 = nsb;
  w.tile += gridDim.x;
  return true;
}

__device__ __forceinline__ void st_global_v8(float *p, float2 a, float2 b, float2 c, float2 d) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(a.x), "f"(a.y),
               "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y)
               : "memory");
}

// 64 outputs of one thread (row t, columns o0 .. o0 + 63; y[OFF ..]) times inv.
template <int OFF = 0, int N = 32>
__device__ __forceinline__ void store_y_row(float *__restrict__ Y, int64_t t, int64_t od, int64_t o0,
                                            const float2 (&y)[N], float inv) {
  static_assert(OFF + 32 <= N, "64 outputs");
  const float2 inv2 = make_float2(inv, inv);
  float *yrow = Y + t * od + o0;
  if ((od & 7) == 0 && (reinterpret_cast<uintptr_t>(Y) & 31) == 0) {
    // 32-byte stores: each row segment of a warp's store is a whole sector
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      if (o0 + 2 * i < od) {
        const float2 a = __fmul2_rn(y[OFF + i], inv2), b = __fmul2_rn(y[OFF + i + 1], inv2);
        const float2 c = __fmul2_rn(y[OFF + i + 2], inv2), d = __fmul2_rn(y[OFF + i + 3], inv2);
        st_global_v8(yrow + 2 * i, a, b, c, d);
      }
    }
  } else if ((od & 3) == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      if (o0 + 2 * i < od) {
        const float2 a = __fmul2_rn(y[OFF + i], inv2), b = __fmul2_rn(y[OFF + i + 1], inv2);
        *reinterpret_cast<float4 *>(yrow + 2 * i) = make_float4(a.x, a.y, b.x, b.y);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float2 a = __fmul2_rn(y[OFF + i], inv2);
      if (o0 + 2 * i < od) yrow[2 * i] = a.x;
      if (o0 + 2 * i + 1 < od) yrow[2 * i + 1] = a.y;
    }
  }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// 32 fp32 values of a TMEM row half to dump[at .. at + 31] (16-byte stores).
__device__ __forceinline__ void dump_half(float *__restrict__ dump, int64_t at, const uint32_t (&r)[32]) {
  float4 *p = reinterpret_cast<float4 *>(dump + at);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    p[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                       __uint_as_float(r[4 * i + 3]));
}

// kDump (a test hook, whole tiles only): each chunk's raw TMEM partial -- the
// exact integer sum of qs times the folded operand -- is also stored, fp32,
// to dump[(t * nb32 + chunk) * od_pad + o].
template <bool kQ4, bool kSK, bool kRaw, bool kB0, bool kDump = false>
__global__ void __launch_bounds__(Shape<kRaw>::kThreads, 1)
    mmq_gemm_kernel(const uint8_t *__restrict__ aplane, const uint8_t *__restrict__ bplane,
                    const uint8_t *__restrict__ rawplane, const uint8_t *__restrict__ b0plane,
                    const uint8_t *__restrict__ bscale, const float *__restrict__ dap,
                    const float *__restrict__ invp, int64_t nt, int64_t od, int64_t nb32, int n_tt,
                    int n_ot, float *__restrict__ Y, WaitCtl wctl, float4 *__restrict__ ws,
                    uint64_t *__restrict__ flags, float *__restrict__ dump) {
  static_assert(!kB0 || (!kQ4 && !kRaw), "the B0 plane is q6_K's, read from the registered planes");
  static_assert(!kDump || (!kSK && !kRaw), "the partial dump runs whole tiles from the registered planes");
  using L = Smem<kQ4, kRaw, kB0>;
  using S = Shape<kRaw, kB0>;
  constexpr int STAGES = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nsb = nb32 / 8;
  const int n_tiles = n_tt * n_ot;

  const uint32_t bar = base + L::kBar;
  auto full = [&](int s) { return bar + 8u * s; };
  auto empty = [&](int s) { return bar + 8u * (STAGES + s); };
  auto rfull = [&](uint32_t i) { return bar + 8u * (2 * STAGES + i); };
  auto rempty = [&](uint32_t i) { return bar + 8u * (2 * STAGES + SLOTS + i); };
  auto sfull = [&](int e) { return bar + 8u * (2 * STAGES + 2 * SLOTS + e); };
  auto sempty = [&](int e) { return bar + 8u * (2 * STAGES + 2 * SLOTS + SRING + e); };
  auto conv = [&](int s) { return bar + 8u * (2 * STAGES + 2 * SLOTS + 2 * SRING + s); };
  auto rawfull = [&](int e) { return bar + 8u * (3 * STAGES + 2 * SLOTS + 2 * SRING + e); };
  auto rawempty = [&](int e) { return bar + 8u * (3 * STAGES + 2 * SLOTS + 2 * SRING + RRING + e); };
  const uint32_t done = bar + 8u * (3 * STAGES + 2 * SLOTS + 2 * SRING + 2 * RRING);
  auto a_smem = [&](int s) { return base + s * L::kStage; };
  auto b_smem = [&](int s) { return base + s * L::kStage + L::kA; };
  auto s_smem = [&](int e) { return base + L::kScaleRing + e * L::kScale; };
  auto raw_smem = [&](int e) { return base + L::kRawRing + e * L::kRaw_; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kB0 ? 1 : ISSUERS);  // one commit per issuer (kB0: its one issuer) frees a stage
    }
    for (uint32_t i = 0; i < SLOTS; ++i) {
      mbar_init(rfull(i), 1);
      mbar_init(rempty(i), EPI_WARPS);
    }
    for (int e = 0; e < SRING; ++e) {
      mbar_init(sfull(e), 1);
      mbar_init(sempty(e), EPI_WARPS);
    }
    if (kRaw) {
      for (int s = 0; s < STAGES; ++s) mbar_init(conv(s), CONVERTERS);
      for (int e = 0; e < RRING; ++e) {
        mbar_init(rawfull(e), 1);
        mbar_init(rawempty(e), CONVERTERS);
      }
    }
    mbar_init(done, ISSUERS);
    fence_mbar_init();
  }
  if (warp == ISSUER_WARP) {
    tmem_alloc(base + L::kSlot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + L::kSlot);
  // The activation plane, da' and 2^-s are written by the kernel before this
  // one, which may still be running (programmatic launch): the producer and
  // the epilogue wait for it before their first read of them; the weight side
  // does not depend on it.
  if (warp >= PRODUCER_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(S::kRegsCtl));
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (warp-uniform control flow); lane 0 copies
    // the activation block, lane 1 the weight block, lane 2 the super-block's
    // scale block into the scale ring.
    griddep_wait();
    uint32_t ks = 0, ns = 0, issued = 0, s_issued = 0, r_issued = 0;
    bool ok = true;
    Work wk = work_begin(kSK, n_tt, n_ot, nsb);
    int tile;
    int64_t sb0, sb1;
    while (ok && work_next(wk, n_tiles, n_tt, nsb, tile, sb0, sb1)) {
      const int tt = tile % n_tt, ot = tile / n_tt;
      for (int64_t sb = sb0; sb < sb1 && ok; ++sb, ++ns) {
        const int e = static_cast<int>(ns % SRING);
        ok = __all_sync(0xffffffffu, mbar_wait(sempty(e), ((ns / SRING) & 1) ^ 1, wctl));
        if (!ok) break;
        if (lane == 2) {
          mbar_arrive_expect_tx(sfull(e), L::kScale);
          bulk_load(s_smem(e), bscale + b_scale_block(ot, sb, nsb, kQ4), L::kScale, sfull(e));
        }
        __syncwarp();
        s_issued = ns + 1;
        if constexpr (kB0) {  // four 64-K stages per super-block: A, B1 and B0 K-blocks
          for (int q = 0; q < 4 && ok; ++q, ++ks) {
            const int half = q >> 1, kb = q & 1;
            const int s = static_cast<int>(ks % STAGES);
            ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ((ks / STAGES) & 1) ^ 1, wctl));
            if (!ok) break;
            const uint32_t ko = static_cast<uint32_t>(kb) * L::kKB;
            if (lane == 0) {
              mbar_arrive_expect_tx(full(s), 3 * L::kKB);
              bulk_load(a_smem(s), aplane + a_block(tt, sb, half, nsb, false) + ko, L::kKB, full(s));
            } else if (lane == 1) {
              bulk_load(b_smem(s), bplane + b_block(ot, sb, half, nsb, false) + ko, L::kKB, full(s));
            } else if (lane == 3) {
              bulk_load(b_smem(s) + L::kB0Off, b0plane + b_block(ot, sb, half, nsb, false) + ko, L::kKB, full(s));
            }
            __syncwarp();
            issued = ks + 1;
          }
        } else {
          for (int half = 0; half < 2; ++half, ++ks) {
            if (kRaw) {  // the raw weight block first: its ring runs ahead of the stages
              const int re = static_cast<int>(ks % RRING);
              ok = __all_sync(0xffffffffu, mbar_wait(rawempty(re), ((ks / RRING) & 1) ^ 1, wctl));
              if (!ok) break;
              if (lane == 3) {
                mbar_arrive_expect_tx(rawfull(re), raw_block_bytes(kQ4));
                bulk_load(raw_smem(re), rawplane + raw_block(ot, sb, half, nsb, kQ4), raw_block_bytes(kQ4),
                          rawfull(re));
              }
              __syncwarp();
              r_issued = ks + 1;
            }
            const int s = static_cast<int>(ks % STAGES);
            ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ((ks / STAGES) & 1) ^ 1, wctl));
            if (!ok) break;
            const uint32_t ab = half ? a_odd_bytes(kQ4) : a_even_bytes();
            // raw arm: only the q4_K min image of the weight block is copied
            const uint32_t bb = kRaw ? ((kQ4 && half) ? kMinBytes : 0) : (half ? b_odd_bytes(kQ4) : b_even_bytes());
            if (lane == 0) {
              mbar_arrive_expect_tx(full(s), ab + bb);
              bulk_load(a_smem(s), aplane + a_block(tt, sb, half, nsb, kQ4), ab, full(s));
            } else if (lane == 1 && bb) {
              if (kRaw)
                bulk_load(b_smem(s) + kBMin, bplane + b_block(ot, sb, half, nsb, kQ4) + kBMin, bb, full(s));
              else
                bulk_load(b_smem(s), bplane + b_block(ot, sb, half, nsb, kQ4), bb, full(s));
            }
            __syncwarp();
            issued = ks + 1;
          }
        }
      }
    }
    if (!ok) {  // drain this CTA's copies still in flight
      for (uint32_t k = issued > STAGES ? issued - STAGES : 0; k < issued; ++k)
        mbar_wait(full(k % STAGES), (k / STAGES) & 1, wctl, false);
      for (uint32_t k = s_issued > SRING ? s_issued - SRING : 0; k < s_issued; ++k)
        mbar_wait(sfull(k % SRING), (k / SRING) & 1, wctl, false);
      for (uint32_t k = r_issued > RRING ? r_issued - RRING : 0; k < r_issued; ++k)
        mbar_wait(rawfull(k % RRING), (k / RRING) & 1, wctl, false);
    }
  } else if (kRaw && warp >= CONVERTER_WARP) {
    // ------------------------------------------------------------ converters
    // Raw arm: per stage, unpack the raw weight block into the stage's fp16
    // operand image once both the block has landed and the stage is free.
    const int r = threadIdx.x - CONVERTER_WARP * 32;  // row of the weight tile
    uint32_t ks = 0;
    bool ok = true;
    Work wk = work_begin(kSK, n_tt, n_ot, nsb);
    int tile;
    int64_t sb0, sb1;
    while (ok && work_next(wk, n_tiles, n_tt, nsb, tile, sb0, sb1)) {
      for (int64_t sb = sb0; sb < sb1 && ok; ++sb) {
        for (int half = 0; half < 2 && ok; ++half, ++ks) {
          const int re = static_cast<int>(ks % RRING), s = static_cast<int>(ks % STAGES);
          ok = __all_sync(0xffffffffu, mbar_wait(rawfull(re), (ks / RRING) & 1, wctl));
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ((ks / STAGES) & 1) ^ 1, wctl));
          if (!ok) break;
          unpack_stage<kQ4>(smem + (raw_smem(re) - base), smem + (b_smem(s) - base), r);
          // generic-proxy writes of the operand image, read next by the
          // tensor core (async proxy); the raw block was read the same way
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(conv(s));
            mbar_arrive(rawempty(re));
          }
        }
      }
    }
  } else if (warp < ISSUER_WARP + ISSUERS) {
    // ------------------------------------------------------------ UMMA issuers
    // Two warps issue, each from one elected lane of a warp-uniform loop: of
    // the eight 32-K chunks of a super-block, issuer 0 takes 0, 2, 4, 6 (and
    // the q4_K min term after chunk 7) and issuer 1 takes 1, 3, 5, 7.  An
    // issuer's items alternate between its two TMEM slots; each is committed
    // on its slot's barrier.  The tensor pipe queues little work, so while
    // one issuer waits for a slot or a stage the other keeps it fed.
    const int iw = warp - ISSUER_WARP;
    uint32_t elected;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(elected));
    constexpr uint32_t idesc = idesc_f16_f32(kTileM, kTileN);
    constexpr uint64_t kStageDesc = L::kStage >> 4;  // descriptor address field step per stage
    const uint64_t a0 = sdesc_kmajor_sw128(a_smem(0)), b0 = sdesc_kmajor_sw128(b_smem(0));
    const uint64_t am0 = sdesc_kmajor_sw32(a_smem(0) + kAMin), bm0 = sdesc_kmajor_sw32(b_smem(0) + kBMin);
    uint32_t ks = 0, j = 0;  // stages consumed, items issued
    bool ok = true;
    // one item: wait for the slot, 1 or 2 UMMAs (kB0: then the same A against
    // the B0 image, so the chunk's partial sums B1 + B0), commit on the slot.
    // Every partial of a chunk stays an integer below 32 * 127 * 4096 < 2^24.
    auto item = [&](uint64_t ad, uint64_t bd, bool two) {
      const uint32_t slot = 2 * iw + (j & 1);
      const bool got = __all_sync(0xffffffffu, mbar_wait(rempty(slot), ((j >> 1) & 1) ^ 1, wctl));
      if (got) {
        tc_fence_after();
        if (elected) {
          const uint32_t d = tbase + slot * kTileN;
          umma_f16(d, ad, bd, idesc, 0);
          if (two) umma_f16(d, ad + 2, bd + 2, idesc, 1);
          if (kB0 && two) {
            constexpr uint64_t kB0Desc = L::kB0Off >> 4;
            umma_f16(d, ad, bd + kB0Desc, idesc, 1);
            umma_f16(d, ad + 2, bd + kB0Desc + 2, idesc, 1);
          }
          umma_commit(rfull(slot));
        }
        __syncwarp();
        ++j;
      }
      return got;
    };
    Work wk = work_begin(kSK, n_tt, n_ot, nsb);
    int tile;
    int64_t sb0, sb1;
    while (ok && work_next(wk, n_tiles, n_tt, nsb, tile, sb0, sb1)) {
      for (int64_t sb = sb0; sb < sb1 && ok; ++sb) {
        if constexpr (kB0) {
          // 64-K stage q = (half, kb) holds chunks 4*half + 2*kb + {0, 1}: issuer
          // kb takes it, so issuer 0 still gets chunks 0, 1, 4, 5 and issuer 1
          // chunks 2, 3, 6, 7 (the order the epilogue reads the slots in)
          for (int q = 0; q < 4 && ok; ++q, ++ks) {
            if ((q & 1) != iw) continue;
            const int s = static_cast<int>(ks % STAGES);
            ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
            if (!ok) break;
            tc_fence_after();
            const uint64_t as = a0 + s * kStageDesc, bs = b0 + s * kStageDesc;
#pragma unroll
            for (int c = 0; c < 2 && ok; ++c) ok = item(as + c * (64 >> 4), bs + c * (64 >> 4), true);
            if (!ok) break;
            if (elected) umma_commit(empty(s));
            __syncwarp();
          }
        } else {
          for (int half = 0; half < 2 && ok; ++half, ++ks) {
            const int s = static_cast<int>(ks % STAGES);
            ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
            if (ok && kRaw) ok = __all_sync(0xffffffffu, mbar_wait(conv(s), (ks / STAGES) & 1, wctl));
            if (!ok) break;
            tc_fence_after();
            const uint64_t as = a0 + s * kStageDesc, bs = b0 + s * kStageDesc;
  #pragma unroll
            for (int q = 0; q < 2 && ok; ++q) {
              const int lc = 2 * iw + q;  // chunk in the stage: K = 32*lc .. 32*lc+31
              const uint64_t off = (lc >> 1) * (16384 >> 4) + (lc & 1) * (64 >> 4);
              ok = item(as + off, bs + off, true);
            }
            if (ok && kQ4 && half == 1 && iw == 0)
              ok = item(am0 + s * kStageDesc, bm0 + s * kStageDesc, false);
            if (!ok) break;
            if (elected) umma_commit(empty(s));
            __syncwarp();
          }
        }
      }
    }
    if (elected) umma_commit(done);  // all UMMAs of both issuers have finished once `done` flips
    __syncwarp();
    mbar_wait(done, 0, wctl, false);
  } else if (warp == PRODUCER_WARP + 3 && lane == 0) {
    // ------------------------------------------------------------ L2 prefetch
    // The first two super-blocks of this CTA's weight (and scale) blocks,
    // pulled into L2 off the producer's path.
    Work wk = work_begin(kSK, n_tt, n_ot, nsb);
    int tile;
    int64_t sb0, sb1;
    if (work_next(wk, n_tiles, n_tt, nsb, tile, sb0, sb1)) {
      const int ot = tile / n_tt;
      for (int64_t sb = sb0; sb < sb1 && sb < sb0 + 2; ++sb) {
        bulk_prefetch_l2(bscale + b_scale_block(ot, sb, nsb, kQ4), L::kScale);
        for (int half = 0; half < 2; ++half) {
          if (kRaw)
            bulk_prefetch_l2(rawplane + raw_block(ot, sb, half, nsb, kQ4), raw_block_bytes(kQ4));
          else
            bulk_prefetch_l2(bplane + b_block(ot, sb, half, nsb, kQ4), half ? b_odd_bytes(kQ4) : b_even_bytes());
          if (kB0) bulk_prefetch_l2(b0plane + b_block(ot, sb, half, nsb, false), kOperandBytes);
        }
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(S::kRegsEpi));
    // ------------------------------------------------------------ epilogue
    // Software-pipelined over 32-column halves: while the packed FMAs of one
    // half run, the TMEM load of the next half and the barrier test of the
    // next item are in flight.  A slot is handed back as soon as both halves
    // of its chunk are in registers.
    const int quad = warp & 3;
    const int chalf = warp >> 2;  // column half 0 / 1
    const int row = quad * 32 + lane;
    const uint32_t taddr = tbase + (static_cast<uint32_t>(quad * 32) << 16) + chalf * 64;
    uint32_t jj[ISSUERS] = {0, 0}, ns = 0;  // items taken from each issuer, scale entries used
    bool ok = true;
    // slot and phase of the next item of issuer iw
    auto next_item = [&](int iw, uint32_t &slot, uint32_t &par) {
      slot = 2 * iw + (jj[iw] & 1);
      par = (jj[iw] >> 1) & 1;
      ++jj[iw];
    };
    auto wait_item = [&](uint32_t slot, uint32_t par, bool ready) {
      const bool got = __all_sync(0xffffffffu, ready || mbar_wait(rfull(slot), par, wctl));
      if (got) tc_fence_after();
      return got;
    };
    auto give = [&](uint32_t slot) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty(slot));
    };
    Work wk = work_begin(kSK, n_tt, n_ot, nsb);
    int tile;
    int64_t sb0, sb1;
    griddep_wait();  // da' and 2^-s come from the kernel before this one
    while (ok && work_next(wk, n_tiles, n_tt, nsb, tile, sb0, sb1)) {
      const int tt = tile % n_tt, ot = tile / n_tt;
      const int64_t t = static_cast<int64_t>(tt) * kTileM + row;  // < nt_pad: planes are padded
      const int64_t o0 = static_cast<int64_t>(ot) * kTileN + chalf * 64;
      float2 y[32], acc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = make_float2(0.f, 0.f);
      const float4 *darow = reinterpret_cast<const float4 *>(dap + t * nb32);
      // da' of the next super-block
      float4 nx0 = __ldg(darow + 2 * sb0), nx1 = __ldg(darow + 2 * sb0 + 1);
      for (int64_t sb = sb0; sb < sb1 && ok; ++sb) {
        const float das[8] = {nx0.x, nx0.y, nx0.z, nx0.w, nx1.x, nx1.y, nx1.z, nx1.w};
        if (sb + 1 < sb1) {
          nx0 = __ldg(darow + 2 * sb + 2);
          nx1 = __ldg(darow + 2 * sb + 3);
        }
        uint32_t r0[32], r1[32];
        // Chunks come in pairs (2p, 2p+1), both from issuer p & 1 and
        // committed in issue order, so the barrier of a pair's second chunk
        // covers the pair: one wait per two chunks.
        const int e = static_cast<int>(ns % SRING);
        const bool s_ready = mbar_test_wait(sfull(e), (ns / SRING) & 1);  // early probe of the scales
        uint32_t slot, slot_b, par, par_b;
        next_item(0, slot, par);
        next_item(0, slot_b, par_b);
        if (!(ok = wait_item(slot_b, par_b, false))) break;
        tmem_ld_32x32b_x32(taddr + slot * kTileN, r0);
        tmem_wait_ld(r0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          // second half of chunk c; in a pair's second chunk, an early test
          // of the next pair
          tmem_ld_32x32b_x32(taddr + slot * kTileN + 32, r1);
          uint32_t na = 0, nb = 0, npb = 0;
          bool ready = true;
          if ((c & 1) && c < 7) {
            const int niw = ((c + 1) >> 1) & 1;
            next_item(niw, na, par);
            next_item(niw, nb, npb);
            ready = mbar_test_wait(rfull(nb), npb);
          }
          reg_fence(r0);
          if constexpr (kDump) dump_half(dump, (t * nb32 + sb * 8 + c) * (n_ot * kTileN) + o0, r0);
          fold_half(acc, 0, r0, das[c], c == 0);
          tmem_wait_ld(r1);
          give(slot);
          if (c < 7) {
            if (c & 1) {
              if (!(ok = wait_item(nb, npb, ready))) break;
              slot = na;
              slot_b = nb;
            } else {
              slot = slot_b;
            }
            tmem_ld_32x32b_x32(taddr + slot * kTileN, r0);
          }
          if constexpr (kDump) dump_half(dump, (t * nb32 + sb * 8 + c) * (n_ot * kTileN) + o0 + 32, r1);
          fold_half(acc, 1, r1, das[c], c == 0);
          if (c < 7) tmem_wait_ld(r0);
        }
        if (!ok) break;
        // super-block end: y += d * acc  (- dmin * MIN for q4_K)
        ok = __all_sync(0xffffffffu, s_ready || mbar_wait(sfull(e), (ns / SRING) & 1, wctl));
        if (!ok) break;
        const uint8_t *sblk = smem + (s_smem(e) - base);
        const float4 *d4 = reinterpret_cast<const float4 *>(sblk) + chalf * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 d = d4[i];
          y[2 * i] = __ffma2_rn(make_float2(d.x, d.y), acc[2 * i], y[2 * i]);
          y[2 * i + 1] = __ffma2_rn(make_float2(d.z, d.w), acc[2 * i + 1], y[2 * i + 1]);
        }
        if (kQ4) {
          // the min-term item needs a wait of its own: its slot is the one
          // chunk 4 held, so it cannot be issued before chunk 4 is loaded
          next_item(0, slot, par);
          if (!(ok = wait_item(slot, par, false))) break;
          tmem_ld_32x32b_x32(taddr + slot * kTileN, r0);
          tmem_ld_32x32b_x32(taddr + slot * kTileN + 32, r1);
          tmem_wait_ld(r0);
          reg_fence(r1);
          give(slot);
          const float4 *m4 = reinterpret_cast<const float4 *>(sblk + kSDmin) + chalf * 16;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 dm = m4[i];
            const uint32_t(&rr)[32] = i < 8 ? r0 : r1;
            const int q = (i & 7) * 4;
            y[2 * i] = __ffma2_rn(make_float2(-dm.x, -dm.y),
                                  make_float2(__uint_as_float(rr[q]), __uint_as_float(rr[q + 1])), y[2 * i]);
            y[2 * i + 1] = __ffma2_rn(make_float2(-dm.z, -dm.w),
                                      make_float2(__uint_as_float(rr[q + 2]), __uint_as_float(rr[q + 3])),
                                      y[2 * i + 1]);
          }
        }
        // the scale block was read through the generic proxy; order those
        // reads before the bulk copy (async proxy) that refills the entry
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(sempty(e));
        ++ns;
      }
      if (!ok) break;
      if (kSK && (sb0 != 0 || sb1 != nsb)) {
        // hand-off tag of this launch: the flags are cleared by the kernel
        // before this one; the tag pairs the epoch with its complement
        const uint64_t tag = (static_cast<uint64_t>(wctl.epoch) << 32) | static_cast<uint32_t>(~wctl.epoch);
        // A tile cut between CTAs.  Its owner is the CTA holding its first
        // super-block, where that CTA's range ends; the others hold the rest
        // at the start of their ranges, so they publish their partial sums
        // first thing and the owner, finishing its range, adds them.  Layout
        // of a partial: 16 float4 per thread at
        // ws[((cta * 8 + warp) * 16 + i) * 32 + lane].
        if (sb0 != 0) {  // not the owner: publish (a CTA's first segment only)
          float4 *dst = ws + static_cast<int64_t>(blockIdx.x * 8 + warp) * 16 * 32 + lane;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            __stcg(dst + i * 32, make_float4(y[2 * i].x, y[2 * i].y, y[2 * i + 1].x, y[2 * i + 1].y));
          epi_bar();
          if (threadIdx.x == 0) {
            __threadfence();
            asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(flags + blockIdx.x), "l"(tag)
                         : "memory");
          }
          continue;
        }
        // owner: add the partials of the same member of the following groups
        // that reach into this tile, in group order (deterministic results)
        const int groups = static_cast<int>(gridDim.x) / n_tt;
        const int64_t gunits = static_cast<int64_t>(n_ot) * nsb;
        const int64_t tile_end = static_cast<int64_t>(ot + 1) * nsb;
        for (int gg = static_cast<int>(blockIdx.x) / n_tt + 1;
             gg < groups && sk_begin(gunits, gg, groups) < tile_end && ok; ++gg) {
          const int j = gg * n_tt + wk.member;
          if (threadIdx.x == 0) {
            const uint64_t t0 = globaltimer_ns();
            uint64_t v = 0;
            for (uint32_t it = 0;; ++it) {
              asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(flags + j) : "memory");
              if (v == tag) break;
              if ((it & 63u) == 63u &&
                  (*reinterpret_cast<volatile unsigned *>(wctl.abort_epoch) == wctl.epoch ||
                   globaltimer_ns() - t0 > wctl.limit_ns)) {
                record_timeout(wctl);
                break;
              }
              __nanosleep(64);
            }
          }
          epi_bar();
          ok = *reinterpret_cast<volatile unsigned *>(wctl.abort_epoch) != wctl.epoch;
          const float4 *src = ws + static_cast<int64_t>(j * 8 + warp) * 16 * 32 + lane;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 v = __ldcg(src + i * 32);
            y[2 * i] = __fadd2_rn(y[2 * i], make_float2(v.x, v.y));
            y[2 * i + 1] = __fadd2_rn(y[2 * i + 1], make_float2(v.z, v.w));
          }
        }
        if (!ok) break;
      }
      if (t < nt) store_y_row(Y, t, od, o0, y, __ldg(invp + t));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == ISSUER_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- the split arm's GEMM
// Same operands and roles as mmq_gemm_kernel, with the activation scale
// folded into A (hi + lo images, tiling.h): per 32-K chunk four UMMAs (hi and
// lo, two K halves each) accumulate into one TMEM region for the whole
// super-block, so the epilogue runs once per super-block:
//   y[t][o] += d[o][sb] * ACC[t][o][sb]  -  dmin[o][sb] * MIN[t][o][sb]
// kWide: output tiles of 128 tokens x 256 weight rows (two weight tiles side
// by side, one N = 256 UMMA), so each activation K-block feeds twice the
// MACs; otherwise 128 x 128.  Regions of kN columns, NR accumulators then
// (q4_K, 128 wide) NR min-term regions: 128 wide q6_K four accumulators, 128
// wide q4_K two of each.  kWide tiles have two regions of 256 columns; a q4_K
// min term then goes into the region its super-block's accumulator just left
// (kShared): the issuer sends the K = 16 min UMMA of super-block n into region
// n % 2 once the epilogue has read the accumulator there, so both regions stay
// double-buffered; its operands wait in a ring of their own until then.
// Stages of 64 K; one issuer; whole tiles per CTA.
// The split arm's register split: its epilogue holds no per-chunk pipeline,
// its producer and issuer more addresses (kShared: the min ring's too).
struct SplitShape {
  static constexpr int kThreads = 384;
  static constexpr int kRegsLaunch = 168;
};
template <bool kShared>
struct SplitRegs {
  static constexpr int kEpi = kShared ? 192 : 208;
  static constexpr int kCtl = kShared ? 120 : 88;
  static_assert(256 * kEpi + (SplitShape::kThreads - 256) * kCtl == SplitShape::kThreads * SplitShape::kRegsLaunch,
                "the register split must add up to what the launch holds");
};

// kB0 (q6_K with |sc| > 64): after the kN / 128 B1 K-blocks of a stage come
// as many B0 K-blocks.
// kSmall (pieces of one token tile of at most kSmallRows tokens): a stage's
// activation region holds only those rows -- the hi K-block's, the lo
// K-block's, (q4_K) the min image's -- so the ring holds twice as many stages;
// the UMMA still reads 128 rows of A from the region's start, the rows beyond
// it (the lo image, the weights) feeding output rows that are never stored.
template <bool kQ4, bool kWide, bool kB0 = false, bool kSmall = false>
struct SplitSmem {
  static constexpr bool kShared = kQ4 && kWide;  // min terms share the accumulator regions
  static constexpr int kN = kWide ? 256 : 128;
  static constexpr int kBK = kTileN * 64 * 2;  // one weight K-block of one tile: 16384
  static constexpr int kSmallRows = 32;
  // A region: hi K-block, lo K-block at kALo, (q4_K) min image at kAMin, kMinA bytes of it copied
  static constexpr int kALo = kSmall ? kSmallRows * 128 : kSplitLo;
  static constexpr int kAMin = kSmall ? 2 * kSmallRows * 128 : kSplitQuarter;
  static constexpr int kMinA = kQ4 && !kShared ? (kSmall ? kSmallRows * 32 : kMinBytes) : 0;
  static constexpr int kMinB = kQ4 && !kShared ? kMinBytes * (kN / 128) : 0;
  static constexpr int kA = ((kAMin + kMinA + 1023) / 1024) * 1024;
  static constexpr int kB = ((kBK * (kN / 128) * (kB0 ? 2 : 1) + kMinB + 1023) / 1024) * 1024;
  static constexpr int kStage = kA + kB;
  static constexpr int kStages = kSmall ? (8 * kStage <= 210 * 1024 ? 8 : 210 * 1024 / kStage)
                                        : kStage * 4 <= 200 * 1024 ? 4 : kStage * 3 <= 200 * 1024 ? 3 : 2;
  static_assert(!kSmall || (!kWide && !kB0), "small activation regions: 128-row one-plane tiles");
  // (kSmall) a UMMA's 128 rows of A from any of the region's images stay inside the stage
  static_assert(!kSmall || kAMin + kMinBytes <= kStage, "A reads inside the stage");
  static_assert(!kSmall || kALo + kOperandBytes / 2 <= kStage, "A reads inside the stage");
  // kShared: min operand ring, entry = A min image then kN / 128 B min images
  static constexpr int kMR = kShared ? 2 : 0;
  static constexpr int kMinEntry = kMinBytes * (1 + kN / 128);
  static constexpr int kMinRing = kStages * kStage;
  static constexpr int kScale = scale_block_bytes(kQ4) * (kN / 128);
  static constexpr int kScaleRing = kMinRing + kMR * kMinEntry;
  static constexpr int kRegions = kWide ? 2 : (kQ4 ? 2 : 4);
  static constexpr int kBar = kScaleRing + SRING * kScale;
  // full, empty per stage; rfull, rempty per region; sfull, sempty per scale
  // entry; (kShared) mfull, mempty per region, mrfull, mrempty per min entry; done
  static constexpr int kNumBars = 2 * kStages + 2 * kRegions + 2 * SRING + (kShared ? 2 * kRegions + 2 * kMR : 0) + 1;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kSlot + 16 + 1024;
  static_assert(kA % 1024 == 0 && kStage % 1024 == 0 && kMinEntry % 1024 == 0,
                "stage and min buffers must keep 1 KB alignment");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(kRegions * kN * (kQ4 && !kShared ? 2 : 1) <= TMEM_COLS, "TMEM columns");
};

// y[c / 2] += s[c] * T[lane][ta + c] for this thread's CW columns c of a TMEM
// region (s negated for kNeg), kG = 32 or 64 columns per TMEM wait (32 holds
// fewer registers, for the variant whose epilogue has 192).
template <int CW, bool kNeg, int kG>
__device__ __forceinline__ void fold_region(uint32_t ta, const float4 *s4, float2 (&y)[CW / 2]) {
  static_assert(kG == 32 || kG == 64, "32 or 64 columns per wait");
#pragma unroll
  for (int g = 0; g < CW / kG; ++g) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(ta + g * kG, r0);
    if (kG == 64) tmem_ld_32x32b_x32(ta + g * kG + 32, r1);
    tmem_wait_ld(r0);
    if (kG == 64) reg_fence(r1);
#pragma unroll
    for (int i = 0; i < kG / 4; ++i) {
      float4 d = s4[g * (kG / 4) + i];
      if (kNeg) d = make_float4(-d.x, -d.y, -d.z, -d.w);
      const uint32_t(&rr)[32] = i < 8 ? r0 : r1;
      const int q = (i & 7) * 4;
      float2 &y0 = y[g * (kG / 2) + 2 * i], &y1 = y[g * (kG / 2) + 2 * i + 1];
      y0 = __ffma2_rn(make_float2(d.x, d.y), make_float2(__uint_as_float(rr[q]), __uint_as_float(rr[q + 1])), y0);
      y1 = __ffma2_rn(make_float2(d.z, d.w), make_float2(__uint_as_float(rr[q + 2]), __uint_as_float(rr[q + 3])), y1);
    }
  }
}

// kKP (one-plane tiles): tiles n_full .. n_tiles-1 -- all of them when the
// tiles fill at most half the SMs, else those of the last, partly filled wave
// -- have their super-blocks cut into n_kp contiguous pieces, one unit of
// work each, after the n_full whole tiles; a CTA takes units blockIdx.x,
// blockIdx.x + gridDim.x, ...  A piece stores its scaled partial sums of the
// token rows below nt to its slot of `part` (64 KB per 128 columns); the last
// CTA of a tile to finish (a counter per pieced tile, zeroed by the prepass)
// adds the tile's pieces in piece order and stores Y, so the sum is the same
// whichever CTA finishes last.  Activation K-blocks are copied only up to the
// tile's last token row (rounded up to 8): rows beyond it feed output rows
// that are never stored.
template <bool kQ4, bool kWide, bool kB0, bool kKP = false, bool kSmall = false>
__global__ void __launch_bounds__(SplitShape::kThreads, 1)
    mmq_gemm_split_kernel(const uint8_t *__restrict__ aplane, const uint8_t *__restrict__ bplane,
                          const uint8_t *__restrict__ bscale, const float *__restrict__ invp, int64_t nt,
                          int64_t od, int64_t nb32, int n_tt, int n_ot, float *__restrict__ Y, WaitCtl wctl,
                          const uint8_t *__restrict__ b0plane, int n_kp, int n_full, float *__restrict__ part,
                          int *__restrict__ cnt) {
  static_assert(!kB0 || !kQ4, "the B0 plane is q6_K's");
  static_assert(!kKP || !kB0, "pieces of one-plane tiles");
  static_assert(!kSmall || kKP, "small activation regions: pieces of one token tile");
  using L = SplitSmem<kQ4, kWide, kB0, kSmall>;
  using S = SplitShape;
  constexpr int STAGES = L::kStages, NR = L::kRegions, NW = L::kN / 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nsb = nb32 / 8;
  const int n_og = (n_ot + NW - 1) / NW;  // groups of NW weight tiles
  const int n_tiles = n_tt * n_og;
  // weight tile w of group og (the last group of an odd n_ot repeats its tile)
  auto wtile = [&](int og, int w) { return min(og * NW + w, n_ot - 1); };
  // units of work: whole tiles, then (kKP) pieces (tile, k) of super-blocks
  const int kp = kKP ? n_kp : 1;
  const int nfull = kKP ? n_full : n_tiles;
  const int n_units = nfull + (n_tiles - nfull) * kp;
  auto unit_tile = [&](int u) { return kKP && u >= nfull ? nfull + (u - nfull) / kp : u; };
  auto unit_piece = [&](int u) { return kKP && u >= nfull ? (u - nfull) % kp : -1; };
  auto unit_sb0 = [&](int u) -> int64_t { return kKP && u >= nfull ? nsb * unit_piece(u) / kp : 0; };
  auto unit_sb1 = [&](int u) -> int64_t { return kKP && u >= nfull ? nsb * (unit_piece(u) + 1) / kp : nsb; };

  const uint32_t bar = base + L::kBar;
  auto full = [&](int s) { return bar + 8u * s; };
  auto empty = [&](int s) { return bar + 8u * (STAGES + s); };
  auto rfull = [&](int r) { return bar + 8u * (2 * STAGES + r); };
  auto rempty = [&](int r) { return bar + 8u * (2 * STAGES + NR + r); };
  auto sfull = [&](int e) { return bar + 8u * (2 * STAGES + 2 * NR + e); };
  auto sempty = [&](int e) { return bar + 8u * (2 * STAGES + 2 * NR + SRING + e); };
  constexpr bool SH = L::kShared;
  constexpr int MR = L::kMR;
  auto mfull = [&](int r) { return bar + 8u * (2 * STAGES + 2 * NR + 2 * SRING + r); };
  auto mempty = [&](int r) { return bar + 8u * (2 * STAGES + 3 * NR + 2 * SRING + r); };
  auto mrfull = [&](int m) { return bar + 8u * (2 * STAGES + 4 * NR + 2 * SRING + m); };
  auto mrempty = [&](int m) { return bar + 8u * (2 * STAGES + 4 * NR + 2 * SRING + MR + m); };
  const uint32_t done = bar + 8u * (L::kNumBars - 1);
  auto a_smem = [&](int s) { return base + s * L::kStage; };
  auto b_smem = [&](int s) { return base + s * L::kStage + L::kA; };
  auto s_smem = [&](int e) { return base + L::kScaleRing + e * L::kScale; };
  auto m_smem = [&](int m) { return base + L::kMinRing + m * L::kMinEntry; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int r = 0; r < NR; ++r) {
      mbar_init(rfull(r), 1);
      mbar_init(rempty(r), EPI_WARPS);
    }
    for (int e = 0; e < SRING; ++e) {
      mbar_init(sfull(e), 1);
      mbar_init(sempty(e), EPI_WARPS);
    }
    if constexpr (SH) {
      for (int r = 0; r < NR; ++r) {
        mbar_init(mfull(r), 1);
        mbar_init(mempty(r), EPI_WARPS);
      }
      for (int m = 0; m < MR; ++m) {
        mbar_init(mrfull(m), 1);
        mbar_init(mrempty(m), 1);
      }
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == ISSUER_WARP) {
    tmem_alloc(base + L::kSlot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + L::kSlot);
  if (warp >= PRODUCER_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(SplitRegs<L::kShared>::kCtl));
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // (kKP) The weight copies of the first unit's first stages do not depend on
    // the quantization kernel: with few token rows it holds few SMs, so this
    // CTA may already run beside it, and they go out before the wait (their
    // bytes expected without an arrival; the activation copies arrive later).
    uint32_t pre = 0;
    if constexpr (kKP) {
      if (static_cast<int>(blockIdx.x) < n_units) {
        const int u = blockIdx.x, og = unit_tile(u) / n_tt;
        const int64_t sb0 = unit_sb0(u);
        pre = static_cast<uint32_t>(min(static_cast<int64_t>(STAGES), 4 * (unit_sb1(u) - sb0)));
        if (lane == 1) {
          for (uint32_t q = 0; q < pre; ++q) {  // (the ring is fresh: these stages are free)
            const int64_t sb = sb0 + q / 4;
            const int qq = static_cast<int>(q % 4), half = qq >> 1, kb = qq & 1;
            const bool mins = kQ4 && !SH && qq == 3;
            mbar_expect_tx(full(static_cast<int>(q)), NW * L::kBK + (mins ? L::kMinB : 0));
            for (int w = 0; w < NW; ++w) {
              const uint8_t *bblk = bplane + b_block(wtile(og, w), sb, half, nsb, kQ4);
              bulk_load(b_smem(q) + w * L::kBK, bblk + kb * L::kBK, L::kBK, full(q));
              if (mins) bulk_load(b_smem(q) + NW * L::kBK + w * kMinBytes, bblk + kBMin, kMinBytes, full(q));
            }
          }
        }
        __syncwarp();
      }
    }
    griddep_wait();  // the activation blocks come from the kernel before this one
    uint32_t ks = 0, ns = 0, issued = 0, s_issued = 0, m_issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int tile = unit_tile(u);
      const int tt = tile % n_tt, og = tile / n_tt;
      // kKP: bytes of each activation K-block's rows that are copied (rows up
      // to the tile's last token, rounded up to 8); otherwise all 128
      const int64_t rows_left = nt - static_cast<int64_t>(tt) * kTileM;
      const uint32_t arow =
          kKP ? static_cast<uint32_t>(((rows_left < kTileM ? rows_left : kTileM) + 7) & ~7) * 128u
              : static_cast<uint32_t>(kSplitLo);
      for (int64_t sb = unit_sb0(u); sb < unit_sb1(u) && ok; ++sb, ++ns) {
        const int e = static_cast<int>(ns % SRING);
        ok = __all_sync(0xffffffffu, mbar_wait(sempty(e), ((ns / SRING) & 1) ^ 1, wctl));
        if (!ok) break;
        if (lane == 2) {
          mbar_arrive_expect_tx(sfull(e), L::kScale);
          for (int w = 0; w < NW; ++w)
            bulk_load(s_smem(e) + w * scale_block_bytes(kQ4), bscale + b_scale_block(wtile(og, w), sb, nsb, kQ4),
                      scale_block_bytes(kQ4), sfull(e));
        }
        __syncwarp();
        s_issued = ns + 1;
        if constexpr (SH) {  // the min images of this super-block, into their own ring
          const int m = static_cast<int>(ns % MR);
          ok = __all_sync(0xffffffffu, mbar_wait(mrempty(m), ((ns / MR) & 1) ^ 1, wctl));
          if (!ok) break;
          if (lane == 3) {
            mbar_arrive_expect_tx(mrfull(m), L::kMinEntry);
            bulk_load(m_smem(m), aplane + as_block(tt, sb, 1, nsb, kQ4) + kSplitMin, kMinBytes, mrfull(m));
            for (int w = 0; w < NW; ++w)
              bulk_load(m_smem(m) + (1 + w) * kMinBytes, bplane + b_block(wtile(og, w), sb, 1, nsb, kQ4) + kBMin,
                        kMinBytes, mrfull(m));
          }
          __syncwarp();
          m_issued = ns + 1;
        }
        for (int qq = 0; qq < 4; ++qq, ++ks) {  // 64-K quarters of the super-block
          const int s = static_cast<int>(ks % STAGES);
          ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ((ks / STAGES) & 1) ^ 1, wctl));
          if (!ok) break;
          const int half = qq >> 1, kb = qq & 1;
          const bool mins = kQ4 && !SH && qq == 3;
          const uint8_t *ablk = aplane + as_block(tt, sb, half, nsb, kQ4);
          const bool w_done = ks < pre;  // (kKP) its weight copies went out before the wait
          if (lane == 0) {
            mbar_arrive_expect_tx(full(s), 2 * arow + (mins ? L::kMinA : 0) +
                                               (w_done ? 0 : NW * L::kBK * (kB0 ? 2 : 1) + (mins ? L::kMinB : 0)));
            if (kKP) {  // the hi and the lo K-block's first rows
              bulk_load(a_smem(s), ablk + kb * kSplitQuarter, arow, full(s));
              bulk_load(a_smem(s) + L::kALo, ablk + kb * kSplitQuarter + kSplitLo, arow, full(s));
            } else {
              bulk_load(a_smem(s), ablk + kb * kSplitQuarter, kSplitQuarter, full(s));
            }
            if (mins) bulk_load(a_smem(s) + L::kAMin, ablk + kSplitMin, L::kMinA, full(s));
          } else if (lane == 1 && !w_done) {
            for (int w = 0; w < NW; ++w) {
              const uint8_t *bblk = bplane + b_block(wtile(og, w), sb, half, nsb, kQ4);
              bulk_load(b_smem(s) + w * L::kBK, bblk + kb * L::kBK, L::kBK, full(s));
              if (mins) bulk_load(b_smem(s) + NW * L::kBK + w * kMinBytes, bblk + kBMin, kMinBytes, full(s));
            }
          } else if constexpr (kB0) {
            if (lane == 4) {
              for (int w = 0; w < NW; ++w)
                bulk_load(b_smem(s) + (NW + w) * L::kBK,
                          b0plane + b_block(wtile(og, w), sb, half, nsb, false) + kb * L::kBK, L::kBK, full(s));
            }
          }
          __syncwarp();
          issued = ks + 1;
        }
      }
    }
    if (!ok) {  // drain this CTA's copies still in flight
      // (kKP: stages whose weight copies went out before the wait but that
      // were never armed get their arrival now, so their phase can complete)
      if (lane == 0)
        for (uint32_t k = issued; k < pre; ++k) mbar_arrive(full(static_cast<int>(k)));
      __syncwarp();
      const uint32_t last = issued > pre ? issued : pre;
      for (uint32_t k = last > STAGES ? last - STAGES : 0; k < last; ++k)
        mbar_wait(full(k % STAGES), (k / STAGES) & 1, wctl, false);
      for (uint32_t k = s_issued > SRING ? s_issued - SRING : 0; k < s_issued; ++k)
        mbar_wait(sfull(k % SRING), (k / SRING) & 1, wctl, false);
      if constexpr (SH)
        for (uint32_t k = m_issued > MR ? m_issued - MR : 0; k < m_issued; ++k)
          mbar_wait(mrfull(k % MR), (k / MR) & 1, wctl, false);
    }
  } else if (warp == ISSUER_WARP) {
    // ------------------------------------------------------------ UMMA issuer
    uint32_t elected;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(elected));
    constexpr uint32_t idesc = idesc_f16_f32(kTileM, L::kN);
    constexpr uint64_t kStageDesc = L::kStage >> 4;
    const uint64_t ah0 = sdesc_kmajor_sw128(a_smem(0)), al0 = sdesc_kmajor_sw128(a_smem(0) + L::kALo);
    const uint64_t b0 = sdesc_kmajor_sw128(b_smem(0));
    const uint64_t am0 = sdesc_kmajor_sw32(SH ? m_smem(0) : a_smem(0) + L::kAMin);
    const uint64_t bm0 = sdesc_kmajor_sw32(SH ? m_smem(0) + kMinBytes : b_smem(0) + NW * L::kBK);
    uint32_t ks = 0, nr = 0;
    bool ok = true;
    // kShared: super-blocks below pmin have their min UMMA issued.  Min term n
    // goes into region n % NR after the epilogue has read accumulator n there
    // (rempty), and must be read (mempty) before accumulator n + NR starts.
    uint32_t pmin = 0;
    auto issue_min = [&](uint32_t n) {
      if constexpr (!SH) return;
      const int r = static_cast<int>(n % NR), m = static_cast<int>(n % (SH ? MR : 1));
      ok = __all_sync(0xffffffffu, mbar_wait(rempty(r), (n / NR) & 1, wctl));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(mrfull(m), (n / (SH ? MR : 1)) & 1, wctl));
      if (!ok) return;
      tc_fence_after();
      if (elected) {
        const uint64_t mo = static_cast<uint64_t>(m) * (L::kMinEntry >> 4);
        umma_f16(tbase + r * L::kN, am0 + mo, bm0 + mo, idesc, 0u);
        umma_commit(mfull(r));
        umma_commit(mrempty(m));
      }
      __syncwarp();
    };
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      for (int64_t sb = unit_sb0(u); sb < unit_sb1(u) && ok; ++sb, ++nr) {
        const int r = static_cast<int>(nr % NR);
        if constexpr (SH) {
          while (ok && pmin + NR <= nr) issue_min(pmin++);  // the region's last min term goes first
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(mempty(r), ((nr / NR) & 1) ^ 1, wctl));
        } else {
          ok = __all_sync(0xffffffffu, mbar_wait(rempty(r), ((nr / NR) & 1) ^ 1, wctl));
        }
        if (!ok) break;
        const uint32_t dacc = tbase + r * L::kN, dmin = tbase + (NR + r) * L::kN;
        for (int qq = 0; qq < 4 && ok; ++qq, ++ks) {
          if constexpr (SH) {
            // The previous super-block's min term: after this one's first
            // stage if its region was read by then, at the latest after the
            // second.  The issuer runs stages ahead of the tensor pipe; waiting
            // longer would queue the min term behind most of this super-block
            // and keep its region from the next accumulator.
            if (pmin < nr && qq >= 1) {
              const uint32_t n = pmin;
              if (qq >= 2 || __all_sync(0xffffffffu, mbar_test_wait(rempty(n % NR), (n / NR) & 1))) {
                issue_min(n);
                ++pmin;
                if (!ok) break;
              }
            }
          }
          const int s = static_cast<int>(ks % STAGES);
          ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
          if (!ok) break;
          tc_fence_after();
          if (elected) {
            const uint64_t so = s * kStageDesc;
#pragma unroll
            for (int lc = 0; lc < 2; ++lc) {  // 32-K chunks: 64 B into the swizzled rows
              const uint64_t off = so + lc * (64 >> 4);
              umma_f16(dacc, ah0 + off, b0 + off, idesc, (qq | lc) ? 1u : 0u);
              umma_f16(dacc, ah0 + off + 2, b0 + off + 2, idesc, 1u);
              umma_f16(dacc, al0 + off, b0 + off, idesc, 1u);
              umma_f16(dacc, al0 + off + 2, b0 + off + 2, idesc, 1u);
              if (kB0) {  // the same A against the B0 images
                constexpr uint64_t kB0Desc = (NW * L::kBK) >> 4;
                umma_f16(dacc, ah0 + off, b0 + kB0Desc + off, idesc, 1u);
                umma_f16(dacc, ah0 + off + 2, b0 + kB0Desc + off + 2, idesc, 1u);
                umma_f16(dacc, al0 + off, b0 + kB0Desc + off, idesc, 1u);
                umma_f16(dacc, al0 + off + 2, b0 + kB0Desc + off + 2, idesc, 1u);
              }
            }
            if (kQ4 && !SH && qq == 3) umma_f16(dmin, am0 + so, bm0 + so, idesc, 0u);
            umma_commit(empty(s));
            if (qq == 3) umma_commit(rfull(r));
          }
          __syncwarp();
        }
      }
    }
    if constexpr (SH)
      while (ok && pmin < nr) issue_min(pmin++);
    if (elected) umma_commit(done);
    __syncwarp();
    mbar_wait(done, 0, wctl, false);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SplitRegs<L::kShared>::kEpi));
    // ------------------------------------------------------------ epilogue
    // warp w: TMEM lanes 32*(w%4).., columns (w/4)*kN/2 .. of a region
    constexpr int CW = L::kN / 2;  // columns per warp
    const int quad = warp & 3;
    const int chalf = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t taddr = tbase + (static_cast<uint32_t>(quad * 32) << 16) + chalf * CW;
    uint32_t nr = 0, ns = 0;
    bool ok = true;
    griddep_wait();  // 2^-s comes from the kernel before this one
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int tile = unit_tile(u);
      const int tt = tile % n_tt, og = tile / n_tt;
      const int64_t t = static_cast<int64_t>(tt) * kTileM + row;
      // this warp's columns: weight tile og*NW + chalf (kWide), else half chalf of tile og
      const int wt = kWide ? og * NW + chalf : og;
      const int64_t o0 = static_cast<int64_t>(wt) * kTileN + (kWide ? 0 : chalf * 64);
      float2 y[CW / 2];
#pragma unroll
      for (int i = 0; i < CW / 2; ++i) y[i] = make_float2(0.f, 0.f);
      for (int64_t sb = unit_sb0(u); sb < unit_sb1(u) && ok; ++sb, ++nr, ++ns) {
        const int r = static_cast<int>(nr % NR), e = static_cast<int>(ns % SRING);
        ok = __all_sync(0xffffffffu, mbar_wait(rfull(r), (nr / NR) & 1, wctl));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(sfull(e), (ns / SRING) & 1, wctl));
        if (!ok) break;
        tc_fence_after();
        const uint8_t *sblk = smem + (s_smem(e) - base) + (kWide ? chalf * scale_block_bytes(kQ4) : 0);
        const float4 *d4 = reinterpret_cast<const float4 *>(sblk) + (kWide ? 0 : chalf * 16);
        fold_region<CW, false, SH ? 32 : 64>(taddr + r * L::kN, d4, y);
        if (kQ4) {
          uint32_t mreg = static_cast<uint32_t>(NR + r) * L::kN;
          if constexpr (SH) {  // the accumulator's region goes back, its min term comes into it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(rempty(r));
            ok = __all_sync(0xffffffffu, mbar_wait(mfull(r), (nr / NR) & 1, wctl));
            if (!ok) break;
            tc_fence_after();
            mreg = static_cast<uint32_t>(r) * L::kN;
          }
          const float4 *m4 = reinterpret_cast<const float4 *>(sblk + kSDmin) + (kWide ? 0 : chalf * 16);
          fold_region<CW, true, SH ? 32 : 64>(taddr + mreg, m4, y);
        }
        // the region and the scale entry go back
        tc_fence_before();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(SH ? mempty(r) : rempty(r));
          mbar_arrive(sempty(e));
        }
      }
      if (!ok) break;
      if constexpr (kKP) {
       if (u >= nfull) {
        __shared__ int s_last;  // whether this CTA finished its tile's last piece
        // this piece's partial sums (times 2^-s_t, exact), then the tile's
        // count; the last of its pieces adds them all, in piece order, from
        // `part`.  Layout per (piece, pieced tile): [column half][float4 i of
        // the warp's CW columns][row], so a warp's 32 rows are 512 contiguous bytes
        const int piece = unit_piece(u), pt = tile - nfull, n_pieced = n_tiles - nfull;
        auto at = [&](int pc) {
          return reinterpret_cast<float4 *>(part) +
                 ((static_cast<int64_t>(pc) * n_pieced + pt) * 2 + chalf) * (CW / 4) * kTileM + row;
        };
        if (t < nt) {
          const float inv = __ldg(invp + t);
          float4 *dst = at(piece);
#pragma unroll
          for (int i = 0; i < CW / 4; ++i) {
            const float2 a = __fmul2_rn(y[2 * i], make_float2(inv, inv));
            const float2 b = __fmul2_rn(y[2 * i + 1], make_float2(inv, inv));
            __stcg(dst + i * kTileM, make_float4(a.x, a.y, b.x, b.y));
          }
        }
        // the CTA's stores, then one thread's count with release and acquire
        // semantics (the barrier orders the other threads' stores before it,
        // and the last piece's reads after it)
        epi_bar();
        if (threadIdx.x == 0) {
          uint32_t prev;
          asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(cnt + pt) : "memory");
          s_last = static_cast<int>(prev) == kp - 1;
        }
        epi_bar();
        const int rows_live =
            static_cast<int>(min(static_cast<int64_t>(kTileM), nt - static_cast<int64_t>(tt) * kTileM));
        if (s_last && !kWide && rows_live <= 8) {
          // Few live rows (below nt): their float4 items -- at most 8 rows x
          // 32 -- shared over the epilogue threads, one each, rows fastest;
          // each the sum of its kp partials in piece order, the loads of up
          // to 4 pieces in flight together
          constexpr int kQ = CW / 4;  // float4 per row of a column half
          const int idx = static_cast<int>(threadIdx.x);
          if (idx < rows_live * 2 * kQ) {
            const int r = idx % rows_live, hq = idx / rows_live, ch = hq / kQ, i = hq % kQ;
            const float4 *src = reinterpret_cast<const float4 *>(part) +
                                ((static_cast<int64_t>(pt) * 2 + ch) * kQ + i) * kTileM + r;
            const int64_t pstride = static_cast<int64_t>(n_pieced) * 2 * kQ * kTileM;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int pc0 = 0; pc0 < kp; pc0 += 4) {
              float4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (pc0 + j < kp) v[j] = __ldcg(src + (pc0 + j) * pstride);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (pc0 + j < kp) {
                  const float2 a = __fadd2_rn(make_float2(acc.x, acc.y), make_float2(v[j].x, v[j].y));
                  const float2 b = __fadd2_rn(make_float2(acc.z, acc.w), make_float2(v[j].z, v[j].w));
                  acc = make_float4(a.x, a.y, b.x, b.y);
                }
            }
            const int64_t tr = static_cast<int64_t>(tt) * kTileM + r;
            const int64_t oc = static_cast<int64_t>(og) * kTileN + ch * 64 + 4 * i;
            float *yp = Y + tr * od + oc;
            if ((od & 3) == 0 && oc + 4 <= od) {
              *reinterpret_cast<float4 *>(yp) = acc;
            } else {
              if (oc < od) yp[0] = acc.x;
              if (oc + 1 < od) yp[1] = acc.y;
              if (oc + 2 < od) yp[2] = acc.z;
              if (oc + 3 < od) yp[3] = acc.w;
            }
          }
        } else if (s_last && t < nt && (!kWide || og * NW + chalf < n_ot)) {
          // each thread its row's CW columns, all pieces' loads of a piece in flight together
#pragma unroll
          for (int i = 0; i < CW / 2; ++i) y[i] = make_float2(0.f, 0.f);
          for (int pc = 0; pc < kp; ++pc) {
            const float4 *src = at(pc);
#pragma unroll
            for (int i = 0; i < CW / 4; ++i) {
              const float4 v = __ldcg(src + i * kTileM);
              y[2 * i] = __fadd2_rn(y[2 * i], make_float2(v.x, v.y));
              y[2 * i + 1] = __fadd2_rn(y[2 * i + 1], make_float2(v.z, v.w));
            }
          }
          store_y_row<0>(Y, t, od, o0, y, 1.0f);
          if constexpr (CW > 64) store_y_row<32>(Y, t, od, o0 + 64, y, 1.0f);
        }
        continue;
       }
      }
      if (t < nt && (!kWide || og * NW + chalf < n_ot)) {  // (a repeated last tile is not stored)
        const float inv = __ldg(invp + t);
        store_y_row<0>(Y, t, od, o0, y, inv);
        if constexpr (CW > 64) store_y_row<32>(Y, t, od, o0 + 64, y, inv);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == ISSUER_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- the pair arm's GEMM
// The split arm's operands and arithmetic on pairs of SMs.  A 2-CTA cluster
// computes output tiles of 256 weight rows x 128 tokens with cta_group::2
// UMMAs of M = 256, N = 128: the weights are the A operand (each CTA stages
// its own weight tile's 128 rows) and the hi and lo activation images the B
// operand (each CTA stages half of the tile's tp = 128, 112 or 96 token rows, from
// the pair layout of tiling.h).  A 64-K stage takes two bulk copies per CTA,
// its weight K-block and its activation rows (hi and lo side by side in the
// pair layout), so six stages are in flight: measured, three or four copies
// per 64-K stage fall behind the tensor pipe while two keep pace with it, and
// three 128-K stages leave the ring waiting on the copies' round trip.  Per
// output the
// exact products and the epilogue's fp32 operations are those of the 128-row
// split kernel, with the tile transposed -- TMEM lane = weight row, column =
// token, so the scales d and dmin are one value per thread; the tensor core's
// summation order inside a super-block may differ.
//
// Roles (both CTAs): warps 0-7 epilogue of the CTA's own 128 weight rows,
// warps 8 and 10 producers (the CTA's own stages, even and odd, and its
// scale blocks).  Warp 9: in the even CTA the UMMA issuer; in the odd CTA a
// relay that, once a stage of its own has landed, arrives on the even CTA's
// barrier for that stage, which so waits for both halves.  The issuer's commits arrive on both CTAs' barriers
// (stage free, accumulator ready); both epilogues arrive on the even CTA's
// accumulator-free barrier.  The q4_K min term: per super-block one K = 16
// pair UMMA of the weight min images (A) against the activation min images
// (B), into a region of its own, issued with the super-block's last stage:
// the activation min image comes in that stage's activation copy (it follows
// the lo K-block in the pair layout), the weight one into a two-entry ring
// that the same stage fills (a commit covers every earlier UMMA, so an entry
// is free again two super-blocks later).
struct PairShape {
  static constexpr int kThreads = 384;
  static constexpr int kRegsLaunch = 168;
  static constexpr int kRegsEpi = 208;
  static constexpr int kRegsCtl = 88;
  static_assert(256 * kRegsEpi + (kThreads - 256) * kRegsCtl == kThreads * kRegsLaunch,
                "the register split must add up to what the launch holds");
};
template <bool kQ4>
struct PairSmem {
  static constexpr int kW = kTileN * 64 * 2;                  // weight K-block: 128 rows x 64 K, 16384
  static constexpr int kAB = 2 * pair_kb_bytes(64) + (kQ4 ? 64 * 32 : 0);  // up to 64 token rows: hi, lo, min
  static constexpr int kStage = kW + (kAB + 1023) / 1024 * 1024;
  static constexpr int kStages = 6;
  static constexpr int kMR = kQ4 ? 2 : 0;                     // weight min-image ring (q4_K)
  static constexpr int kMinRing = kStages * kStage;
  static constexpr int kScale = scale_block_bytes(kQ4);
  static constexpr int kScaleRing = kMinRing + kMR * kMinBytes;
  static constexpr int kRegions = kQ4 ? 2 : 4;  // accumulators of 128 columns (q4_K: then as many min regions)
  static constexpr int kBar = kScaleRing + SRING * kScale;
  // full, empty per stage; rfull, rempty per region; sfull, sempty per scale entry; done
  static constexpr int kNumBars = 2 * kStages + 2 * kRegions + 2 * SRING + 1;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kSlot + 16 + 1024;
  static_assert(kStage % 1024 == 0 && kMinBytes % 1024 == 0, "stage buffers keep 1 KB alignment");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(kRegions * 128 * (kQ4 ? 2 : 1) <= TMEM_COLS, "TMEM columns");
};

template <bool kQ4>
__global__ void __launch_bounds__(PairShape::kThreads, 1)
    mmq_gemm_pair_kernel(const uint8_t *__restrict__ aplane, const uint8_t *__restrict__ bplane,
                         const uint8_t *__restrict__ bscale, const float *__restrict__ invp, int64_t nt,
                         int64_t od, int64_t nb32, int n_tt, int n_ot, float *__restrict__ Y, WaitCtl wctl,
                         int tp) {
  using L = PairSmem<kQ4>;
  constexpr int STAGES = L::kStages, NR = L::kRegions;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the UMMAs; 1: its peer
  const int pair = static_cast<int>(blockIdx.x >> 1), n_pairs = static_cast<int>(gridDim.x >> 1);
  const int64_t nsb = nb32 / 8;
  const int h = tp / 2;             // token rows each CTA stages (a multiple of 8, at most 64)
  const int n_wp = (n_ot + 1) / 2;  // pairs of weight tiles
  const int n_units = n_tt * n_wp;  // token tiles fastest
  // this CTA's weight tile of pair wp (an odd n_ot's last pair repeats its tile, not stored)
  auto wtile = [&](int wp) { return min(2 * wp + static_cast<int>(rank), n_ot - 1); };

  const uint32_t bar = base + L::kBar;
  auto full = [&](int s) { return bar + 8u * s; };
  auto empty = [&](int s) { return bar + 8u * (STAGES + s); };
  auto rfull = [&](int r) { return bar + 8u * (2 * STAGES + r); };
  auto rempty = [&](int r) { return bar + 8u * (2 * STAGES + NR + r); };
  auto sfull = [&](int e) { return bar + 8u * (2 * STAGES + 2 * NR + e); };
  auto sempty = [&](int e) { return bar + 8u * (2 * STAGES + 2 * NR + SRING + e); };
  const uint32_t done = bar + 8u * (L::kNumBars - 1);
  auto w_smem = [&](int s) { return base + s * L::kStage; };
  auto a_smem = [&](int s) { return base + s * L::kStage + L::kW; };
  auto m_smem = [&](int m) { return base + L::kMinRing + m * kMinBytes; };
  auto s_smem = [&](int e) { return base + L::kScaleRing + e * L::kScale; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), rank == 0 ? 2 : 1);  // the even CTA's: its own copies and the peer's relay
      mbar_init(empty(s), 1);
    }
    for (int r = 0; r < NR; ++r) {
      mbar_init(rfull(r), 1);
      mbar_init(rempty(r), 2 * EPI_WARPS);  // (the even CTA's is the one used: both epilogues)
    }
    for (int e = 0; e < SRING; ++e) {
      mbar_init(sfull(e), 1);
      mbar_init(sempty(e), EPI_WARPS);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == ISSUER_WARP) {
    tmem_alloc_pair(base + L::kSlot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers are initialised before either arrives on the other's
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + L::kSlot);
  if (warp >= PRODUCER_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PairShape::kRegsCtl));
    if (warp == PRODUCER_WARP || warp == PRODUCER2_WARP) {
      // ------------------------------------------------------------ producers
      // two warps, the even and the odd stages (the scale blocks with the
      // even ones); one warp's per-stage code spilled in the q4_K variant
      const int p = warp == PRODUCER_WARP ? 0 : 1;
      // The first unit's first stages' weight copies (and min images) do not
      // depend on the quantization kernel: they go out before the wait for
      // it, their bytes expected without an arrival (the ring is fresh).
      uint32_t pre = 0;
      if (pair < n_units) {
        const int w = wtile(pair / n_tt);
        pre = static_cast<uint32_t>(min(static_cast<int64_t>(STAGES), 4 * nsb));
        if (lane == 0)
          for (uint32_t q = p; q < pre; q += 2) {
            const int64_t sb = q / 4;
            const int qq = static_cast<int>(q % 4), half = qq >> 1, kb = qq & 1;
            const bool mins = kQ4 && qq == 3;
            mbar_expect_tx(full(static_cast<int>(q)), L::kW + (mins ? kMinBytes : 0));
            bulk_load(w_smem(static_cast<int>(q)), bplane + b_block(w, sb, half, nsb, kQ4) + kb * L::kW, L::kW,
                      full(static_cast<int>(q)));
            if (mins)
              bulk_load(m_smem(static_cast<int>(sb % (kQ4 ? L::kMR : 1))), bplane + b_block(w, sb, 1, nsb, kQ4) + kBMin,
                        kMinBytes, full(static_cast<int>(q)));
          }
        __syncwarp();
      }
      griddep_wait();  // the activation blocks come from the kernel before this one
      uint32_t ks = 0, ns = 0, issued = 0, s_issued = 0;
      bool ok = true;
      for (int u = pair; u < n_units && ok; u += n_pairs) {
        const int tt = u % n_tt, w = wtile(u / n_tt);
        for (int64_t sb = 0; sb < nsb && ok; ++sb, ++ns) {
          const int e = static_cast<int>(ns % SRING);
          if (p == 0) ok = __all_sync(0xffffffffu, mbar_wait(sempty(e), ((ns / SRING) & 1) ^ 1, wctl));
          if (!ok) break;
          for (int qq = 0; qq < 4; ++qq, ++ks) {  // 64-K quarters of the super-block
            if (static_cast<int>(ks & 1) != p) continue;
            const int s = static_cast<int>(ks % STAGES);
            ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ((ks / STAGES) & 1) ^ 1, wctl));
            if (!ok) break;
            if (lane == 0) {
              const int half = qq >> 1, kb = qq & 1;
              const bool mins = kQ4 && qq == 3;
              const bool w_done = ks < pre;  // its weight copies went out before the wait
              // this CTA's rows of the hi and the lo K-block (and, last quarter, the min image after them)
              const uint32_t ab = 2 * pair_kb_bytes(h) + (mins ? h * 32 : 0);
              mbar_arrive_expect_tx(full(s), ab + (w_done ? 0 : L::kW + (mins ? kMinBytes : 0)));
              if (!w_done) bulk_load(w_smem(s), bplane + b_block(w, sb, half, nsb, kQ4) + kb * L::kW, L::kW, full(s));
              bulk_load(a_smem(s),
                        aplane + pair_block(tt, sb, half, nsb, kQ4, h) + rank * pair_rank_bytes(kQ4, half, h) +
                            kb * 2 * pair_kb_bytes(h),
                        ab, full(s));
              if (mins && !w_done)
                bulk_load(m_smem(static_cast<int>(ns % (kQ4 ? L::kMR : 1))),
                          bplane + b_block(w, sb, 1, nsb, kQ4) + kBMin, kMinBytes, full(s));
            }
            __syncwarp();
            issued = ks + 1;
            if (qq == 0) {  // (producer 0) the super-block's scales, after its first stage's operands
              if (lane == 1) {
                mbar_arrive_expect_tx(sfull(e), L::kScale);
                bulk_load(s_smem(e), bscale + b_scale_block(w, sb, nsb, kQ4), L::kScale, sfull(e));
              }
              __syncwarp();
              s_issued = ns + 1;
            }
          }
        }
      }
      if (!ok) {  // drain this warp's copies still in flight
        // (stages whose weight copies went out before the wait but that were
        // never armed get this CTA's arrival now)
        if (lane == 0)
          for (uint32_t k = issued; k < pre; ++k)
            if (static_cast<int>(k & 1) == p) mbar_arrive(full(static_cast<int>(k)));
        __syncwarp();
        const uint32_t last = issued > pre ? issued : pre;
        for (uint32_t k = last > STAGES ? last - STAGES : 0; k < last; ++k)
          if (static_cast<int>(k & 1) == p) mbar_wait(full(k % STAGES), (k / STAGES) & 1, wctl, false);
        for (uint32_t k = s_issued > SRING ? s_issued - SRING : 0; k < s_issued; ++k)
          mbar_wait(sfull(k % SRING), (k / SRING) & 1, wctl, false);
      }
    } else if (warp == ISSUER_WARP && rank == 1) {
      // ------------------------------------------------------------ relay (odd CTA)
      uint32_t ks = 0;
      bool ok = true;
      for (int u = pair; u < n_units && ok; u += n_pairs) {
        for (int64_t q = 0; q < 4 * nsb && ok; ++q, ++ks) {
          const int s = static_cast<int>(ks % STAGES);
          ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
          if (ok && lane == 0) mbar_arrive_cluster(mapa_shared(full(s), 0));
          __syncwarp();
        }
      }
      mbar_wait(done, 0, wctl, false);  // the even CTA's last UMMA has read this CTA's stages
    } else if (warp == ISSUER_WARP) {
      // ------------------------------------------------------------ UMMA issuer (even CTA)
      uint32_t elected;
      asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(elected));
      const uint32_t idesc = idesc_f16_f32(256, tp);
      constexpr uint64_t kStageDesc = L::kStage >> 4;
      const uint64_t w0 = sdesc_kmajor_sw128(w_smem(0)), h0 = sdesc_kmajor_sw128(a_smem(0));
      const uint64_t l0 = sdesc_kmajor_sw128(a_smem(0) + pair_kb_bytes(h));
      const uint64_t am0 = sdesc_kmajor_sw32(a_smem(0) + 2 * pair_kb_bytes(h));
      const uint64_t wm0 = sdesc_kmajor_sw32(m_smem(0));
      uint32_t ks = 0, nr = 0;
      bool ok = true;
      for (int u = pair; u < n_units && ok; u += n_pairs) {
        for (int64_t sb = 0; sb < nsb && ok; ++sb, ++nr) {
          const int r = static_cast<int>(nr % NR);
          ok = __all_sync(0xffffffffu, mbar_wait(rempty(r), ((nr / NR) & 1) ^ 1, wctl));
          if (!ok) break;
          const uint32_t dacc = tbase + r * 128, dmin = tbase + (NR + r) * 128;
          for (int qq = 0; qq < 4 && ok; ++qq, ++ks) {
            const int s = static_cast<int>(ks % STAGES);
            ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
            if (!ok) break;
            tc_fence_after();
            if (elected) {
              const uint64_t so = s * kStageDesc;
#pragma unroll
              for (int lc = 0; lc < 2; ++lc) {  // 32-K chunks: 64 B into the swizzled rows
                const uint64_t off = so + lc * (64 >> 4);
                umma_pair_f16(dacc, w0 + off, h0 + off, idesc, (qq | lc) ? 1u : 0u);
                umma_pair_f16(dacc, w0 + off + 2, h0 + off + 2, idesc, 1u);
                umma_pair_f16(dacc, w0 + off, l0 + off, idesc, 1u);
                umma_pair_f16(dacc, w0 + off + 2, l0 + off + 2, idesc, 1u);
              }
              if (kQ4 && qq == 3)
                umma_pair_f16(dmin, wm0 + static_cast<uint64_t>(nr % 2) * (kMinBytes >> 4), am0 + so, idesc, 0u);
              umma_pair_commit(empty(s));
              if (qq == 3) umma_pair_commit(rfull(r));
            }
            __syncwarp();
          }
        }
      }
      if (elected) umma_pair_commit(done);
      __syncwarp();
      mbar_wait(done, 0, wctl, false);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PairShape::kRegsEpi));
    // ------------------------------------------------------------ epilogue
    // warp w: TMEM lanes (weight rows) 32*(w%4).., columns 64*(w/4) .. +63 (those below tp are tokens)
    const int quad = warp & 3, chalf = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t taddr = tbase + (static_cast<uint32_t>(quad * 32) << 16) + chalf * 64;
    uint32_t nr = 0, ns = 0;
    bool ok = true;
    griddep_wait();  // 2^-s comes from the kernel before this one
    for (int u = pair; u < n_units && ok; u += n_pairs) {
      const int tt = u % n_tt, wp = u / n_tt, w = wtile(wp);
      float2 y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = make_float2(0.f, 0.f);
      for (int64_t sb = 0; sb < nsb && ok; ++sb, ++nr, ++ns) {
        const int r = static_cast<int>(nr % NR), e = static_cast<int>(ns % SRING);
        ok = __all_sync(0xffffffffu, mbar_wait(rfull(r), (nr / NR) & 1, wctl));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(sfull(e), (ns / SRING) & 1, wctl));
        if (!ok) break;
        tc_fence_after();
        const float *sc = reinterpret_cast<const float *>(smem + (s_smem(e) - base));
        const float d = sc[row];
        const float2 d2 = make_float2(d, d);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t t0[32];
          tmem_ld_32x32b_x32(taddr + r * 128 + g * 32, t0);
          tmem_wait_ld(t0);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            y[g * 16 + i] = __ffma2_rn(d2, make_float2(__uint_as_float(t0[2 * i]), __uint_as_float(t0[2 * i + 1])),
                                       y[g * 16 + i]);
        }
        if constexpr (kQ4) {
          const float nm = -sc[kScaleBytes / 4 + row];  // -dmin of this row
          const float2 m2 = make_float2(nm, nm);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t t0[32];
            tmem_ld_32x32b_x32(taddr + (NR + r) * 128 + g * 32, t0);
            tmem_wait_ld(t0);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              y[g * 16 + i] = __ffma2_rn(m2, make_float2(__uint_as_float(t0[2 * i]), __uint_as_float(t0[2 * i + 1])),
                                         y[g * 16 + i]);
          }
        }
        // the regions go back to the issuer, the scale entry to the producer
        tc_fence_before();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(mapa_shared(rempty(r), 0));
          mbar_arrive(sempty(e));
        }
      }
      if (!ok) break;
      const int64_t o = static_cast<int64_t>(w) * kTileN + row;
      if (2 * wp + static_cast<int>(rank) < n_ot && o < od) {
        // columns chalf*64 + c below tp are tokens tt*tp + chalf*64 + c
        const int64_t t0 = static_cast<int64_t>(tt) * tp + chalf * 64;
        const int64_t tend = min(nt, static_cast<int64_t>(tt) * tp + tp);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int64_t t = t0 + 2 * i;
          if (t < tend) Y[t * od + o] = __fmul_rn(y[i].x, __ldg(invp + t));
          if (t + 1 < tend) Y[(t + 1) * od + o] = __fmul_rn(y[i].y, __ldg(invp + t + 1));
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the other may still use its barriers, stages or TMEM
  if (warp == ISSUER_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, TMEM_COLS);
  }
}

// One CTA that waits on a barrier nothing arrives at: checks that a bounded
// wait returns and reports instead of hanging.
__global__ void wait_selftest_kernel(WaitCtl wctl) {
  __shared__ __align__(8) uint64_t b;
  const uint32_t a = smem_addr(&b);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    fence_mbar_init();
    mbar_wait(a, 0, wctl, false);
  }
}

}  // namespace

// Scratch for mmq_gemm_noalloc: a fixed device array in this module, so that
// entry point allocates nothing.  Every device that loads the library holds
// it until the process exits.  Its contents persist between calls; the
// launch below clears every part that must start at zero.
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

cudaError_t noalloc_scratch(int dev, void **out) {
  // host code sees g_noalloc_scratch only as a stand-in: fetch the real
  // device address once per device, with that device current
  static void *addr[64];
  static std::mutex mu;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

namespace {
template <bool kQ4, bool kSK, bool kRaw, bool kB0, bool kDump>
cudaError_t prepare_variant(int dev);
}  // namespace

// Everything the whole-tile fp16-plane GEMM of a handle needs loaded on its
// device: the module holding the fixed scratch array (its address looked up),
// the activation prepass and the GEMM kernel variant.  With lazy module
// loading these load on first use, and loading allocates device memory (the
// array, the kernels' code); registration calls this, so a later
// mmq_gemm_noalloc on the same handle loads nothing.
cudaError_t prepare_noalloc(const mmq_weights_s *h) {
  void *p = nullptr;
  cudaError_t e = noalloc_scratch(h->device, &p);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  const bool q4 = h->type == MMQ_Q4_K;
  e = q4 ? cudaFuncGetAttributes(&fa, gemm_prepass_kernel<true>) : cudaFuncGetAttributes(&fa, gemm_prepass_kernel<false>);
  if (e != cudaSuccess) return e;
  if (q4) return prepare_variant<true, false, false, false, false>(h->device);
  return h->b0plane ? prepare_variant<false, false, false, true, false>(h->device)
                    : prepare_variant<false, false, false, false, false>(h->device);
}

namespace {

// SM count of a device, read once.
int num_sms(int dev) {
  static std::atomic<int> cached[64];
  int v = cached[dev].load();
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cached[dev].store(v);
  }
  return v;
}

// Launch shape and scratch layout of one GEMM call.
struct GemmPlan {
  bool q4, streamk;
  int64_t n_tt, nt_pad, nsb, nb32;
  int n_ot, n_tiles, grid;
  size_t a_off, da_off, inv_off, ws_off, flag_off, bytes;
};

GemmPlan plan_gemm(const mmq_weights_s *h, int64_t nt, bool streamk_allowed) {
  GemmPlan p{};
  p.q4 = h->type == MMQ_Q4_K;
  p.n_tt = (nt + kTileM - 1) / kTileM;
  p.nt_pad = p.n_tt * kTileM;
  p.nsb = h->nsb;
  p.nb32 = h->nb32;
  p.n_ot = static_cast<int>(h->od_pad / kTileN);
  p.n_tiles = static_cast<int>(p.n_tt) * p.n_ot;
  const int sms = num_sms(h->device);
  // Whole tiles per CTA, unless groups of n_tt CTAs sharing the (weight
  // tile, super-block) units evenly cut the longest CTA's work by more than a
  // tenth and by more than three super-blocks: publishing and collecting a
  // split tile's partial sums costs about three super-blocks of work
  // (measured on the 3584 x 3584 q-proj shapes, where whole tiles win).
  const int64_t waves = (p.n_tiles + sms - 1) / sms;
  const int64_t gunits = static_cast<int64_t>(p.n_ot) * p.nsb;
  int64_t groups = p.n_tt <= sms ? sms / p.n_tt : 0;
  if (groups > gunits) groups = gunits;
  const int64_t sk_max = groups > 0 ? (gunits + groups - 1) / groups : 0;
  const int64_t tile_max = waves * p.nsb;
  p.streamk = streamk_allowed && groups >= 2 && 10 * sk_max < 9 * tile_max && tile_max - sk_max > 3;
  p.grid = p.streamk ? static_cast<int>(groups * p.n_tt) : (p.n_tiles < sms ? p.n_tiles : sms);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  p.a_off = 0;
  p.da_off = up(static_cast<size_t>(p.n_tt * p.nsb) * a_pair_bytes(p.q4));
  p.inv_off = p.da_off + up(static_cast<size_t>(p.nt_pad * p.nb32) * 4);
  p.ws_off = p.inv_off + up(static_cast<size_t>(p.nt_pad) * 4);
  p.flag_off = p.ws_off + (p.streamk ? static_cast<size_t>(p.grid) * kTileM * kTileN * 4 : 0);
  p.bytes = p.flag_off + (p.streamk ? up(static_cast<size_t>(p.grid) * 8) : 0);
  return p;
}

}  // namespace

size_t gemm_scratch_bytes(const mmq_weights_s *h, int64_t nt, bool streamk_allowed, bool raw) {
  (void)raw;  // both arms use the same scratch
  return plan_gemm(h, nt, streamk_allowed).bytes;
}

namespace {

// One GEMM kernel variant: its function, launch shape and a one-time check,
// per device, of the shared-memory opt-in and of the register count the
// register split was planned for (a mismatch would stall setmaxnreg).
template <bool kQ4, bool kSK, bool kRaw, bool kB0, bool kDump = false>
cudaError_t prepare_variant(int dev) {
  auto kern = mmq_gemm_kernel<kQ4, kSK, kRaw, kB0, kDump>;
  constexpr int smem = Smem<kQ4, kRaw, kB0>::kBytes;
  static std::atomic<int> ready[64];  // 0 unknown, 1 ready, 2 unusable
  int st = ready[dev].load();
  if (st == 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    st = fa.numRegs == Shape<kRaw>::kRegsLaunch ? 1 : 2;
    ready[dev].store(st);
  }
  return st == 1 ? cudaSuccess : cudaErrorInvalidKernelImage;
}

template <bool kQ4, bool kSK, bool kRaw, bool kB0, bool kDump = false>
cudaError_t launch_variant(int dev, int grid, cudaStream_t s, const uint8_t *aplane, const uint8_t *bplane,
                           const uint8_t *rawplane, const uint8_t *b0plane, const uint8_t *bscale, const float *dap,
                           const float *invp, int64_t nt, int64_t od, int64_t nb32, int n_tt, int n_ot,
                           float *Y, WaitCtl w, float4 *ws, uint64_t *flags, bool pdl,
                           float *dump = nullptr) {
  auto kern = mmq_gemm_kernel<kQ4, kSK, kRaw, kB0, kDump>;
  constexpr int smem = Smem<kQ4, kRaw, kB0>::kBytes;
  if (const cudaError_t e = prepare_variant<kQ4, kSK, kRaw, kB0, kDump>(dev); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Shape<kRaw>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, aplane, bplane, rawplane, b0plane, bscale, dap, invp, nt, od, nb32,
                            n_tt, n_ot, Y, w, ws, flags, dump);
}

}  // namespace

cudaError_t launch_gemm(const mmq_weights_s *h, const uint8_t *Q, const float *X, int64_t nt,
                        float *Y, void *scratch, bool streamk_allowed, bool raw, DevStatus *st,
                        unsigned epoch, uint64_t limit_ns, cudaStream_t s, cudaEvent_t ev0,
                        cudaEvent_t ev1, unsigned ev_flags, float *dump) {
  if (raw && (!h->rawplane || h->b0plane)) return cudaErrorInvalidValue;
  if (dump && (raw || streamk_allowed)) return cudaErrorInvalidValue;
  const GemmPlan p = plan_gemm(h, nt, streamk_allowed);
  const bool q4 = p.q4;
  const int64_t n_tt = p.n_tt, nt_pad = p.nt_pad, nsb = p.nsb, nb32 = p.nb32;
  uint8_t *base8 = static_cast<uint8_t *>(scratch);
  uint8_t *aplane = base8 + p.a_off;
  float *dap = reinterpret_cast<float *>(base8 + p.da_off);
  float *invp = reinterpret_cast<float *>(base8 + p.inv_off);
  float4 *ws = p.streamk ? reinterpret_cast<float4 *>(base8 + p.ws_off) : nullptr;
  uint64_t *flags = p.streamk ? reinterpret_cast<uint64_t *>(base8 + p.flag_off) : nullptr;

  // activation operand plane: from pad40 blocks, or quantized from fp32 X.
  // One CTA per row of the padded token tiles: rows nt .. nt_pad - 1 quantize
  // a zero activation row, so the last tile's padding reads as zero.
  cudaError_t e = cudaSuccess;
  const unsigned pgrid = static_cast<unsigned>(nt_pad);
  // (the hand-off tags repeat when a CUDA graph replays this launch, so the
  // flags are cleared before every GEMM, by the kernel before it)
  const int nflags = p.streamk ? p.grid : 0;
  if (X) {
    const size_t stash = static_cast<size_t>(nb32) * kStashBytesPerBlock;
    if (!q4)
      quantize_prepass_kernel<false, false>
          <<<pgrid, 32 * kQuantWarps, 0, s>>>(X, nt, nb32, aplane, dap, invp, flags, nflags);
    else if (stash <= static_cast<size_t>(kStashMaxBytes))
      quantize_prepass_kernel<true, true>
          <<<pgrid, 32 * kQuantWarps, stash, s>>>(X, nt, nb32, aplane, dap, invp, flags, nflags);
    else
      quantize_prepass_kernel<true, false>
          <<<pgrid, 32 * kQuantWarps, 0, s>>>(X, nt, nb32, aplane, dap, invp, flags, nflags);
  } else if (q4) {
    gemm_prepass_kernel<true><<<pgrid, 128, 0, s>>>(Q, nt, nb32, aplane, dap, invp, flags, nflags);
  } else {
    gemm_prepass_kernel<false><<<pgrid, 128, 0, s>>>(Q, nt, nb32, aplane, dap, invp, flags, nflags);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int dev = h->device;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  if (ev0 && (e = cudaEventRecordWithFlags(ev0, s, ev_flags)) != cudaSuccess) return e;
  const uint8_t *bp = static_cast<const uint8_t *>(h->bplane);
  const uint8_t *bs = bp + b_scale_region(p.n_ot, nsb, q4);
  const uint8_t *rp = h->rawplane;
  const int nti = static_cast<int>(n_tt);
#define MMQ_LAUNCH(Q4, SK, RAW, B0)                                                                   \
  launch_variant<Q4, SK, RAW, B0>(dev, p.grid, s, aplane, bp, rp, h->b0plane, bs, dap, invp, nt, h->od, nb32, \
                                  nti, p.n_ot, Y, w, ws, flags, ev0 == nullptr)
#define MMQ_LAUNCH_DUMP(Q4, B0)                                                                          \
  launch_variant<Q4, false, false, B0, true>(dev, p.grid, s, aplane, bp, rp, h->b0plane, bs, dap, invp, nt, \
                                             h->od, nb32, nti, p.n_ot, Y, w, ws, flags, ev0 == nullptr, dump)
  if (dump)
    e = q4 ? MMQ_LAUNCH_DUMP(true, false) : h->b0plane ? MMQ_LAUNCH_DUMP(false, true) : MMQ_LAUNCH_DUMP(false, false);
  else if (q4)
    e = p.streamk ? (raw ? MMQ_LAUNCH(true, true, true, false) : MMQ_LAUNCH(true, true, false, false))
                  : (raw ? MMQ_LAUNCH(true, false, true, false) : MMQ_LAUNCH(true, false, false, false));
  else if (h->b0plane)  // (the raw arm has no B0 image: the API refuses it for such handles)
    e = p.streamk ? MMQ_LAUNCH(false, true, false, true) : MMQ_LAUNCH(false, false, false, true);
  else
    e = p.streamk ? (raw ? MMQ_LAUNCH(false, true, true, false) : MMQ_LAUNCH(false, true, false, false))
                  : (raw ? MMQ_LAUNCH(false, false, true, false) : MMQ_LAUNCH(false, false, false, false));
#undef MMQ_LAUNCH
#undef MMQ_LAUNCH_DUMP
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e == cudaSuccess && ev1) e = cudaEventRecordWithFlags(ev1, s, ev_flags);
  return e;
}

// ---------------------------------------------------------------- split arm launch
namespace {

// Launch shape and scratch layout of one split-arm GEMM: whole tiles of 128
// or 256 weight rows per CTA, whichever gives the busiest CTA the least time
// by the per-super-block costs measured on the GB300 (clk, one CTA per SM): a
// 128 x 128 super-block is bound by operand ingest at ~3150, a 128 x 256 one
// by the tensor pipe at ~4100 (q6_K) and ~4450 (q4_K, with its min term);
// with a B0 plane (twice the UMMAs) ~4200 and ~8200.
// (Stream-K over these tiles measured slower on the 3584 x 3584 x 512 shapes:
// the groups' first super-blocks pull most of the working set from HBM at
// once, the 128-row tiles are bound by the L2's total bandwidth rather than
// by the SM count, and the owner's read of the other pieces' partial sums is
// latency-bound.)
struct SplitPlan {
  bool q4, wide;
  int kp;      // pieces per pieced tile (1: whole tiles only)
  int n_full;  // tiles done whole, before the pieced ones
  int tp;      // tokens per tile (the pair arm: 128, 112 or 96; else 128)
  int64_t n_tt, nt_pad, nsb, rows;  // rows: activation rows the prepass writes
  int n_ot, n_tiles, grid;
  size_t inv_off, part_off, cnt_off, bytes;
};

// How many SM pairs the device holds at once for the pair kernel (one CTA per
// SM; how many pairs a device offers depends on how its SMs group), asked once
// per device; -1 if the kernel is unusable (its register count is not the
// one its register split was planned for).
template <bool kQ4>
int pair_capacity(int dev) {
  static std::atomic<int> cached[64];  // 0 unknown
  int pairs = cached[dev].load();
  if (pairs != 0) return pairs;
  auto kern = mmq_gemm_pair_kernel<kQ4>;
  constexpr int smem = PairSmem<kQ4>::kBytes;
  cudaFuncAttributes fa;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != PairShape::kRegsLaunch) {
    pairs = -1;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(num_sms(dev) / 2));
    cfg.blockDim = dim3(PairShape::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    pairs = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0 ? n : -1;
  }
  cached[dev].store(pairs);
  return pairs;
}

SplitPlan plan_split(const mmq_weights_s *h, int64_t nt, bool pair) {
  SplitPlan p{};
  p.q4 = h->type == MMQ_Q4_K;
  p.n_tt = (nt + kTileM - 1) / kTileM;
  p.nt_pad = p.n_tt * kTileM;
  p.nsb = h->nsb;
  p.n_ot = static_cast<int>(h->od_pad / kTileN);
  const int64_t sms = num_sms(h->device);
  int64_t best = -1;
  for (int wide = 0; wide < 2; ++wide) {
    const int64_t cost = h->b0plane ? (wide ? 8200 : 4200) : wide ? (p.q4 ? 4450 : 4100) : 3150;
    const int64_t tiles = p.n_tt * (wide ? (p.n_ot + 1) / 2 : p.n_ot);
    const int64_t est = (tiles + sms - 1) / sms * cost;
    if (best < 0 || est < best) {
      best = est;
      p.wide = wide;
      p.n_tiles = static_cast<int>(tiles);
      p.grid = static_cast<int>(tiles < sms ? tiles : sms);
    }
  }
  p.kp = 1;
  p.n_full = p.n_tiles;
  p.rows = p.nt_pad;
  p.tp = kTileM;
  if (pair) {
    // the pair arm: whole tiles of 256 weight rows x tp tokens, one SM pair
    // each; tp = 112 or 96 when that leaves fewer SM pairs idle (the q-proj
    // shapes at 512 tokens: 70 tiles over 140 SMs instead of 56 over 112)
    const int cap = p.q4 ? pair_capacity<true>(h->device) : pair_capacity<false>(h->device);
    const int64_t pairs = cap > 0 ? cap : 1, n_wp = (p.n_ot + 1) / 2;
    // waves of tiles times the tile's UMMA time: tp over the pair UMMA's
    // measured rate at N = tp (N = 128 and 112: the full rate, 96: 0.973)
    double best_est = -1;
    for (int tp : {128, 112, 96}) {
      const int64_t units = (nt + tp - 1) / tp * n_wp;
      const double est = static_cast<double>((units + pairs - 1) / pairs) * tp / (tp == 96 ? 0.973 : 1.0);
      if (best_est < 0 || est < best_est) {
        best_est = est;
        p.tp = tp;
      }
    }
    p.wide = false;
    p.n_tt = (nt + p.tp - 1) / p.tp;
    p.nt_pad = p.n_tt * p.tp;
    p.rows = p.nt_pad;
    p.n_tiles = static_cast<int>(p.n_tt * n_wp);
    p.n_full = p.n_tiles;
    p.grid = static_cast<int>(2 * std::min<int64_t>(p.n_tiles, pairs));
  } else if (!h->b0plane && p.nsb >= 2) {
    // Few 128-row tiles: every tile's super-blocks in pieces over the SMs,
    // when the busiest CTA then does fewer super-blocks (tensor-bound at ~2600
    // clk each with the activation rows trimmed to the tokens) plus ~1500 clk
    // of partial sums
    const int64_t tiles128 = p.n_tt * p.n_ot;
    if (2 * tiles128 <= sms) {
      const int64_t kp = std::min<int64_t>(p.nsb, sms / tiles128);
      const int64_t est = (p.nsb + kp - 1) / kp * 2600 + 1500;
      if (est < best * p.nsb) {  // (best: the whole-tile plan's clk per super-block)
        p.wide = false;
        p.kp = static_cast<int>(kp);
        p.n_tiles = static_cast<int>(tiles128);
        p.n_full = 0;
        p.grid = static_cast<int>(tiles128 * kp);
        // the last tile is copied only up to its last token row, rounded up to 8
        p.rows = (p.n_tt - 1) * kTileM + ((nt - (p.n_tt - 1) * kTileM + 7) & ~int64_t(7));
      }
    } else {
      // Several waves of whole tiles whose last wave leaves SMs idle: the
      // tiles of that wave in pieces over every CTA instead, when that saves
      // more than ~3000 clk of partial sums on the busiest CTA.  Not for q4_K
      // with 256-row tiles: that variant's epilogue (192 registers, the min
      // term sharing the accumulator regions) spills with the piece code and
      // measured 12 % slower on the FFN-up workload (476 against 424 us).
      const int64_t grid = p.grid, waves = (p.n_tiles + grid - 1) / grid;
      const int64_t rest = p.n_tiles - (waves - 1) * grid;
      const int64_t kp = std::min<int64_t>(p.nsb, rest > 0 ? grid / rest : 0);
      if (!(p.q4 && p.wide) && waves >= 2 && kp >= 2 && (p.nsb - (p.nsb + kp - 1) / kp) * (best / waves) > 3000) {
        p.kp = static_cast<int>(kp);
        p.n_full = static_cast<int>((waves - 1) * grid);
      }
    }
  }
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t per_sb = pair ? pair_sb_bytes(p.q4, p.tp / 2) : as_pair_bytes(p.q4);
  p.inv_off = up(static_cast<size_t>(p.n_tt * p.nsb) * per_sb);
  p.part_off = up(p.inv_off + static_cast<size_t>(p.nt_pad) * 4);
  const size_t pieced = static_cast<size_t>(p.n_tiles - p.n_full);
  p.cnt_off = p.part_off + (p.kp > 1 ? up(p.kp * pieced * kTileM * kTileN * 4 * (p.wide ? 2 : 1)) : 0);
  p.bytes = p.cnt_off + (p.kp > 1 ? up(pieced * 4) : 0);
  return p;
}

}  // namespace

size_t gemm_split_scratch_bytes(const mmq_weights_s *h, int64_t nt, bool pair) {
  return plan_split(h, nt, pair).bytes;
}

bool gemm_split_wide(const mmq_weights_s *h, int64_t nt) {
  const SplitPlan p = plan_split(h, nt, false);
  return p.wide || p.kp > 1;
}

// The library's choice of the pair arm (measured on the GB300, fused calls on
// the 3584 x 3584 weights at 16 .. 2048 tokens and the two FFN workloads):
// faster than every other arm above 128 tokens for both weight types (the
// one near-tie, within 1.5 %, at 768 tokens, where a second wave of tiles is
// mostly empty), slower than the split arm's pieces up to 128 tokens; for
// q6_K the split arm's 256-row tiles stay ahead (by 4 % on the FFN-down
// workload) when they fill at least two waves to 85 % or more.
bool gemm_pair_preferred(const mmq_weights_s *h, int64_t nt) {
  if (h->b0plane || nt <= kTileM) return false;
  const bool q4 = h->type == MMQ_Q4_K;
  if ((q4 ? pair_capacity<true>(h->device) : pair_capacity<false>(h->device)) < 0) return false;
  if (!q4) {
    const SplitPlan p = plan_split(h, nt, false);
    if (p.wide) {
      const int64_t sms = num_sms(h->device), waves = (p.n_tiles + sms - 1) / sms;
      if (waves >= 2 && 100 * static_cast<int64_t>(p.n_tiles) >= 85 * waves * sms) return false;
    }
  }
  return true;
}

namespace {

// The split and pair arms' activation prepass: from fp32 X (the token's codes
// kept in shared memory when they fit) or from pad40 blocks Q.
template <bool kQ4, bool kPair>
void split_prepass(const uint8_t *Q, const float *X, int64_t nt, int64_t nb32, uint8_t *aplane, float *invp, int *cnt,
                   int ncnt, unsigned pgrid, int tp, cudaStream_t s) {
  if (X) {
    const size_t stash = static_cast<size_t>(nb32) * kSplitStashBytesPerBlock;
    if (stash <= static_cast<size_t>(kStashMaxBytes))
      split_prepass_f32_kernel<kQ4, true, kPair><<<pgrid, 32 * kQuantWarps, stash, s>>>(X, nt, nb32, aplane, invp,
                                                                                         cnt, ncnt, tp);
    else
      split_prepass_f32_kernel<kQ4, false, kPair><<<pgrid, 32 * kQuantWarps, 0, s>>>(X, nt, nb32, aplane, invp,
                                                                                      cnt, ncnt, tp);
  } else {
    split_prepass_q_kernel<kQ4, kPair><<<pgrid, 128, 0, s>>>(Q, nt, nb32, aplane, invp, cnt, ncnt, tp);
  }
}

// The pair arm's kernel: launched as 2-CTA clusters, `grid` CTAs (pairs of
// CTAs, at most as many pairs as the device holds at once).
template <bool kQ4>
cudaError_t launch_pair(int dev, int grid, cudaStream_t s, bool pdl, const uint8_t *aplane, const uint8_t *bp,
                        const uint8_t *bs, const float *invp, int64_t nt, int64_t od, int64_t nb32, int n_tt,
                        int n_ot, float *Y, WaitCtl w, int tp) {
  if (pair_capacity<kQ4>(dev) < 0) return cudaErrorInvalidKernelImage;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(PairShape::kThreads);
  cfg.dynamicSmemBytes = PairSmem<kQ4>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, mmq_gemm_pair_kernel<kQ4>, aplane, bp, bs, invp, nt, od, nb32, n_tt, n_ot, Y, w,
                            tp);
}

}  // namespace

cudaError_t launch_gemm_split(const mmq_weights_s *h, const uint8_t *Q, const float *X, int64_t nt, float *Y,
                              void *scratch, DevStatus *st, unsigned epoch, uint64_t limit_ns,
                              cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, unsigned ev_flags, bool pair) {
  if (pair && h->b0plane) return cudaErrorInvalidValue;
  const SplitPlan p = plan_split(h, nt, pair);
  const bool q4 = p.q4, wide = p.wide;
  const int64_t n_tt = p.n_tt, nt_pad = p.nt_pad, nsb = p.nsb, nb32 = h->nb32;
  const int n_ot = p.n_ot;
  uint8_t *base8 = static_cast<uint8_t *>(scratch);
  uint8_t *aplane = base8;
  float *invp = reinterpret_cast<float *>(base8 + p.inv_off);
  float *part = p.kp > 1 ? reinterpret_cast<float *>(base8 + p.part_off) : nullptr;
  int *cnt = p.kp > 1 ? reinterpret_cast<int *>(base8 + p.cnt_off) : nullptr;
  const int ncnt = p.kp > 1 ? p.n_tiles - p.n_full : 0;
  const int dev = h->device;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t e = cudaSuccess;
  // one CTA per row of the padded token tiles (padding rows: a zero activation
  // row), or, with pieces, up to the last token row the GEMM copies
  const unsigned pgrid = static_cast<unsigned>(p.rows);
  if (q4)
    pair ? split_prepass<true, true>(Q, X, nt, nb32, aplane, invp, cnt, ncnt, pgrid, p.tp, s)
         : split_prepass<true, false>(Q, X, nt, nb32, aplane, invp, cnt, ncnt, pgrid, kTileM, s);
  else
    pair ? split_prepass<false, true>(Q, X, nt, nb32, aplane, invp, cnt, ncnt, pgrid, p.tp, s)
         : split_prepass<false, false>(Q, X, nt, nb32, aplane, invp, cnt, ncnt, pgrid, kTileM, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  if (ev0 && (e = cudaEventRecordWithFlags(ev0, s, ev_flags)) != cudaSuccess) return e;
  const uint8_t *bp = static_cast<const uint8_t *>(h->bplane);
  const uint8_t *bs = bp + b_scale_region(n_ot, nsb, q4);
  if (pair) {
    e = q4 ? launch_pair<true>(dev, p.grid, s, ev0 == nullptr, aplane, bp, bs, invp, nt, h->od, nb32,
                               static_cast<int>(n_tt), n_ot, Y, w, p.tp)
           : launch_pair<false>(dev, p.grid, s, ev0 == nullptr, aplane, bp, bs, invp, nt, h->od, nb32,
                                static_cast<int>(n_tt), n_ot, Y, w, p.tp);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) == cudaSuccess && ev1) e = cudaEventRecordWithFlags(ev1, s, ev_flags);
    return e;
  }
  const int grid = p.grid;
  auto go = [&](auto kern, int smem, int variant) -> cudaError_t {
    static std::atomic<int> ready[12][64];  // per kernel variant: 0 unknown, 1 ready, 2 unusable
    std::atomic<int> &rd = ready[variant][dev];
    int stt = rd.load();
    if (stt == 0) {
      cudaFuncAttributes fa;
      cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e2 == cudaSuccess) e2 = cudaFuncGetAttributes(&fa, kern);
      if (e2 != cudaSuccess) return e2;
      stt = fa.numRegs == SplitShape::kRegsLaunch ? 1 : 2;
      rd.store(stt);
    }
    if (stt != 1) return cudaErrorInvalidKernelImage;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(SplitShape::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ev0 ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t *>(aplane), bp, bs,
                              static_cast<const float *>(invp), nt, h->od, nb32, static_cast<int>(n_tt), n_ot, Y, w,
                              static_cast<const uint8_t *>(h->b0plane), p.kp, p.n_full, part, cnt);
  };
  // pieces of one token tile of at most 32 tokens: the stages' activation
  // regions hold only those rows, so twice as many stages fit in the ring and
  // go out before the wait for the quantization kernel
  const bool small = p.kp > 1 && !wide && p.n_full == 0 && n_tt == 1 && p.rows <= SplitSmem<true, false, false, true>::kSmallRows;
  if (p.kp > 1 && wide)  // (q6_K only: the plan keeps q4_K's 256-row tiles whole)
    e = go(mmq_gemm_split_kernel<false, true, false, true>, SplitSmem<false, true>::kBytes, 9);
  else if (small)
    e = q4 ? go(mmq_gemm_split_kernel<true, false, false, true, true>, SplitSmem<true, false, false, true>::kBytes, 10)
           : go(mmq_gemm_split_kernel<false, false, false, true, true>, SplitSmem<false, false, false, true>::kBytes,
                11);
  else if (p.kp > 1)
    e = q4 ? go(mmq_gemm_split_kernel<true, false, false, true>, SplitSmem<true, false>::kBytes, 6)
           : go(mmq_gemm_split_kernel<false, false, false, true>, SplitSmem<false, false>::kBytes, 7);
  else if (q4)
    e = wide ? go(mmq_gemm_split_kernel<true, true, false>, SplitSmem<true, true>::kBytes, 3)
             : go(mmq_gemm_split_kernel<true, false, false>, SplitSmem<true, false>::kBytes, 0);
  else if (h->b0plane)
    e = wide ? go(mmq_gemm_split_kernel<false, true, true>, SplitSmem<false, true, true>::kBytes, 5)
             : go(mmq_gemm_split_kernel<false, false, true>, SplitSmem<false, false, true>::kBytes, 4);
  else
    e = wide ? go(mmq_gemm_split_kernel<false, true, false>, SplitSmem<false, true>::kBytes, 1)
             : go(mmq_gemm_split_kernel<false, false, false>, SplitSmem<false, false>::kBytes, 2);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) == cudaSuccess && ev1) e = cudaEventRecordWithFlags(ev1, s, ev_flags);
  return e;
}

cudaError_t launch_wait_selftest(DevStatus *st, unsigned epoch, uint64_t limit_ns,
                                 cudaStream_t s) {
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  wait_selftest_kernel<<<1, 32, 0, s>>>(w);
  return cudaGetLastError();
}

}  // namespace mmq
