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
// super-block one K=16 UMMA of  g' = da*ssum*2^s_t  split exactly into fp16
// hi + lo  against the integer mins m  (MIN above); s_t is a per-token power
// of two that keeps g' in fp16 range, and da' = da*2^s_t carries the same
// factor so the final scaling by 2^-s_t is exact.
//
// Data movement: operands arrive pre-tiled and pre-swizzled (tiling.h), two
// bulk copies per 128-K stage (activation block, weight block with its scale
// rows), issued by two lanes of the producer warp into a 3-stage ring.
//
// Kernel shape: persistent, one CTA of 384 threads per SM, 128 x 128 tiles,
// token tiles fastest so concurrently running CTAs share weight tiles in L2.
//   warps 0..7  epilogue: warp w reads TMEM lanes 32*(w%4).. and columns
//               64*(w/4)..: TMEM -> registers -> packed fp32x2 FMAs
//   warp 8      producer: lane 0 the activation block, lane 1 the weight block
//   warp 9      TMEM owner + UMMA issuer (one elected lane of a warp-uniform
//               loop): per 32-K chunk two 128x128x16 UMMAs; chunks go in pairs
//               into a ring of two TMEM slot pairs, one commit per pair
//               (+ the min-term UMMA per q4_K super-block, in a pair of its own)
//   warps 10-11 idle (complete the register-donating warpgroup)
// Every wait is bounded (ptx.cuh); a CTA that gives up drains its own copies
// and UMMAs, frees TMEM and returns.
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tiling.h"

namespace mmq {
namespace {

using namespace tiling;

constexpr int STAGES = 3;
constexpr int RING = 2;  // TMEM slot pairs, 2 x kTileN columns each (one hand-off per 2 chunks)
constexpr int EPI_WARPS = 8;     // warpgroups 0 and 1
constexpr int PRODUCER_WARP = 8;  // warpgroup 2: producer, UMMA issuer, two idle warps
constexpr int MMA_WARP = 9;
constexpr int THREADS = 384;
// Register split: launched at 168 per thread (384 x 168 = 64512); warpgroup 2
// drops to 56 and the epilogue warpgroups rise to 216: 2*128*216 + 128*56 =
// 62464 <= 64512.
constexpr int REGS_EPI = 216;
constexpr int REGS_CTL = 56;
constexpr int TMEM_COLS = RING * 2 * kTileN;  // 512

template <bool kQ4>
struct Smem {
  static constexpr int kA = a_odd_bytes(kQ4);                          // A region per stage
  static constexpr int kB = ((b_odd_bytes(kQ4) + 1023) / 1024) * 1024;  // B region per stage
  static constexpr int kStage = kA + kB;
  static constexpr int kBar = STAGES * kStage;
  static constexpr int kNumBars = 2 * STAGES + 2 * RING + 1;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kUsed = kSlot + 16;
  static constexpr int kBytes = kUsed + 1024;  // slack for 1024-byte alignment
  static_assert(kA % 1024 == 0 && kStage % 1024 == 0, "stage buffers must keep 1 KB alignment");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t cnt) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(cnt) : "memory");
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
                                                           float *__restrict__ invp) {
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x;
  const uint8_t *qrow = Q + t * nb32 * MMQ_Q8_BLOCK_BYTES;
  const int64_t nsb = nb32 / 8;
  int s = 0;
  if (kQ4) {  // s_t: the token's largest |g| lands in [2^14, 2^15)
    __shared__ float wmax[4];
    float gmax = 0.f;
    for (int64_t c = tid; c < nb32; c += 128) {
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
    const uint2 w0 = __ldg(src + 0), w1 = __ldg(src + 1), w2 = __ldg(src + 2),
                w3 = __ldg(src + 3), w4 = __ldg(src + 4);
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

// ---------------------------------------------------------------- the GEMM
template <bool kQ4>
__global__ void __launch_bounds__(THREADS, 1)
    mmq_gemm_kernel(const uint8_t *__restrict__ aplane, const uint8_t *__restrict__ bplane,
                    const float *__restrict__ dap, const float *__restrict__ invp, int64_t nt,
                    int64_t od, int64_t nb32, int n_tt, int n_ot, float *__restrict__ Y,
                    WaitCtl wctl) {
  using L = Smem<kQ4>;
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
  auto rfull = [&](int i) { return bar + 8u * (2 * STAGES + i); };
  auto rempty = [&](int i) { return bar + 8u * (2 * STAGES + RING + i); };
  const uint32_t done = bar + 8u * (2 * STAGES + 2 * RING);
  auto a_smem = [&](int s) { return base + s * L::kStage; };
  auto b_smem = [&](int s) { return base + s * L::kStage + L::kA; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1 + EPI_WARPS);  // UMMA commit + 8 epilogue arrivals (scale reads)
    }
    for (int i = 0; i < RING; ++i) {
      mbar_init(rfull(i), 1);
      mbar_init(rempty(i), EPI_WARPS);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(base + L::kSlot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + L::kSlot);
  if (warp >= PRODUCER_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTL));
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (warp-uniform control flow); lane 0 copies
    // the activation block, lane 1 the weight block.
    uint32_t ks = 0, issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int tt = tile % n_tt, ot = tile / n_tt;
      for (int64_t sb = 0; sb < nsb && ok; ++sb) {
        for (int half = 0; half < 2; ++half, ++ks) {
          const int s = static_cast<int>(ks % STAGES);
          ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ((ks / STAGES) & 1) ^ 1, wctl));
          if (!ok) break;
          const uint32_t ab = half ? a_odd_bytes(kQ4) : a_even_bytes();
          const uint32_t bb = half ? b_odd_bytes(kQ4) : b_even_bytes();
          if (lane == 0) {
            mbar_arrive_expect_tx(full(s), ab + bb);
            bulk_load(a_smem(s), aplane + a_block(tt, sb, half, nsb, kQ4), ab, full(s));
          } else if (lane == 1) {
            bulk_load(b_smem(s), bplane + b_block(ot, sb, half, nsb, kQ4), bb, full(s));
          }
          __syncwarp();
          issued = ks + 1;
        }
      }
    }
    if (!ok)  // drain this CTA's copies still in flight
      for (uint32_t k = issued > STAGES ? issued - STAGES : 0; k < issued; ++k)
        mbar_wait(full(k % STAGES), (k / STAGES) & 1, wctl, false);
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp runs the loop and waits; one elected lane issues the
    // UMMAs and commits (keeps the issue path warp-uniform).  Chunks go in
    // pairs into a ring of two slot pairs: one hand-off per 64 of K.
    uint32_t elected;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(elected));
    constexpr uint32_t idesc = idesc_f16_f32(kTileM, kTileN);
    constexpr uint64_t kStageDesc = L::kStage >> 4;  // descriptor address field step per stage
    const uint64_t a0 = sdesc_kmajor_sw128(a_smem(0)), b0 = sdesc_kmajor_sw128(b_smem(0));
    const uint64_t am0 = sdesc_kmajor_sw32(a_smem(0) + kAMin), bm0 = sdesc_kmajor_sw32(b_smem(0) + kBMin);
    uint32_t ks = 0, p = 0;
    bool ok = true;
    auto next_pair = [&](uint32_t &ps) {
      ps = p % RING;
      const bool got = __all_sync(0xffffffffu, mbar_wait(rempty(ps), ((p / RING) & 1) ^ 1, wctl));
      if (got) tc_fence_after();
      return got;
    };
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      for (int64_t sb = 0; sb < nsb && ok; ++sb) {
        for (int half = 0; half < 2 && ok; ++half, ++ks) {
          const int s = static_cast<int>(ks % STAGES);
          ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
          if (!ok) break;
          tc_fence_after();
          const uint64_t as = a0 + s * kStageDesc, bs = b0 + s * kStageDesc;
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {
            uint32_t ps;
            if (!(ok = next_pair(ps))) break;
            if (elected) {
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * cp + cc;  // chunk in the stage: K = 32c .. 32c+31
                const uint64_t off = (c >> 1) * (16384 >> 4) + (c & 1) * (64 >> 4);
                const uint32_t d = tbase + (ps * 2 + cc) * kTileN;
                umma_f16(d, as + off, bs + off, idesc, 0);
                umma_f16(d, as + off + 2, bs + off + 2, idesc, 1);
              }
              umma_commit(rfull(ps));
            }
            __syncwarp();
            ++p;
          }
          if (ok && kQ4 && half == 1) {
            uint32_t ps;
            if ((ok = next_pair(ps))) {
              if (elected) {
                umma_f16(tbase + ps * 2 * kTileN, am0 + s * kStageDesc, bm0 + s * kStageDesc, idesc, 0);
                umma_commit(rfull(ps));
              }
              __syncwarp();
              ++p;
            }
          }
          if (!ok) break;
          if (elected) {
            umma_commit(empty(s));
            if (half == 0) mbar_arrive_cnt(empty(s), EPI_WARPS);  // epilogue reads odd stages only
          }
          __syncwarp();
        }
      }
    }
    if (elected) umma_commit(done);  // every UMMA of this CTA has finished once `done` flips
    mbar_wait(done, 0, wctl, false);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_EPI));
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int chalf = warp >> 2;  // column half 0 / 1
    const int row = quad * 32 + lane;
    const uint32_t taddr = tbase + (static_cast<uint32_t>(quad * 32) << 16) + chalf * 64;
    uint32_t ks = 0, u = 0;
    bool ok = true;
    // Wait for the next slot pair; false (after recording) if the wait expired.
    auto acquire = [&](uint32_t &ps) {
      ps = u % RING;
      const bool got = __all_sync(0xffffffffu, mbar_wait(rfull(ps), (u / RING) & 1, wctl));
      if (got) tc_fence_after();
      return got;
    };
    auto release = [&](uint32_t ps) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty(ps));
      ++u;
    };
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int tt = tile % n_tt, ot = tile / n_tt;
      const int64_t t = static_cast<int64_t>(tt) * kTileM + row;  // < nt_pad: planes are padded
      const int64_t o0 = static_cast<int64_t>(ot) * kTileN + chalf * 64;
      float2 y[32], acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) y[j] = make_float2(0.f, 0.f);
      const float4 *darow = reinterpret_cast<const float4 *>(dap + t * nb32);
      for (int64_t sb = 0; sb < nsb && ok; ++sb) {
        const float4 d0 = __ldg(darow + 2 * sb), d1 = __ldg(darow + 2 * sb + 1);
        const float das[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        // Four 32-column quarters per slot pair (chunk c then c+1, low then
        // high columns), software-pipelined: the load of quarter q+1 is in
        // flight while quarter q is folded into acc.
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
          uint32_t ps;
          if (!(ok = acquire(ps))) break;
          uint32_t r[2][32];
          tmem_ld_32x32b_x32(taddr + (ps * 2) * kTileN, r[0]);
          tmem_wait_ld(r[0]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q < 3)
              tmem_ld_32x32b_x32(taddr + (ps * 2 + ((q + 1) >> 1)) * kTileN + ((q + 1) & 1) * 32,
                                 r[(q + 1) & 1]);
            const int cc = c + (q >> 1);
            const float2 da2 = make_float2(das[cc], das[cc]);
            const uint32_t(&v)[32] = r[q & 1];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 x = make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
              float2 &a = acc[(q & 1) * 16 + j];
              a = cc == 0 ? fmul2(da2, x) : ffma2(da2, x, a);
            }
            if (q < 3) tmem_wait_ld(r[(q + 1) & 1]);
            if (q == 2) release(ps);  // every quarter of the pair is in registers
          }
        }
        if (!ok) break;
        ks += 1;  // the even stage of this super-block; the odd one holds d (and dmin)
        const int s = static_cast<int>(ks % STAGES);
        ok = __all_sync(0xffffffffu, mbar_wait(full(s), (ks / STAGES) & 1, wctl));
        if (!ok) break;
        const float *bsm = reinterpret_cast<const float *>(smem + s * L::kStage + L::kA);
        const float2 *d2 = reinterpret_cast<const float2 *>(bsm + kBD / 4 + chalf * 64);
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = ffma2(d2[j], acc[j], y[j]);
        if (kQ4) {
          uint32_t ps;
          if (!(ok = acquire(ps))) break;
          const float2 *dm2 = reinterpret_cast<const float2 *>(bsm + kBDmin / 4 + chalf * 64);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ps * 2 * kTileN + hh * 32, r);
            tmem_wait_ld(r);
            if (hh == 1) release(ps);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 dm = dm2[hh * 16 + j];
              y[hh * 16 + j] = ffma2(make_float2(-dm.x, -dm.y),
                                     make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])),
                                     y[hh * 16 + j]);
            }
          }
        }
        // the stage's scale rows were read through the generic proxy; order
        // those reads before the TMA (async proxy) that refills the buffer
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        ks += 1;
      }
      if (!ok) break;
      if (t < nt) {
        const float inv = __ldg(invp + t);
        const float2 inv2 = make_float2(inv, inv);
        float *yrow = Y + t * od + o0;
        if ((od & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            if (o0 + 2 * j < od) {
              const float2 a = fmul2(y[j], inv2), b = fmul2(y[j + 1], inv2);
              *reinterpret_cast<float4 *>(yrow + 2 * j) = make_float4(a.x, a.y, b.x, b.y);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float2 a = fmul2(y[j], inv2);
            if (o0 + 2 * j < od) yrow[2 * j] = a.x;
            if (o0 + 2 * j + 1 < od) yrow[2 * j + 1] = a.y;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
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

int g_num_sms[64];

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

size_t gemm_scratch_bytes(int type, int64_t nt, int64_t id) {
  const bool q4 = type == MMQ_Q4_K;
  const int64_t n_tt = (nt + kTileM - 1) / kTileM, nt_pad = n_tt * kTileM;
  const int64_t nsb = id / MMQ_QK, nb32 = id / 32;
  const size_t a = static_cast<size_t>(n_tt * nsb) * a_pair_bytes(q4);
  const size_t da = static_cast<size_t>(nt_pad * nb32) * 4;
  const size_t inv = static_cast<size_t>(nt_pad) * 4;
  return ((a + 255) / 256 + (da + 255) / 256 + (inv + 255) / 256) * 256;
}

cudaError_t launch_gemm(const mmq_weights_s *h, const uint8_t *Q, int64_t nt, float *Y,
                        void *scratch, DevStatus *st, unsigned epoch, uint64_t limit_ns,
                        cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, unsigned ev_flags) {
  const bool q4 = h->type == MMQ_Q4_K;
  const int64_t n_tt = (nt + kTileM - 1) / kTileM, nt_pad = n_tt * kTileM;
  const int64_t nsb = h->nsb, nb32 = h->nb32;
  const size_t a_bytes = static_cast<size_t>(n_tt * nsb) * a_pair_bytes(q4);
  uint8_t *aplane = static_cast<uint8_t *>(scratch);
  float *dap = reinterpret_cast<float *>(aplane + (a_bytes + 255) / 256 * 256);
  float *invp = dap + ((static_cast<size_t>(nt_pad * nb32) * 4 + 255) / 256 * 64);

  // the last token tile's padding rows must read as zero
  cudaError_t e = cudaSuccess;
  if (nt_pad != nt) {
    const uint64_t tail = static_cast<uint64_t>((n_tt - 1) * nsb) * a_pair_bytes(q4);
    e = cudaMemsetAsync(aplane + tail, 0, a_bytes - tail, s);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(dap + nt * nb32, 0, static_cast<size_t>((nt_pad - nt) * nb32) * 4, s);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(invp + nt, 0, static_cast<size_t>(nt_pad - nt) * 4, s);
    if (e != cudaSuccess) return e;
  }
  const unsigned pgrid = static_cast<unsigned>(nt);
  if (q4)
    gemm_prepass_kernel<true><<<pgrid, 128, 0, s>>>(Q, nt, nb32, aplane, dap, invp);
  else
    gemm_prepass_kernel<false><<<pgrid, 128, 0, s>>>(Q, nt, nb32, aplane, dap, invp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  auto kern = q4 ? mmq_gemm_kernel<true> : mmq_gemm_kernel<false>;
  const int smem = q4 ? Smem<true>::kBytes : Smem<false>::kBytes;
  // the shared-memory opt-in and the SM count are read once per device,
  // outside any stream capture the first call is not part of
  static std::atomic<uint32_t> attr_done[64][2];
  const int dev = h->device;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev][q4].load()) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr_done[dev][q4].store(1);
  }
  const int n_ot = static_cast<int>(h->od_pad / kTileN);
  const int n_tiles = static_cast<int>(n_tt) * n_ot;
  const int grid = n_tiles < g_num_sms[dev] ? n_tiles : g_num_sms[dev];
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  if (ev0 && (e = cudaEventRecordWithFlags(ev0, s, ev_flags)) != cudaSuccess) return e;
  kern<<<grid, THREADS, smem, s>>>(aplane, static_cast<const uint8_t *>(h->bplane), dap, invp, nt,
                                   h->od, nb32, static_cast<int>(n_tt), n_ot, Y, w);
  e = cudaGetLastError();
  if (e == cudaSuccess && ev1) e = cudaEventRecordWithFlags(ev1, s, ev_flags);
  return e;
}

cudaError_t launch_wait_selftest(DevStatus *st, unsigned epoch, uint64_t limit_ns,
                                 cudaStream_t s) {
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  wait_selftest_kernel<<<1, 32, 0, s>>>(w);
  return cudaGetLastError();
}

}  // namespace mmq
