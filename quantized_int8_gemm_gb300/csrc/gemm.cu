// gemm.cu -- the k-quant x q8_0 MMQ GEMM on sm_103a tensor cores.
//
// The contraction the pages run on int8 IMMA ("25 · r20: Split-phase A
// staging", §2.2: one m16n8k32 per 4096 MACs) runs here on tcgen05 UMMA of
// kind::f16.  sm_103a has no kind::i8, so the integers travel as fp16:
//   A = qs in [-127, 127]           exact in fp16,
//   B = sc*(q-32) (q6_K, |sc| <= 64) or sc*q (q4_K), |B| <= 2048, exact,
// and every product is exact in the fp32 accumulator.  A 32-element chunk
// sums to at most 32 * 127 * 2048 < 2^24, so the per-chunk partial
//   S[t][o][c] = sum_{k in c} qs[t][k] * B[o][k]
// lands in TMEM exactly -- the pages' "integer sub-block dot product" with
// the sub-block scale already applied.  The epilogue rescales each chunk:
//   q6_K:  Y += da[t][c] * d[o][sb] * S
//   q4_K:  Y += da[t][c] * d[o][sb] * S  -  da[t][c]*ssum[t][c] * dmin*m[o][c]
// (the q4_K min term through ssum, the reason the pad40 block carries it).
//
// Kernel shape: one 128-token x 128-row output tile per CTA, 192 threads.
//   warp 0      TMA producer: A (fp16 activations), B (fp16 operand plane),
//               d / dmin*m scale rows, into a 4-stage ring of 64-K stages
//   warp 1      TMEM owner + single-thread UMMA issuer: per 32-K chunk two
//               128x128x16 UMMAs into one of two TMEM partial buffers
//   warps 2..5  epilogue: TMEM -> registers, per-chunk rescale into fp32
//               accumulators (one token row per thread), then the store
// Every wait is bounded (see ptx.cuh); a CTA that gives up drains its own
// TMA copies and UMMAs, frees TMEM and returns.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

constexpr int BM = 128;  // tokens per tile   (UMMA M, TMEM lanes)
constexpr int BN = 128;  // weight rows per tile (UMMA N, TMEM columns)
constexpr int BK = 64;   // K per pipeline stage: one 128-byte swizzle row of fp16
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 2 * BN;  // two per-chunk partial buffers

constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int D_BYTES = BN * 4;
constexpr int MM_BYTES = 2 * BN * 4;

constexpr int A_OFF = 0;
constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
constexpr int D_OFF = B_OFF + STAGES * B_BYTES;
constexpr int MM_OFF = D_OFF + STAGES * D_BYTES;
constexpr int BAR_OFF = MM_OFF + STAGES * MM_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr int SLOT_OFF = BAR_OFF + NUM_BARS * 8;
constexpr int SMEM_USED = SLOT_OFF + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment

static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// pad40 -> fp16 operand a16[t][k] = qs, and per (t, c) {da, da*ssum}.
__global__ void __launch_bounds__(256) gemm_prepass_kernel(const uint8_t *__restrict__ Q,
                                                           int64_t nblocks,
                                                           __half *__restrict__ a16,
                                                           float2 *__restrict__ sc) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  const uint2 *src = reinterpret_cast<const uint2 *>(Q + b * MMQ_Q8_BLOCK_BYTES);
  const uint2 w0 = __ldg(src + 0), w1 = __ldg(src + 1), w2 = __ldg(src + 2),
              w3 = __ldg(src + 3), w4 = __ldg(src + 4);
  // byte 0..1 d16 | 4..35 qs | 36..39 ssum
  const uint32_t qw[8] = {w0.y, w1.x, w1.y, w2.x, w2.y, w3.x, w3.y, w4.x};
  uint4 *dst = reinterpret_cast<uint4 *>(a16 + b * 32);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half h[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w = qw[2 * i + (j >> 2)];
      h[j] = __int2half_rn(static_cast<int8_t>((w >> (8 * (j & 3))) & 0xFF));
    }
    dst[i] = *reinterpret_cast<const uint4 *>(h);
  }
  const float da = __half2float(__ushort_as_half(static_cast<unsigned short>(w0.x & 0xFFFFu)));
  const int ssum = static_cast<int>(w4.y);
  sc[b] = make_float2(da, da * static_cast<float>(ssum));  // exact: 11 x 13 bits
}

template <bool kQ4K>
__global__ void __launch_bounds__(THREADS, 1)
    mmq_gemm_f16_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_d,
                        const __grid_constant__ CUtensorMap tm_mm, const float2 *__restrict__ sc,
                        int64_t nt, int64_t od, int64_t nb32, float *__restrict__ Y,
                        WaitCtl wctl) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t o0 = static_cast<int64_t>(blockIdx.x) * BN;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * BM;
  const int nkb = static_cast<int>(nb32 / 2);

  const uint32_t bar = base + BAR_OFF;
  auto full = [&](int s) { return bar + 8u * s; };
  auto empty = [&](int s) { return bar + 8u * (STAGES + s); };
  auto tfull = [&](int b) { return bar + 8u * (2 * STAGES + b); };
  auto tempty = [&](int b) { return bar + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done = bar + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1 + EPI_WARPS);  // UMMA commit + epilogue warps (scale reads)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), EPI_WARPS);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_d);
    if (kQ4K) tma_prefetch_desc(&tm_mm);
  }
  if (warp == 1) {
    tmem_alloc(base + SLOT_OFF, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + SLOT_OFF);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      constexpr uint32_t kTx = A_BYTES + B_BYTES + D_BYTES + (kQ4K ? MM_BYTES : 0);
      int issued = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(empty(s), ((kb / STAGES) & 1) ^ 1, wctl)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full(s), kTx);
        tma_load_2d(base + A_OFF + s * A_BYTES, &tm_a, full(s), kb * BK, static_cast<int>(t0));
        tma_load_2d(base + B_OFF + s * B_BYTES, &tm_b, full(s), kb * BK, static_cast<int>(o0));
        tma_load_2d(base + D_OFF + s * D_BYTES, &tm_d, full(s), static_cast<int>(o0), kb / 4);
        if (kQ4K)
          tma_load_2d(base + MM_OFF + s * MM_BYTES, &tm_mm, full(s), static_cast<int>(o0), kb * 2);
        issued = kb + 1;
      }
      if (!ok)  // drain the copies still in flight before the CTA exits
        for (int kb = issued > STAGES ? issued - STAGES : 0; kb < issued; ++kb)
          mbar_wait(full(kb % STAGES), (kb / STAGES) & 1, wctl, false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(full(s), (kb / STAGES) & 1, wctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_s = base + A_OFF + s * A_BYTES;
        const uint32_t b_s = base + B_OFF + s * B_BYTES;
        for (int h = 0; h < 2; ++h) {
          const int c = kb * 2 + h, buf = c & 1;
          if (!mbar_wait(tempty(buf), ((c >> 1) & 1) ^ 1, wctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint32_t koff = (h * 2 + kk) * 32;  // 16 fp16 of K per UMMA
            umma_f16(tbase + buf * BN, sdesc_kmajor_sw128(a_s + koff),
                     sdesc_kmajor_sw128(b_s + koff), idesc, kk);
          }
          umma_commit(tfull(buf));
        }
        if (ok) umma_commit(empty(s));
      }
      umma_commit(done);  // every UMMA of this CTA has finished once `done` flips
      mbar_wait(done, 0, wctl, false);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const int64_t t = t0 + row;
    const bool trow = t < nt;
    const float2 *scrow = sc + (trow ? t : 0) * nb32;
    const uint32_t trow_addr = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    float acc[BN];
#pragma unroll
    for (int j = 0; j < BN; ++j) acc[j] = 0.f;
    float2 s_cur = trow ? __ldg(scrow) : make_float2(0.f, 0.f);
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % STAGES;
      ok = __all_sync(0xffffffffu, mbar_wait(full(s), (kb / STAGES) & 1, wctl));
      if (!ok) break;
      const float *dsc = reinterpret_cast<const float *>(smem + D_OFF + s * D_BYTES);
      const float *mm = reinterpret_cast<const float *>(smem + MM_OFF + s * MM_BYTES);
      for (int h = 0; h < 2; ++h) {
        const int c = kb * 2 + h, buf = c & 1;
        const float2 s_nxt =
            (trow && c + 1 < nb32) ? __ldg(scrow + c + 1) : make_float2(0.f, 0.f);
        ok = __all_sync(0xffffffffu, mbar_wait(tfull(buf), (c >> 1) & 1, wctl));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cb = 0; cb < BN / 32; ++cb) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(trow_addr + buf * BN + cb * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = cb * 32 + j;
            float a = acc[col];
            if (kQ4K) a = fmaf(-s_cur.y, mm[h * BN + col], a);
            acc[col] = fmaf(s_cur.x * dsc[col], __uint_as_float(r[j]), a);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(buf));
        s_cur = s_nxt;
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));
    }
    if (ok && trow) {
      float *yrow = Y + t * od + o0;
      if ((od & 3) == 0) {
#pragma unroll
        for (int j = 0; j < BN; j += 4)
          if (o0 + j < od)
            *reinterpret_cast<float4 *>(yrow + j) =
                make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < BN; ++j)
          if (o0 + j < od) yrow[j] = acc[j];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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

}  // namespace

cudaError_t launch_gemm_prepass(const uint8_t *Q, int64_t nt, int64_t id, void *a16, void *sc,
                                cudaStream_t s) {
  const int64_t nblocks = nt * (id / 32);
  const int bs = 256;
  gemm_prepass_kernel<<<static_cast<unsigned>((nblocks + bs - 1) / bs), bs, 0, s>>>(
      Q, nblocks, static_cast<__half *>(a16), static_cast<float2 *>(sc));
  return cudaGetLastError();
}

cudaError_t launch_gemm_f16(const mmq_weights_s *h, const CUtensorMap &tm_a, const void *sc,
                            int64_t nt, float *Y, DevStatus *st, unsigned epoch,
                            uint64_t limit_ns, cudaStream_t s) {
  const bool q4 = h->type == MMQ_Q4_K;
  auto kern = q4 ? mmq_gemm_f16_kernel<true> : mmq_gemm_f16_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(h->od_pad / BN), static_cast<unsigned>((nt + BM - 1) / BM));
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  kern<<<grid, THREADS, SMEM_BYTES, s>>>(tm_a, h->tm_b, h->tm_d, q4 ? h->tm_mm : h->tm_d,
                                         static_cast<const float2 *>(sc), nt, h->od, h->nb32, Y,
                                         w);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(DevStatus *st, unsigned epoch, uint64_t limit_ns,
                                 cudaStream_t s) {
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  wait_selftest_kernel<<<1, 32, 0, s>>>(w);
  return cudaGetLastError();
}

}  // namespace mmq
