// probe.cu -- microbenchmarks of the GB300's exact-integer-capable engines,
// the measurements behind the choice of tensor-core kind and of the roofline
// peak (mmq_probe_engine_rates in mmq.h).  Not part of the GEMM.
//
//   umma_rate_kernel<N>  one CTA per SM issues back-to-back tcgen05.mma
//                        kind::f16 (M = 128, N, K = 16) from one warp into one
//                        TMEM accumulator, operands (zeros) in shared memory;
//                        the issuing thread's clock64 over the loop and the
//                        final commit gives clk per UMMA
//   umma_pair_rate_kernel<N>  the same on 2-CTA clusters: the even CTA issues
//                        cta_group::2 UMMAs of M = 256 (128 A rows and N / 2 B
//                        rows in each CTA's shared memory, the rates the pair
//                        arm's tiles of 256 weight rows x N tokens run at)
//   mma_sync_s8_kernel   warp-level mma.sync m16n8k32 s8 -> s32, eight
//                        independent accumulators per warp
//   mma_sync_f16_kernel  warp-level mma.sync m16n8k16 f16 -> f32, likewise
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

constexpr int kUmmaIters = 4096;

// Operands in dynamic shared memory, 1024-byte aligned: A = one 64-K K-block
// of 128 rows (16 KB), B = one of N rows (N * 128 B, read whole by every
// UMMA).  The launch asks for kUmmaSmem bytes so that one CTA runs per SM.
template <int N>
__host__ __device__ constexpr int umma_ops_bytes() { return 16384 + N * 128; }
// TMEM columns for an N-column accumulator: a power of two, at least 32
template <int N>
__host__ __device__ constexpr int tmem_cols() { return N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256; }
constexpr int kUmmaSmem = 120 * 1024;
static_assert(umma_ops_bytes<256>() + 1024 <= kUmmaSmem, "operands fit the request");

template <int N>
__global__ void __launch_bounds__(128, 1) umma_rate_kernel(WaitCtl wctl, long long *clk_per_cta) {
  extern __shared__ uint8_t dyn[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const uint32_t raw = smem_addr(dyn);
  uint8_t *ops = dyn + (((raw + 1023u) & ~1023u) - raw);
  for (int i = threadIdx.x; i < umma_ops_bytes<N>() / 16; i += blockDim.x)
    reinterpret_cast<uint4 *>(ops)[i] = make_uint4(0, 0, 0, 0);
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_addr(&tslot), tmem_cols<N>());
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeroed operands, for the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(&tslot);
  if (threadIdx.x < 32) {
    uint32_t elected;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(elected));
    constexpr uint32_t idesc = idesc_f16_f32(128, N);
    const uint64_t ad = sdesc_kmajor_sw128(smem_addr(ops)), bd = sdesc_kmajor_sw128(smem_addr(ops + 16384));
    long long t0 = 0;
    if (elected) {
      t0 = clock64();
      for (int i = 0; i < kUmmaIters; ++i) umma_f16(tbase, ad + 2 * (i & 3), bd + 2 * (i & 3), idesc, i ? 1u : 0u);
      umma_commit(b);
    }
    __syncwarp();
    const bool ok = mbar_wait(b, 0, wctl, false);
    if (elected) clk_per_cta[blockIdx.x] = ok ? clock64() - t0 : -1;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tbase, tmem_cols<N>());
  }
}

template <int N>
__global__ void __launch_bounds__(128, 1) umma_pair_rate_kernel(WaitCtl wctl, long long *clk_per_pair) {
  extern __shared__ uint8_t dyn[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const uint32_t rank = cluster_ctarank();
  const uint32_t raw = smem_addr(dyn);
  uint8_t *ops = dyn + (((raw + 1023u) & ~1023u) - raw);
  for (int i = threadIdx.x; i < umma_ops_bytes<N / 2>() / 16; i += blockDim.x)
    reinterpret_cast<uint4 *>(ops)[i] = make_uint4(0, 0, 0, 0);
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {  // one warp of each CTA of the pair, together
    tmem_alloc_pair(smem_addr(&tslot), tmem_cols<N>());
    tmem_relinquish_pair();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(&tslot);
  if (threadIdx.x < 32) {
    uint32_t elected;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(elected));
    constexpr uint32_t idesc = idesc_f16_f32(256, N);
    const uint64_t ad = sdesc_kmajor_sw128(smem_addr(ops)), bd = sdesc_kmajor_sw128(smem_addr(ops + 16384));
    long long t0 = 0;
    if (rank == 0 && elected) {
      t0 = clock64();
      for (int i = 0; i < kUmmaIters; ++i) umma_pair_f16(tbase, ad + 2 * (i & 3), bd + 2 * (i & 3), idesc, i ? 1u : 0u);
      umma_pair_commit(b);  // arrives on both CTAs' barrier
    }
    __syncwarp();
    const bool ok = mbar_wait(b, 0, wctl, false);
    if (rank == 0 && elected) clk_per_pair[blockIdx.x >> 1] = ok ? clock64() - t0 : -1;
  }
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the other's UMMAs may still read its operands
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, tmem_cols<N>());
  }
}

constexpr int kMmaIters = 4096;

__global__ void __launch_bounds__(256) mma_sync_s8_kernel(int *out) {
  // operand registers that differ per thread (constant operands let the
  // f16 loop report more than the tensor peak)
  const uint32_t x = threadIdx.x;
  const uint32_t a[4] = {x, x * 3u, x * 5u, x * 7u}, bb[2] = {x * 11u, x * 13u};
  int c[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[j][i] = 0;
  for (int it = 0; it < kMmaIters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(bb[0]), "r"(bb[1]));
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  if (s == 0x7fffffff) out[0] = s;  // keep the loop
}

__global__ void __launch_bounds__(256) mma_sync_f16_kernel(float *out) {
  const uint32_t x = threadIdx.x;  // per-thread operand registers, as above
  const uint32_t a[4] = {x, x * 3u, x * 5u, x * 7u}, bb[2] = {x * 11u, x * 13u};
  float c[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[j][i] = 0.f;
  for (int it = 0; it < kMmaIters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(bb[0]), "r"(bb[1]));
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  if (s == 1234.5f) out[0] = s;  // keep the loop
}

template <typename F>
cudaError_t time_ms(cudaStream_t s, F launch, float *ms) {
  cudaEvent_t e0, e1;
  cudaError_t e = cudaEventCreate(&e0);
  if (e != cudaSuccess) return e;
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
    cudaEventDestroy(e0);
    return e;
  }
  launch();  // warm-up
  e = cudaEventRecord(e0, s);
  launch();
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return e;
}

template <int N>
cudaError_t umma_rate(int sms, WaitCtl w, long long *clk, cudaStream_t s, double *mac_per_clk) {
  cudaError_t e = cudaFuncSetAttribute(umma_rate_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kUmmaSmem);
  if (e != cudaSuccess) return e;
  umma_rate_kernel<N><<<sms, 128, kUmmaSmem, s>>>(w, clk);
  e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  long long *h = new long long[sms];
  e = cudaMemcpy(h, clk, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
  double sum = 0;
  int n = 0;
  for (int i = 0; e == cudaSuccess && i < sms; ++i)
    if (h[i] > 0) {
      sum += static_cast<double>(h[i]);
      ++n;
    }
  delete[] h;
  if (e != cudaSuccess) return e;
  *mac_per_clk = n ? 128.0 * N * 16 * kUmmaIters / (sum / n) : 0.0;
  return cudaSuccess;
}

template <int N>
cudaError_t umma_pair_rate(int sms, WaitCtl w, long long *clk, cudaStream_t s, double *mac_per_clk) {
  auto kern = umma_pair_rate_kernel<N>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kUmmaSmem);
  if (e != cudaSuccess) return e;
  const int pairs = sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * static_cast<unsigned>(pairs));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kUmmaSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, w, clk);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  long long *h = new long long[pairs];
  e = cudaMemcpy(h, clk, sizeof(long long) * pairs, cudaMemcpyDeviceToHost);
  double sum = 0;
  int n = 0;
  for (int i = 0; e == cudaSuccess && i < pairs; ++i)
    if (h[i] > 0) {
      sum += static_cast<double>(h[i]);
      ++n;
    }
  delete[] h;
  if (e != cudaSuccess) return e;
  *mac_per_clk = n ? 256.0 * N * 16 * kUmmaIters / (sum / n) / 2.0 : 0.0;  // per SM of the pair
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_engine_probes(DevStatus *st, unsigned epoch, uint64_t limit_ns, cudaStream_t s, double *out) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  WaitCtl w{&st->status, &st->abort_epoch, epoch, limit_ns};
  long long *clk = nullptr;
  if ((e = cudaMalloc(&clk, sizeof(long long) * sms)) != cudaSuccess) return e;
  e = umma_rate<64>(sms, w, clk, s, &out[0]);
  if (e == cudaSuccess) e = umma_rate<128>(sms, w, clk, s, &out[1]);
  if (e == cudaSuccess) e = umma_rate<256>(sms, w, clk, s, &out[2]);
  if (e == cudaSuccess) e = umma_rate<96>(sms, w, clk, s, &out[5]);
  if (e == cudaSuccess) e = umma_rate<112>(sms, w, clk, s, &out[6]);
  if (e == cudaSuccess) e = umma_pair_rate<64>(sms, w, clk, s, &out[7]);
  if (e == cudaSuccess) e = umma_pair_rate<96>(sms, w, clk, s, &out[8]);
  if (e == cudaSuccess) e = umma_pair_rate<112>(sms, w, clk, s, &out[9]);
  if (e == cudaSuccess) e = umma_pair_rate<128>(sms, w, clk, s, &out[10]);
  if (e == cudaSuccess) e = umma_pair_rate<256>(sms, w, clk, s, &out[11]);
  cudaFree(clk);
  if (e != cudaSuccess) return e;
  int *sink = nullptr;
  if ((e = cudaMalloc(&sink, 16)) != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(sms) * 4;
  const double mmas = static_cast<double>(grid) * 8 /* warps */ * kMmaIters * 8;
  float ms = 0.f;
  e = time_ms(s, [&] { mma_sync_s8_kernel<<<grid, 256, 0, s>>>(sink); }, &ms);
  if (e == cudaSuccess) out[3] = mmas * 2.0 * 16 * 8 * 32 / (ms * 1e-3) / 1e12;
  if (e == cudaSuccess) e = time_ms(s, [&] { mma_sync_f16_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<float *>(sink)); }, &ms);
  if (e == cudaSuccess) out[4] = mmas * 2.0 * 16 * 8 * 16 / (ms * 1e-3) / 1e12;
  cudaFree(sink);
  return e;
}

}  // namespace mmq
