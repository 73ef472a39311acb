// quantize.cu -- fp32 activations -> q8_0 "pad40" blocks.
//
// Block (t, c) of 32 values, at byte (t*nb32 + c)*40 (the pad40 plane of
// "26 · r21 — Coalesced block-linear A staging", §2.1):
//   d = amax/127 (fp32, IEEE division), q_i = roundf(x_i / d) (half away
//   from zero), stored d16 = fp16_rn(d), bytes [2,4) = 0, ssum = sum q_i
//   (q8.cuh holds the rule, shared with the GEMM's quantizing prepasses).
//
// HBM-bound: 128 B read and 40 B written per block.  Eight lanes share a
// block, each loading one float4 and storing one 4-byte qs word; lane 0 of
// the eight also writes the d word and ssum.
#include <cuda_fp16.h>

#include "internal.h"
#include "q8.cuh"

namespace mmq {
namespace {

// One 32-value block handled by 8 lanes (one float4 each), the rule of q8.cuh.
__device__ __forceinline__ void quantize_block(float4 v, int64_t blk, bool valid, int part,
                                               uint8_t *__restrict__ Q) {
  float d16f, q[4];
  q8_lane(v, d16f, q);
  const float ssum = q8_ssum(q);
  if (!valid) return;
  uint8_t *b = Q + blk * MMQ_Q8_BLOCK_BYTES;
  const uint32_t word = (static_cast<uint32_t>(static_cast<int>(q[0])) & 0xFFu) |
                        ((static_cast<uint32_t>(static_cast<int>(q[1])) & 0xFFu) << 8) |
                        ((static_cast<uint32_t>(static_cast<int>(q[2])) & 0xFFu) << 16) |
                        (static_cast<uint32_t>(static_cast<int>(q[3])) << 24);
  reinterpret_cast<uint32_t *>(b + MMQ_Q8_QS_OFF)[part] = word;
  if (part == 0) {
    *reinterpret_cast<uint32_t *>(b + MMQ_Q8_D_OFF) = __half_as_ushort(__float2half_rn(d16f));  // d16 | zero pad
    *reinterpret_cast<int32_t *>(b + MMQ_Q8_SSUM_OFF) = static_cast<int>(ssum);
  }
}

// Grid-stride over groups of 16 blocks per warp: the four float4 loads of a
// lane are issued before any block is reduced, so each lane keeps 64 B of
// loads in flight.
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float4 *__restrict__ X,
                                                            int64_t nblocks,
                                                            uint8_t *__restrict__ Q) {
  const int lane = threadIdx.x & 31, part = lane & 7, grp = lane >> 3;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp * 16; base < nblocks; base += nwarps * 16) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t blk = base + u * 4 + grp;
      v[u] = blk < nblocks ? __ldg(X + blk * 8 + part) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t blk = base + u * 4 + grp;
      quantize_block(v[u], blk, blk < nblocks, part, Q);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_q8_0(const float *X, int64_t nt, int64_t id, uint8_t *Q,
                                 cudaStream_t s) {
  const int64_t nblocks = nt * (id / 32);
  if (nblocks == 0) return cudaSuccess;
  const int bs = 256;  // 8 warps, 128 blocks per CTA pass
  const int64_t want = (nblocks + 127) / 128;
  const int64_t grid = want < 152 * 16 ? want : 152 * 16;
  quantize_q8_0_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(
      reinterpret_cast<const float4 *>(X), nblocks, Q);
  return cudaGetLastError();
}

}  // namespace mmq
