// register.cu -- one-time expansion of packed k-quant weights.
//
// The pages move the q6_K recombination out of the GEMM loop into a
// registration-time plane ("46 · r43 — PC-sampling attribution", §3.2; the
// dense layout contract of "47 · r44 — W_exp stride mismatch root cause",
// §2.2).  Here registration writes, per weight element (o, k):
//   b16[o][k]      fp16 operand with the sub-block scale folded in
//                  q6_K: sc[k/16] * (q - 32)   (|.| <= 64*32, exact in fp16)
//                  q4_K: sc[k/32] * q          (<= 63*15, exact in fp16)
//   wexp[o*id + k] int8 q - 32 (q6_K, optional): the pages' dense W_exp,
//                  row pitch id, super-block pitch 256
// and per block the fp32 scale planes dplane[sb][o] = d and (q4_K)
// mmplane[sb*8 + j][o] = dmin * m_j.
//
// One CTA of 256 threads per packed block, thread e = element e.
#include <cuda_fp16.h>

#include "internal.h"

namespace mmq {
namespace {

// q6_K element e: low nibble from ql[(e/128)*64 + e%64] (nibble (e%128)/64),
// 2-bit high part from qh[(e/128)*32 + e%32] (field (e%128)/32).
__device__ __forceinline__ int q6k_centered(const uint8_t *blk, int e) {
  const int half = e >> 7, r = e & 127;
  const int lo = (blk[MMQ_Q6K_QL_OFF + half * 64 + (r & 63)] >> ((r >> 6) * 4)) & 0xF;
  const int hi = (blk[MMQ_Q6K_QH_OFF + half * 32 + (r & 31)] >> ((r >> 5) * 2)) & 0x3;
  return (lo | (hi << 4)) - 32;
}

// q4_K (ggml layout): 6-bit scale and min of sub-block j.
__device__ __forceinline__ void q4k_scale_min(const uint8_t *s, int j, int &sc, int &m) {
  if (j < 4) {
    sc = s[j] & 63;
    m = s[j + 4] & 63;
  } else {
    sc = (s[j + 4] & 0xF) | ((s[j - 4] >> 6) << 4);
    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

__global__ void __launch_bounds__(256) register_q6k_kernel(
    const uint8_t *__restrict__ W, int64_t od, int64_t id, int64_t od_pad, __half *__restrict__ b16,
    float *__restrict__ dplane, int8_t *__restrict__ wexp, int *__restrict__ bad_scale) {
  __shared__ uint8_t blk[MMQ_Q6K_BLOCK_BYTES + 2];
  const int64_t nsb = id / MMQ_QK;
  const int64_t o = blockIdx.x, sb = blockIdx.y;
  const uint8_t *src = W + (o * nsb + sb) * MMQ_Q6K_BLOCK_BYTES;
  const int e = threadIdx.x;
  if (e < MMQ_Q6K_BLOCK_BYTES) blk[e] = src[e];
  __syncthreads();
  const int c = q6k_centered(blk, e);
  const int sc = static_cast<int8_t>(blk[MMQ_Q6K_SC_OFF + (e >> 4)]);
  const int64_t k = sb * MMQ_QK + e;
  b16[o * id + k] = __int2half_rn(sc * c);
  if (wexp) wexp[o * id + k] = static_cast<int8_t>(c);
  if ((e & 15) == 0 && (sc > 64 || sc < -64)) atomicOr(bad_scale, 1);
  if (e == 0) {
    const __half d = __ushort_as_half(static_cast<unsigned short>(
        blk[MMQ_Q6K_D_OFF] | (blk[MMQ_Q6K_D_OFF + 1] << 8)));
    dplane[sb * od_pad + o] = __half2float(d);
  }
}

__global__ void __launch_bounds__(256) register_q4k_kernel(
    const uint8_t *__restrict__ W, int64_t od, int64_t id, int64_t od_pad, __half *__restrict__ b16,
    float *__restrict__ dplane, float *__restrict__ mmplane) {
  __shared__ uint8_t blk[MMQ_Q4K_BLOCK_BYTES];
  const int64_t nsb = id / MMQ_QK;
  const int64_t o = blockIdx.x, sb = blockIdx.y;
  const uint8_t *src = W + (o * nsb + sb) * MMQ_Q4K_BLOCK_BYTES;
  const int e = threadIdx.x;
  if (e < MMQ_Q4K_BLOCK_BYTES) blk[e] = src[e];
  __syncthreads();
  const int j = e >> 5;
  const int byte = blk[MMQ_Q4K_QS_OFF + 32 * (j >> 1) + (e & 31)];
  const int q = (j & 1) ? (byte >> 4) : (byte & 0xF);
  int sc, m;
  q4k_scale_min(blk + MMQ_Q4K_SC_OFF, j, sc, m);
  b16[o * id + sb * MMQ_QK + e] = __int2half_rn(sc * q);
  if ((e & 31) == 0) {
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(
        blk[MMQ_Q4K_DMIN_OFF] | (blk[MMQ_Q4K_DMIN_OFF + 1] << 8))));
    mmplane[(sb * 8 + j) * od_pad + o] = dmin * static_cast<float>(m);  // exact: 11 x 6 bits
  }
  if (e == 0) {
    dplane[sb * od_pad + o] = __half2float(__ushort_as_half(
        static_cast<unsigned short>(blk[MMQ_Q4K_D_OFF] | (blk[MMQ_Q4K_D_OFF + 1] << 8))));
  }
}

}  // namespace

cudaError_t launch_register(const mmq_weights_s *h, const uint8_t *W, int *bad_scale,
                            cudaStream_t s) {
  // padded rows and padding columns of the scale planes stay zero
  cudaError_t e = cudaMemsetAsync(h->b16, 0, h->b16_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->dplane, 0, h->dplane_bytes, s);
  if (e == cudaSuccess && h->mmplane) e = cudaMemsetAsync(h->mmplane, 0, h->mm_bytes, s);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(h->od), static_cast<unsigned>(h->nsb));
  if (h->type == MMQ_Q6_K) {
    register_q6k_kernel<<<grid, 256, 0, s>>>(W, h->od, h->id, h->od_pad,
                                             static_cast<__half *>(h->b16), h->dplane, h->wexp,
                                             bad_scale);
  } else {
    register_q4k_kernel<<<grid, 256, 0, s>>>(W, h->od, h->id, h->od_pad,
                                             static_cast<__half *>(h->b16), h->dplane,
                                             h->mmplane);
  }
  return cudaGetLastError();
}

}  // namespace mmq
