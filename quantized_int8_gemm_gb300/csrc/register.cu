// register.cu -- one-time expansion of packed k-quant weights.
//
// The pages move the q6_K recombination out of the GEMM loop into a
// registration-time plane ("46 · r43 — PC-sampling attribution", §3.2) with
// a dense layout contract ("47 · r44 — W_exp stride mismatch root cause",
// §2.2: element (j, sb, e) at j*id + sb*256 + e).  Registration here writes
// the GEMM's pre-tiled weight plane (tiling.h), per weight element (o, k):
//   operand  fp16  q6_K: sc[k/16] * (q - 32)   (exact while |sc| <= 64)
//                  q4_K: sc[k/32] * q          (<= 63*15, exact)
// A q6_K tensor with some |sc| > 64 (the int8 range allows 128) gets a second
// pass: with c = q - 32, B1 = 2*sc*(c >> 1) (even, |.| <= 4096) in the
// operand plane and B0 = sc*(c & 1) (|.| <= 128) in a second plane of the
// same layout; both are exact fp16 integers and B1 + B0 = sc*c.
// and per (row, super-block) the fp32 scale d, plus for q4_K dmin (both in
// the plane's scale region) and the integer mins m of the eight sub-blocks
// (the min-term image).
//
// With MMQ_REG_WEXP the dense centered-int8 plane wexp[o*id + k] = q - 32 is
// written first and the q6_K operand is then built by reading it back with
// the dense strides, so every GEMM run on such a handle checks the plane's
// offsets (the pages' consumer-side gate), not only its bytes.
//
// One CTA of 256 threads per packed block, thread e = element e.
#include <cuda_fp16.h>

#include "internal.h"
#include "tiling.h"

namespace mmq {
namespace {

using namespace tiling;

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

__device__ __forceinline__ float f16_at(const uint8_t *p) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(p[0] | (p[1] << 8))));
}

// q4_K element e: nibble (e/32)%2 of qs[32*(e/64) + e%32].
__device__ __forceinline__ int q4k_code(const uint8_t *blk, int e) {
  const int j = e >> 5;
  const int byte = blk[MMQ_Q4K_QS_OFF + 32 * (j >> 1) + (e & 31)];
  return (j & 1) ? (byte >> 4) : (byte & 0xF);
}

// dense W_exp plane, element (o, sb*256 + e) at o*id + sb*256 + e: q6_K the
// centered code q - 32, q4_K the code q
template <bool kQ4>
__global__ void __launch_bounds__(256) expand_wexp_kernel(const uint8_t *__restrict__ W,
                                                          int64_t id, int8_t *__restrict__ wexp) {
  constexpr int kBytes = kQ4 ? MMQ_Q4K_BLOCK_BYTES : MMQ_Q6K_BLOCK_BYTES;
  __shared__ uint8_t blk[kBytes + 2];
  const int64_t nsb = id / MMQ_QK;
  const int64_t o = blockIdx.x, sb = blockIdx.y;
  const int e = threadIdx.x;
  if (e < kBytes) blk[e] = W[(o * nsb + sb) * kBytes + e];
  __syncthreads();
  wexp[o * id + sb * MMQ_QK + e] = static_cast<int8_t>(kQ4 ? q4k_code(blk, e) : q6k_centered(blk, e));
}

template <bool kQ4, bool kFromWexp, bool kB0 = false>
__global__ void __launch_bounds__(256) register_kernel(const uint8_t *__restrict__ W,
                                                       const int8_t *__restrict__ wexp, int64_t id,
                                                       uint8_t *__restrict__ bplane,
                                                       uint64_t scale_region,
                                                       int *__restrict__ bad_scale,
                                                       uint8_t *__restrict__ b0plane = nullptr) {
  constexpr int kBytes = kQ4 ? MMQ_Q4K_BLOCK_BYTES : MMQ_Q6K_BLOCK_BYTES;
  __shared__ uint8_t blk[kBytes + 2];
  const int64_t nsb = id / MMQ_QK;
  const int64_t o = blockIdx.x, sb = blockIdx.y;
  const int e = threadIdx.x;
  if (e < kBytes) blk[e] = W[(o * nsb + sb) * kBytes + e];
  __syncthreads();
  const int64_t ot = o / kTileN;
  const int r = static_cast<int>(o % kTileN);
  const int half = e >> 7, k = e & 127;
  uint8_t *dst = bplane + b_block(ot, sb, half, nsb, kQ4);
  uint8_t *odd = bplane + b_block(ot, sb, 1, nsb, kQ4);
  float *scl = reinterpret_cast<float *>(bplane + scale_region + b_scale_block(ot, sb, nsb, kQ4));
  int val;
  float d;
  if constexpr (kQ4) {
    const int j = e >> 5;
    int q;
    if constexpr (kFromWexp) q = wexp[o * id + sb * MMQ_QK + e];  // the dense plane's strides
    else q = q4k_code(blk, e);
    int sc, m;
    q4k_scale_min(blk + MMQ_Q4K_SC_OFF, j, sc, m);
    val = sc * q;
    d = f16_at(blk + MMQ_Q4K_D_OFF);
    if ((e & 31) == 0) {  // min image: slots 2j and 2j+1 both hold m_j
      const uint32_t mh = __half_as_ushort(__int2half_rn(m));
      *reinterpret_cast<uint32_t *>(odd + kBMin + min_off(r, 2 * j)) = mh | (mh << 16);
    }
    if (e == 0) scl[kSDmin / 4 + r] = f16_at(blk + MMQ_Q4K_DMIN_OFF);
  } else {
    int c;
    if constexpr (kFromWexp) c = wexp[o * id + sb * MMQ_QK + e];
    else c = q6k_centered(blk, e);
    const int sc = static_cast<int8_t>(blk[MMQ_Q6K_SC_OFF + (e >> 4)]);
    if (!kB0 && (e & 15) == 0 && (sc > 64 || sc < -64)) atomicOr(bad_scale, 1);
    if constexpr (kB0) {
      val = 2 * sc * (c >> 1);  // arithmetic shift: floor(c / 2)
      *reinterpret_cast<__half *>(b0plane + b_block(ot, sb, half, nsb, false) + operand_off(r, k)) =
          __int2half_rn(sc * (c & 1));
    } else {
      val = sc * c;
    }
    d = f16_at(blk + MMQ_Q6K_D_OFF);
  }
  *reinterpret_cast<__half *>(dst + operand_off(r, k)) = __int2half_rn(val);
  if (e == 0) scl[r] = d;
}

// Raw plane (tiling.h): the packed bytes of row o, super-block sb regrouped
// for the GEMM's in-kernel unpack; scales as fp16.  One CTA per block.
template <bool kQ4>
__global__ void __launch_bounds__(64) register_raw_kernel(const uint8_t *__restrict__ W, int64_t id,
                                                          uint8_t *__restrict__ raw) {
  constexpr int kBytes = kQ4 ? MMQ_Q4K_BLOCK_BYTES : MMQ_Q6K_BLOCK_BYTES;
  __shared__ __align__(8) uint8_t blk[kBytes + 6];
  const int64_t nsb = id / MMQ_QK;
  const int64_t o = blockIdx.x, sb = blockIdx.y;
  const int tid = threadIdx.x;
  for (int i = tid; i < kBytes; i += 64) blk[i] = W[(o * nsb + sb) * kBytes + i];
  __syncthreads();
  const int64_t ot = o / kTileN;
  const int r = static_cast<int>(o % kTileN);
  auto word8 = [&](int off) {  // 8 bytes at byte offset off of the packed block
    uint64_t v = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) v |= static_cast<uint64_t>(blk[off + i]) << (8 * i);
    return v;
  };
  if constexpr (kQ4) {
    // per half: 8 qs words and 4 scales
    if (tid < 16) {
      const int half = tid >> 3, g = tid & 7, kb = g >> 2, j = g & 3;
      uint8_t *dst = raw + raw_block(ot, sb, half, nsb, true);
      reinterpret_cast<uint64_t *>(dst + kRawQ4Qs)[g * 128 + r] =
          word8(MMQ_Q4K_QS_OFF + 64 * half + 32 * kb + 8 * j);
    } else if (tid < 24) {
      const int half = (tid - 16) >> 2, sub = (tid - 16) & 3;
      int sc, m;
      q4k_scale_min(blk + MMQ_Q4K_SC_OFF, 4 * half + sub, sc, m);
      uint8_t *dst = raw + raw_block(ot, sb, half, nsb, true);
      reinterpret_cast<__half *>(dst + kRawQ4Sc)[sub * 128 + r] = __int2half_rn(sc);
    }
  } else {
    // per half: 8 ql words, 4 qh words and 8 scales
    if (tid < 16) {
      const int half = tid >> 3, j = tid & 7;
      uint8_t *dst = raw + raw_block(ot, sb, half, nsb, false);
      reinterpret_cast<uint64_t *>(dst + kRawQ6Ql)[j * 128 + r] = word8(MMQ_Q6K_QL_OFF + 64 * half + 8 * j);
    } else if (tid < 24) {
      const int half = (tid - 16) >> 2, j = (tid - 16) & 3;
      uint8_t *dst = raw + raw_block(ot, sb, half, nsb, false);
      reinterpret_cast<uint64_t *>(dst + kRawQ6Qh)[j * 128 + r] = word8(MMQ_Q6K_QH_OFF + 32 * half + 8 * j);
    } else if (tid < 40) {
      const int half = (tid - 24) >> 3, sub = (tid - 24) & 7;
      const int sc = static_cast<int8_t>(blk[MMQ_Q6K_SC_OFF + 8 * half + sub]);
      uint8_t *dst = raw + raw_block(ot, sb, half, nsb, false);
      reinterpret_cast<__half *>(dst + kRawQ6Sc)[sub * 128 + r] = __int2half_rn(sc);
    }
  }
}

// Dequantization fallback: weight (o, sb*256 + e), exact in fp64, rounded
// once to the output type.  One CTA of 256 threads per block.
template <bool kQ4, typename T>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ W, int64_t id,
                                                      T *__restrict__ out) {
  constexpr int kBytes = kQ4 ? MMQ_Q4K_BLOCK_BYTES : MMQ_Q6K_BLOCK_BYTES;
  __shared__ uint8_t blk[kBytes + 2];
  const int64_t nsb = id / MMQ_QK;
  const int64_t o = blockIdx.x, sb = blockIdx.y;
  const int e = threadIdx.x;
  if (e < kBytes) blk[e] = W[(o * nsb + sb) * kBytes + e];
  __syncthreads();
  double w;
  if constexpr (kQ4) {
    int sc, m;
    q4k_scale_min(blk + MMQ_Q4K_SC_OFF, e >> 5, sc, m);
    const double d = static_cast<double>(f16_at(blk + MMQ_Q4K_D_OFF));
    const double dmin = static_cast<double>(f16_at(blk + MMQ_Q4K_DMIN_OFF));
    w = d * sc * q4k_code(blk, e) - dmin * m;  // both products exact in fp64
  } else {
    const int sc = static_cast<int8_t>(blk[MMQ_Q6K_SC_OFF + (e >> 4)]);
    w = static_cast<double>(f16_at(blk + MMQ_Q6K_D_OFF)) * sc * q6k_centered(blk, e);
  }
  T v;
  if constexpr (sizeof(T) == 2) v = __double2half(w);
  else v = __double2float_rn(w);
  out[o * id + sb * MMQ_QK + e] = v;
}

}  // namespace

cudaError_t launch_dequant(int type, const uint8_t *W, int64_t od, int64_t id, void *out,
                           int out_type, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(od), static_cast<unsigned>(id / MMQ_QK));
  const bool q4 = type == MMQ_Q4_K;
  if (out_type == MMQ_OUT_F16) {
    __half *o = static_cast<__half *>(out);
    if (q4) dequant_kernel<true, __half><<<grid, 256, 0, s>>>(W, id, o);
    else dequant_kernel<false, __half><<<grid, 256, 0, s>>>(W, id, o);
  } else {
    float *o = static_cast<float *>(out);
    if (q4) dequant_kernel<true, float><<<grid, 256, 0, s>>>(W, id, o);
    else dequant_kernel<false, float><<<grid, 256, 0, s>>>(W, id, o);
  }
  return cudaGetLastError();
}

size_t rawplane_bytes(int type, int64_t od, int64_t id) {
  const bool q4 = type == MMQ_Q4_K;
  const int64_t n_ot = (od + kTileN - 1) / kTileN;
  return static_cast<size_t>(n_ot * (id / MMQ_QK) * 2) * raw_block_bytes(q4);
}

size_t bplane_bytes(int type, int64_t od, int64_t id) {
  const bool q4 = type == MMQ_Q4_K;
  const int64_t n_ot = (od + kTileN - 1) / kTileN, nsb = id / MMQ_QK;
  return static_cast<size_t>(b_scale_region(n_ot, nsb, q4) + b_scale_block(n_ot, 0, nsb, q4));
}

size_t bplane_operand_bytes(int type, int64_t od, int64_t id) {
  const int64_t n_ot = (od + kTileN - 1) / kTileN;
  return static_cast<size_t>(b_scale_region(n_ot, id / MMQ_QK, type == MMQ_Q4_K));
}

cudaError_t launch_register(const mmq_weights_s *h, const uint8_t *W, int *bad_scale,
                            cudaStream_t s) {
  // rows od..od_pad-1 of the last weight tile stay zero
  cudaError_t e = cudaMemsetAsync(h->bplane, 0, h->bplane_bytes, s);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(h->od), static_cast<unsigned>(h->nsb));
  uint8_t *bp = static_cast<uint8_t *>(h->bplane);
  const bool q4 = h->type == MMQ_Q4_K;
  const uint64_t sr = b_scale_region(h->od_pad / kTileN, h->nsb, q4);
  if (h->rawplane) {
    e = cudaMemsetAsync(h->rawplane, 0, h->rawplane_bytes, s);
    if (e != cudaSuccess) return e;
    if (q4)
      register_raw_kernel<true><<<grid, 64, 0, s>>>(W, h->id, h->rawplane);
    else
      register_raw_kernel<false><<<grid, 64, 0, s>>>(W, h->id, h->rawplane);
  }
  if (q4 && h->wexp) {
    expand_wexp_kernel<true><<<grid, 256, 0, s>>>(W, h->id, h->wexp);
    register_kernel<true, true><<<grid, 256, 0, s>>>(W, h->wexp, h->id, bp, sr, bad_scale);
  } else if (q4) {
    register_kernel<true, false><<<grid, 256, 0, s>>>(W, nullptr, h->id, bp, sr, bad_scale);
  } else if (h->wexp) {
    expand_wexp_kernel<false><<<grid, 256, 0, s>>>(W, h->id, h->wexp);
    register_kernel<false, true><<<grid, 256, 0, s>>>(W, h->wexp, h->id, bp, sr, bad_scale);
  } else {
    register_kernel<false, false><<<grid, 256, 0, s>>>(W, nullptr, h->id, bp, sr, bad_scale);
  }
  return cudaGetLastError();
}

cudaError_t launch_register_b0(const mmq_weights_s *h, const uint8_t *W, cudaStream_t s) {
  if (h->type != MMQ_Q6_K || !h->b0plane) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(h->b0plane, 0, h->b0plane_bytes, s);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(h->od), static_cast<unsigned>(h->nsb));
  uint8_t *bp = static_cast<uint8_t *>(h->bplane);
  const uint64_t sr = b_scale_region(h->od_pad / kTileN, h->nsb, false);
  if (h->wexp)
    register_kernel<false, true, true><<<grid, 256, 0, s>>>(W, h->wexp, h->id, bp, sr, nullptr, h->b0plane);
  else
    register_kernel<false, false, true><<<grid, 256, 0, s>>>(W, nullptr, h->id, bp, sr, nullptr, h->b0plane);
  return cudaGetLastError();
}

}  // namespace mmq
