// q8.cuh -- the q8_0 block rule, shared by the library's three quantization
// kernels (mmq_quantize_act and the two GEMM prepasses), so their codes are
// the same bit for bit.
//
// One 32-value block on eight lanes, one float4 each:
//   amax = max |x|;  d = amax / 127  (fp32, IEEE division);
//   q_i  = roundf(x_i / d)           (half away from zero), 0 when amax = 0;
//   d16  = fp16 round-to-nearest-even of d (0 when amax = 0).
// x_i / d is formed without a division per element: from r = 1/d correctly
// rounded, Markstein's correction (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34,
// 1990) gives the correctly rounded quotient in three operations,
//   p = x*r,  e = fma(-p, d, x)  (exact),  q = fma(e, r, p).
// Checked against CUDA's IEEE division: roundf of both agree on every fp32
// significand of d in five binades from 2^-97 to 2^22, for every x within
// 64 ulps of each half-integer n + 1/2 (n = 0..126) of q8_0, both signs --
// the only quotients where a last-bit difference could change the code.
// Blocks with amax below 2^-90 (where the remainder could underflow) divide.
// |x_i| <= amax gives |x_i / d| <= 127 (1 + 2^-23), so |q_i| <= 127 without
// a clamp.
#pragma once
#include <cuda_fp16.h>

namespace mmq {

constexpr float kQ8FastAmax = 0x1p-90f;

__device__ __forceinline__ float q8_quot(float x, float d, float r) {
  const float p = x * r;
  const float e = fmaf(-p, d, x);
  return fmaf(e, r, p);
}

// The block's stored scale d16 (as fp32) and this lane's four codes, as
// floats (exact integers); the eight lanes of a block are lanes 8g .. 8g+7.
__device__ __forceinline__ void q8_lane(float4 v, float &d16f, float (&q)[4]) {
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  const float d = amax / 127.0f;
  const float xs[4] = {v.x, v.y, v.z, v.w};
  if (amax >= kQ8FastAmax) {
    // q8_quot on pairs: the packed fp32x2 multiply and fmas round each lane
    // as the scalar ones do
    const float r = __frcp_rn(d);
    const float2 d2 = make_float2(d, d), r2 = make_float2(r, r);
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      const float2 x = make_float2(xs[i], xs[i + 1]);
      const float2 p = __fmul2_rn(x, r2);
      const float2 e = __ffma2_rn(make_float2(-p.x, -p.y), d2, x);
      const float2 qq = __ffma2_rn(e, r2, p);
      q[i] = roundf(qq.x);
      q[i + 1] = roundf(qq.y);
    }
  } else if (amax != 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = roundf(xs[i] / d);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = 0.0f;
  }
  d16f = amax != 0.0f ? __half2float(__float2half_rn(d)) : 0.0f;
}

// sum of the block's 32 codes (exact in fp32: |ssum| <= 4064), on every lane
__device__ __forceinline__ float q8_ssum(const float (&q)[4]) {
  float s = (q[0] + q[1]) + (q[2] + q[3]);
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
  return s;
}

// two codes as one half2 word (exact: |q| <= 127)
__device__ __forceinline__ uint32_t q8_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

}  // namespace mmq
