// internal.h -- declarations shared by the translation units of libmmq.so.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mmq.h"

// A registered weight.  Planes (all device memory owned by the handle):
//   b16     fp16 [od_pad][id]   operand with the sub-block scale folded in:
//                               q6_K sc*(q-32), q4_K sc*q  (exact integers)
//   dplane  fp32 [nsb][od_pad]  super-block scale d
//   mmplane fp32 [nb32][od_pad] q4_K only: dmin*m per 32-element sub-block
//   wexp    int8 [od][id]       optional dense centered q6_K plane, q-32
// Rows od..od_pad-1 of every padded plane are zero.
struct mmq_weights_s {
  int type = 0;
  int device = 0;
  uint32_t flags = 0;
  int64_t od = 0, id = 0, od_pad = 0, nsb = 0, nb32 = 0;
  void *b16 = nullptr;
  float *dplane = nullptr;
  float *mmplane = nullptr;
  int8_t *wexp = nullptr;
  size_t b16_bytes = 0, dplane_bytes = 0, mm_bytes = 0, wexp_bytes = 0;
  CUtensorMap tm_b{}, tm_d{}, tm_mm{};
};

namespace mmq {

struct WaitCtl;

// Per-device status words (device memory), see WaitCtl in ptx.cuh.
struct DevStatus {
  int status;
  unsigned abort_epoch;
};

constexpr int kRowTile = 128;  // od padding granule == GEMM N tile

bool encode_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle sw);

cudaError_t launch_quantize_q8_0(const float *X, int64_t nt, int64_t id, uint8_t *Q,
                                 cudaStream_t s);

// Registration: expand packed blocks into the handle's planes.  *bad_scale
// (device int) receives a nonzero value if a q6_K sub-block scale |sc| > 64.
cudaError_t launch_register(const mmq_weights_s *h, const uint8_t *W, int *bad_scale,
                            cudaStream_t s);

// GEMM: activation prepass (pad40 -> fp16 operand + per-chunk scales) and the
// tcgen05 kernel.
cudaError_t launch_gemm_prepass(const uint8_t *Q, int64_t nt, int64_t id, void *a16, void *sc,
                                cudaStream_t s);
cudaError_t launch_gemm_f16(const mmq_weights_s *h, const CUtensorMap &tm_a, const void *sc,
                            int64_t nt, float *Y, DevStatus *st, unsigned epoch,
                            uint64_t limit_ns, cudaStream_t s);

cudaError_t launch_wait_selftest(DevStatus *st, unsigned epoch, uint64_t limit_ns,
                                 cudaStream_t s);

}  // namespace mmq
