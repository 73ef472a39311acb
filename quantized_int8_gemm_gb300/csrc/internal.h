// internal.h -- declarations shared by the translation units of libmmq.so.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "mmq.h"

// A registered weight.  Device memory owned by the handle:
//   bplane  the GEMM's pre-tiled weight plane (tiling.h): per 128-row tile,
//           super-block and half, the fp16 operand image with the sub-block
//           scale folded in and, for q4_K, the integer-min image; then the
//           scale region (d and, for q4_K, dmin rows).  Rows od..od_pad-1
//           are zero.
//   wexp    optional dense centered q6_K plane, int8 [od][id], q - 32
//   rawplane  optional packed bytes of W regrouped per tile (tiling.h), read
//           by the GEMM's raw arm
struct mmq_weights_s {
  int type = 0;
  int device = 0;
  uint32_t flags = 0;
  int64_t od = 0, id = 0, od_pad = 0, nsb = 0, nb32 = 0;
  void *bplane = nullptr;
  int8_t *wexp = nullptr;
  uint8_t *rawplane = nullptr;  // MMQ_REG_RAW: packed bytes regrouped for the raw arm
  // q6_K with a sub-block scale |sc| > 64: sc*(q - 32) needs up to 13 bits, so
  // the operand plane holds B1 = 2*sc*((q-32) >> 1) and this plane, same
  // layout, B0 = sc*((q-32) & 1); both exact in fp16, B1 + B0 = sc*(q - 32)
  uint8_t *b0plane = nullptr;
  size_t bplane_bytes = 0, wexp_bytes = 0, rawplane_bytes = 0, b0plane_bytes = 0;
};

namespace mmq {

struct WaitCtl;

// Per-device status words (device memory), see WaitCtl in ptx.cuh.
struct DevStatus {
  int status;
  unsigned abort_epoch;
};

constexpr int kRowTile = 128;  // od padding granule == GEMM weight tile

cudaError_t launch_quantize_q8_0(const float *X, int64_t nt, int64_t id, uint8_t *Q,
                                 cudaStream_t s);

// Registration: bytes of the tiled weight plane, and the expansion kernels.
// *bad_scale (device int) becomes nonzero if a q6_K sub-block scale |sc| > 64.
size_t bplane_bytes(int type, int64_t od, int64_t id);
size_t bplane_operand_bytes(int type, int64_t od, int64_t id);  // without the scale region
size_t rawplane_bytes(int type, int64_t od, int64_t id);
cudaError_t launch_dequant(int type, const uint8_t *W, int64_t od, int64_t id, void *out,
                           int out_type, cudaStream_t s);
cudaError_t launch_register(const mmq_weights_s *h, const uint8_t *W, int *bad_scale,
                            cudaStream_t s);
// second pass for q6_K handles with |sc| > 64: B1 into the operand plane, B0
// into h->b0plane (allocated by the caller, b0plane_bytes)
cudaError_t launch_register_b0(const mmq_weights_s *h, const uint8_t *W, cudaStream_t s);

// GEMM: scratch bytes for nt tokens, and the launch of the activation
// prepass + GEMM kernel.  With streamk_allowed the GEMM may split tiles
// between CTAs (and then needs more scratch).  ev0/ev1 (optional) are
// recorded around the GEMM kernel with cudaEventRecordWithFlags(ev, s,
// ev_flags).
// raw: stream the handle's raw plane and unpack it in the kernel.
size_t gemm_scratch_bytes(const mmq_weights_s *h, int64_t nt, bool streamk_allowed, bool raw);
// dump (test hook; whole tiles, not the raw arm): also store every chunk's raw
// partial, fp32, at dump[(t * nb32 + chunk) * od_pad + o] (nt_pad x nb32 x od_pad)
cudaError_t launch_gemm(const mmq_weights_s *h, const uint8_t *Q, const float *X, int64_t nt,
                        float *Y, void *scratch, bool streamk_allowed, bool raw, DevStatus *st,
                        unsigned epoch, uint64_t limit_ns, cudaStream_t s, cudaEvent_t ev0,
                        cudaEvent_t ev1, unsigned ev_flags, float *dump = nullptr);

// Split arm (activation scale folded into A as an exact fp16 hi + lo pair):
// scratch bytes, and the prepass + GEMM launch.  pair: the same operands and
// arithmetic on 2-CTA clusters (cta_group::2 UMMAs of 256 weight rows by 128
// tokens; one-plane handles only).
size_t gemm_split_scratch_bytes(const mmq_weights_s *h, int64_t nt, bool pair);
// whether the split arm would run 256-row weight tiles or pieces of tiles for this many tokens
bool gemm_split_wide(const mmq_weights_s *h, int64_t nt);
// whether MMQ_ARM_AUTO takes the pair arm for this many tokens
bool gemm_pair_preferred(const mmq_weights_s *h, int64_t nt);
cudaError_t launch_gemm_split(const mmq_weights_s *h, const uint8_t *Q, const float *X, int64_t nt, float *Y,
                              void *scratch, DevStatus *st, unsigned epoch, uint64_t limit_ns,
                              cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, unsigned ev_flags, bool pair);

cudaError_t launch_wait_selftest(DevStatus *st, unsigned epoch, uint64_t limit_ns,
                                 cudaStream_t s);

// Engine-rate microbenchmarks (probe.cu); out[0..4] as mmq_probe_engine_rates.
cudaError_t launch_engine_probes(DevStatus *st, unsigned epoch, uint64_t limit_ns, cudaStream_t s, double *out);

// Fixed scratch of mmq_gemm_noalloc (a static device array in gemm.cu).
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
cudaError_t noalloc_scratch(int dev, void **out);
// Loads, on the handle's device, the scratch array's module and the kernels
// mmq_gemm_noalloc launches for this handle (registration calls it).
cudaError_t prepare_noalloc(const mmq_weights_s *h);

}  // namespace mmq
