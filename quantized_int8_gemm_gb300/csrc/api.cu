// api.cu -- the extern "C" entry points of libmmq.so (declared in mmq.h):
// argument validation, per-device state, registration bookkeeping, scratch
// and launches.  No arithmetic of the method happens on the host.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxTokens = 65535LL * 128;  // GEMM grid.y limit x token tile

struct DeviceState {
  bool probed = false;
  bool usable = false;
  mmq::DevStatus *words = nullptr;  // device memory
  cudaMemPool_t pool = nullptr;     // stream-ordered GEMM scratch
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_limit_ns{2000000000ull};
std::atomic<unsigned> g_epoch{1};

unsigned next_epoch() {
  unsigned e = g_epoch.fetch_add(1);
  if (e == 0) e = g_epoch.fetch_add(1);  // 0 never names a launch
  return e;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device, checked to be an sm_103 part, with its state initialised.
int device_state(int *dev_out, DeviceState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MMQ_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState &d = g_dev[dev];
  if (!d.probed) {
    d.probed = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return MMQ_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return MMQ_ERR_NO_DEVICE;
    if (cudaMalloc(&d.words, sizeof(mmq::DevStatus)) != cudaSuccess ||
        cudaMemset(d.words, 0, sizeof(mmq::DevStatus)) != cudaSuccess) {
      cudaGetLastError();
      return MMQ_ERR_CUDA;
    }
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return MMQ_ERR_CUDA;
    }
    uint64_t keep = UINT64_MAX;  // keep freed scratch cached in the pool
    cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    d.usable = true;
  }
  if (!d.usable) return MMQ_ERR_NO_DEVICE;
  *dev_out = dev;
  *out = &d;
  return MMQ_OK;
}

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return MMQ_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? MMQ_ERR_OOM : MMQ_ERR_CUDA;
}

void free_planes(mmq_weights_s *h) {
  if (h->bplane) cudaFree(h->bplane);
  if (h->wexp) cudaFree(h->wexp);
  if (h->rawplane) cudaFree(h->rawplane);
  if (h->b0plane) cudaFree(h->b0plane);
  h->bplane = nullptr;
  h->wexp = nullptr;
  h->rawplane = nullptr;
  h->b0plane = nullptr;
}

}  // namespace

extern "C" {

const char *mmq_strerror(int code) {
  switch (code) {
    case MMQ_OK: return "ok";
    case MMQ_ERR_ARG: return "invalid argument";
    case MMQ_ERR_ALIGN: return "misaligned pointer";
    case MMQ_ERR_TYPE: return "unknown weight type";
    case MMQ_ERR_CUDA: return "CUDA runtime error";
    case MMQ_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
    case MMQ_ERR_OOM: return "device out of memory";
    case MMQ_ERR_UNSUPPORTED: return "unsupported input for this build";
    case MMQ_ERR_NO_DEVICE: return "current device is not an sm_103 GPU";
    case MMQ_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than mmq_gemm_noalloc's fixed 16 MiB buffer";
    default: return "unknown status code";
  }
}

void mmq_set_wait_timeout_ns(uint64_t ns) { g_limit_ns.store(ns ? ns : 1); }

int mmq_quantize_act(const float *X, int64_t nt, int64_t id, void *Q, mmq_stream_t stream) {
  if (nt < 0 || id <= 0 || id % 32 != 0) return MMQ_ERR_ARG;
  if (nt == 0) return MMQ_OK;
  if (!X || !Q) return MMQ_ERR_ARG;
  if (!aligned16(X) || !aligned16(Q)) return MMQ_ERR_ALIGN;
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  return cuda_rc(mmq::launch_quantize_q8_0(X, nt, id, static_cast<uint8_t *>(Q),
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int mmq_register_weights(int type, const void *W, int64_t od, int64_t id, uint32_t flags,
                         mmq_stream_t stream, mmq_weights_t *out) {
  if (!out) return MMQ_ERR_ARG;
  *out = nullptr;
  if (type != MMQ_Q4_K && type != MMQ_Q6_K) return MMQ_ERR_TYPE;
  if (!W || od <= 0 || id <= 0 || id % MMQ_QK != 0) return MMQ_ERR_ARG;
  if (od > 0x7fffffffLL || id / MMQ_QK > 65535) return MMQ_ERR_ARG;
  if (flags & ~(MMQ_REG_WEXP | MMQ_REG_RAW)) return MMQ_ERR_ARG;
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  mmq_weights_s *h = new (std::nothrow) mmq_weights_s();
  if (!h) return MMQ_ERR_OOM;
  h->type = type;
  h->device = dev;
  h->flags = flags;
  h->od = od;
  h->id = id;
  h->od_pad = (od + mmq::kRowTile - 1) / mmq::kRowTile * mmq::kRowTile;
  h->nsb = id / MMQ_QK;
  h->nb32 = id / 32;
  h->bplane_bytes = mmq::bplane_bytes(type, od, id);
  h->wexp_bytes = (flags & MMQ_REG_WEXP) ? static_cast<size_t>(od) * id : 0;
  h->rawplane_bytes = (flags & MMQ_REG_RAW) ? mmq::rawplane_bytes(type, od, id) : 0;

  int rc = MMQ_OK;
  int *bad = nullptr;
  cudaError_t e = cudaMalloc(&h->bplane, h->bplane_bytes);
  if (e == cudaSuccess && h->wexp_bytes) e = cudaMalloc(&h->wexp, h->wexp_bytes);
  if (e == cudaSuccess && h->rawplane_bytes)
    e = cudaMalloc(reinterpret_cast<void **>(&h->rawplane), h->rawplane_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&bad, sizeof(int));
  if (e == cudaSuccess) e = cudaMemsetAsync(bad, 0, sizeof(int), s);
  if (e == cudaSuccess) e = mmq::launch_register(h, static_cast<const uint8_t *>(W), bad, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  int bad_h = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bad_h, bad, sizeof(int), cudaMemcpyDeviceToHost);
  if (bad) cudaFree(bad);
  // q6_K sub-block scales beyond +-64: a second pass splits the operand into
  // the B1 plane and the B0 plane
  if (e == cudaSuccess && bad_h) {
    h->b0plane_bytes = mmq::bplane_operand_bytes(type, od, id);
    e = cudaMalloc(reinterpret_cast<void **>(&h->b0plane), h->b0plane_bytes);
    if (e == cudaSuccess) e = mmq::launch_register_b0(h, static_cast<const uint8_t *>(W), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  // load what mmq_gemm_noalloc will launch for this handle now, while
  // allocating is allowed (lazy module loading would otherwise do it, and
  // allocate, inside that call)
  if (e == cudaSuccess) e = mmq::prepare_noalloc(h);
  if (e != cudaSuccess) rc = cuda_rc(e);
  if (rc != MMQ_OK) {
    free_planes(h);
    delete h;
    return rc;
  }
  *out = h;
  return MMQ_OK;
}

int mmq_dequantize_weights(int type, const void *W, int64_t od, int64_t id, void *out,
                           int out_type, mmq_stream_t stream) {
  if (type != MMQ_Q4_K && type != MMQ_Q6_K) return MMQ_ERR_TYPE;
  if (!W || !out || od <= 0 || id <= 0 || id % MMQ_QK != 0) return MMQ_ERR_ARG;
  if (od > 0x7fffffffLL || id / MMQ_QK > 65535) return MMQ_ERR_ARG;
  if (out_type != MMQ_OUT_F16 && out_type != MMQ_OUT_F32) return MMQ_ERR_ARG;
  if (!aligned16(out)) return MMQ_ERR_ALIGN;
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  return cuda_rc(mmq::launch_dequant(type, static_cast<const uint8_t *>(W), od, id, out, out_type,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int mmq_release_weights(mmq_weights_t h) {
  if (!h) return MMQ_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != h->device) cudaSetDevice(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  free_planes(h);
  if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  delete h;
  return cuda_rc(e);
}

int mmq_weights_wexp(mmq_weights_t h, const int8_t **plane, int64_t *row_pitch) {
  if (!h || !plane || !row_pitch) return MMQ_ERR_ARG;
  if (!h->wexp) return MMQ_ERR_UNSUPPORTED;
  *plane = h->wexp;
  *row_pitch = h->id;
  return MMQ_OK;
}

int mmq_weights_info(mmq_weights_t h, int *type, int64_t *od, int64_t *id,
                     int64_t *operand_bytes, int64_t *scale_bytes, int64_t *wexp_bytes) {
  if (!h) return MMQ_ERR_ARG;
  if (type) *type = h->type;
  if (od) *od = h->od;
  if (id) *id = h->id;
  const int64_t operand = static_cast<int64_t>(mmq::bplane_operand_bytes(h->type, h->od, h->id));
  if (operand_bytes) *operand_bytes = operand + static_cast<int64_t>(h->b0plane_bytes);
  if (scale_bytes) *scale_bytes = static_cast<int64_t>(h->bplane_bytes) - operand;
  if (wexp_bytes) *wexp_bytes = static_cast<int64_t>(h->wexp_bytes);
  return MMQ_OK;
}

// Q (pad40 blocks) or X (fp32 activations, quantized on the fly) -> Y.
static int gemm_impl(mmq_weights_t h, const void *Q, const float *X, int64_t nt, float *Y,
                     mmq_stream_t stream, uint32_t flags, int *arm_used, cudaEvent_t ev0,
                     cudaEvent_t ev1) {
  if (!h || nt < 0 || nt > kMaxTokens) return MMQ_ERR_ARG;
  if (flags != MMQ_ARM_AUTO && flags != MMQ_ARM_F16 && flags != MMQ_ARM_RAW && flags != MMQ_ARM_SPLIT &&
      flags != MMQ_ARM_PAIR)
    return MMQ_ERR_UNSUPPORTED;
  if (flags == MMQ_ARM_RAW && (!h->rawplane || h->b0plane)) return MMQ_ERR_UNSUPPORTED;
  if (flags == MMQ_ARM_PAIR && h->b0plane) return MMQ_ERR_UNSUPPORTED;
  // library choice: the pair arm above 128 tokens (one-plane operands; not for q6_K whose
  // 256-row split tiles fill two or more waves); else the split arm for one-plane q6_K, and
  // for q4_K where it runs 256-row tiles or pieces of tiles; else the fp16-plane arm (a
  // two-plane q6_K operand doubles the split arm's tensor work but hides in the other's hand-off)
  const bool raw = flags == MMQ_ARM_RAW;
  const bool pair = flags == MMQ_ARM_PAIR || (flags == MMQ_ARM_AUTO && mmq::gemm_pair_preferred(h, nt));
  const bool split = pair || flags == MMQ_ARM_SPLIT ||
                     (flags == MMQ_ARM_AUTO && ((h->type == MMQ_Q6_K && !h->b0plane) ||
                                                (h->type == MMQ_Q4_K && mmq::gemm_split_wide(h, nt))));
  if (arm_used) *arm_used = raw ? MMQ_ARM_RAW : pair ? MMQ_ARM_PAIR : split ? MMQ_ARM_SPLIT : MMQ_ARM_F16;
  if (nt == 0) return MMQ_OK;
  const void *A = X ? static_cast<const void *>(X) : Q;
  if (!A || !Y) return MMQ_ERR_ARG;
  if (!aligned16(A) || !aligned16(Y)) return MMQ_ERR_ALIGN;
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  if (dev != h->device) return MMQ_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // Scratch is stream-ordered: from the library pool, or -- while the stream
  // is being captured into a CUDA graph -- a graph memory node.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return cuda_rc(e);
  const bool capturing = cap == cudaStreamCaptureStatusActive;
  const size_t bytes =
      split ? mmq::gemm_split_scratch_bytes(h, nt, pair) : mmq::gemm_scratch_bytes(h, nt, true, raw);
  void *scratch = nullptr;
  e = capturing ? cudaMallocAsync(&scratch, bytes, s)
                : cudaMallocFromPoolAsync(&scratch, bytes, d->pool, s);
  if (e != cudaSuccess) return cuda_rc(e);
  // inside a capture the events must become real record nodes of the graph
  const unsigned ev_flags = capturing ? cudaEventRecordExternal : cudaEventRecordDefault;
  if (split)
    e = mmq::launch_gemm_split(h, static_cast<const uint8_t *>(Q), X, nt, Y, scratch, d->words, next_epoch(),
                               g_limit_ns.load(), s, ev0, ev1, ev_flags, pair);
  else
    e = mmq::launch_gemm(h, static_cast<const uint8_t *>(Q), X, nt, Y, scratch, true, raw,
                         d->words, next_epoch(), g_limit_ns.load(), s, ev0, ev1, ev_flags);
  cudaError_t ef = cudaFreeAsync(scratch, s);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

int mmq_gemm(mmq_weights_t h, const void *Q, int64_t nt, float *Y, mmq_stream_t stream,
             uint32_t flags, int *arm_used) {
  return gemm_impl(h, Q, nullptr, nt, Y, stream, flags, arm_used, nullptr, nullptr);
}

int mmq_gemm_f32(mmq_weights_t h, const float *X, int64_t nt, float *Y, mmq_stream_t stream,
                 uint32_t flags, int *arm_used) {
  if (!X && nt > 0) return MMQ_ERR_ARG;
  return gemm_impl(h, nullptr, X, nt, Y, stream, flags, arm_used, nullptr, nullptr);
}

int mmq_gemm_f32_profiled(mmq_weights_t h, const float *X, int64_t nt, float *Y,
                          mmq_stream_t stream, uint32_t flags, int *arm_used, void *ev_start,
                          void *ev_stop) {
  if (!X && nt > 0) return MMQ_ERR_ARG;
  return gemm_impl(h, nullptr, X, nt, Y, stream, flags, arm_used,
                   static_cast<cudaEvent_t>(ev_start), static_cast<cudaEvent_t>(ev_stop));
}

int mmq_gemm_profiled(mmq_weights_t h, const void *Q, int64_t nt, float *Y, mmq_stream_t stream,
                      uint32_t flags, int *arm_used, void *ev_start, void *ev_stop) {
  return gemm_impl(h, Q, nullptr, nt, Y, stream, flags, arm_used, static_cast<cudaEvent_t>(ev_start),
                   static_cast<cudaEvent_t>(ev_stop));
}

int mmq_debug_chunk_partials(mmq_weights_t h, const void *Q, int64_t nt, float *P, mmq_stream_t stream) {
  if (!h || nt < 0 || nt > kMaxTokens) return MMQ_ERR_ARG;
  if (nt == 0) return MMQ_OK;
  if (!Q || !P) return MMQ_ERR_ARG;
  if (!aligned16(Q) || !aligned16(P)) return MMQ_ERR_ALIGN;
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  if (dev != h->device) return MMQ_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const int64_t nt_pad = (nt + 127) / 128 * 128;
  const size_t gemm_bytes = up(mmq::gemm_scratch_bytes(h, nt, false, false));
  const size_t dump_bytes = up(static_cast<size_t>(nt_pad * h->nb32 * h->od_pad) * sizeof(float));
  const size_t y_bytes = static_cast<size_t>(nt * h->od) * sizeof(float);
  void *scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, gemm_bytes + dump_bytes + y_bytes, d->pool, s);
  if (e != cudaSuccess) return cuda_rc(e);
  uint8_t *base = static_cast<uint8_t *>(scratch);
  float *dump = reinterpret_cast<float *>(base + gemm_bytes);
  float *Y = reinterpret_cast<float *>(base + gemm_bytes + dump_bytes);
  e = mmq::launch_gemm(h, static_cast<const uint8_t *>(Q), nullptr, nt, Y, scratch, false, false, d->words,
                       next_epoch(), g_limit_ns.load(), s, nullptr, nullptr, 0, dump);
  if (e == cudaSuccess)  // rows (t, chunk) of od partials, out of rows of od_pad
    e = cudaMemcpy2DAsync(P, static_cast<size_t>(h->od) * sizeof(float), dump,
                          static_cast<size_t>(h->od_pad) * sizeof(float), static_cast<size_t>(h->od) * sizeof(float),
                          static_cast<size_t>(nt * h->nb32), cudaMemcpyDeviceToDevice, s);
  cudaError_t ef = cudaFreeAsync(scratch, s);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

int mmq_gemm_noalloc(mmq_weights_t h, const void *Q, int64_t nt, float *Y, mmq_stream_t stream) {
  if (!h || nt < 0 || nt > kMaxTokens) return MMQ_ERR_ARG;
  if (nt == 0) return MMQ_OK;
  if (!Q || !Y) return MMQ_ERR_ARG;
  if (!aligned16(Q) || !aligned16(Y)) return MMQ_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MMQ_ERR_NO_DEVICE;
  }
  if (dev != h->device) return MMQ_ERR_ARG;
  // A valid handle means registration already set up this device's state;
  // look it up without ever initialising (initialising would allocate).
  DeviceState *d = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[dev].usable) d = &g_dev[dev];
  }
  if (!d) return MMQ_ERR_ARG;
  if (mmq::gemm_scratch_bytes(h, nt, false, false) > mmq::kNoallocScratchBytes)
    return MMQ_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  cudaError_t e = mmq::noalloc_scratch(dev, &scratch);
  if (e == cudaSuccess)
    e = mmq::launch_gemm(h, static_cast<const uint8_t *>(Q), nullptr, nt, Y, scratch, false, false, d->words,
                         next_epoch(), g_limit_ns.load(), reinterpret_cast<cudaStream_t>(stream),
                         nullptr, nullptr, cudaEventRecordDefault);
  return cuda_rc(e);
}

int mmq_last_device_error(void) {
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return cuda_rc(cudaErrorUnknown);
  mmq::DevStatus w;
  if (cudaMemcpy(&w, d->words, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_rc(cudaErrorUnknown);
  const int zero = 0;
  if (cudaMemcpy(&d->words->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return cuda_rc(cudaErrorUnknown);
  return w.status ? MMQ_ERR_DEVICE_TIMEOUT : MMQ_OK;
}

int mmq_probe_engine_rates(double *out, mmq_stream_t stream) {
  if (!out) return MMQ_ERR_ARG;
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  cudaError_t e = mmq::launch_engine_probes(d->words, next_epoch(), g_limit_ns.load(),
                                            reinterpret_cast<cudaStream_t>(stream), out);
  if (e != cudaSuccess) return cuda_rc(e);
  return mmq_last_device_error();
}

int mmq_selftest_wait_timeout(uint64_t timeout_ns, mmq_stream_t stream) {
  int dev;
  DeviceState *d;
  if (int rc = device_state(&dev, &d)) return rc;
  cudaError_t e = mmq::launch_wait_selftest(d->words, next_epoch(), timeout_ns ? timeout_ns : 1,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_rc(e);
  return mmq_last_device_error();
}

}  // extern "C"
