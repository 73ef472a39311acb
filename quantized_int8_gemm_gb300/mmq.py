"""Python binding of libmmq.so: the C-ABI entry points under the same names.

Argument marshalling only.  Device buffers are torch CUDA tensors (PyTorch
supplies device memory and streams); every step of the computation runs in
the library's CUDA kernels.  If the library is missing the import of any
entry point raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmmq.so")

MMQ_OK = 0
MMQ_ERR_ARG = -1
MMQ_ERR_ALIGN = -2
MMQ_ERR_TYPE = -3
MMQ_ERR_CUDA = -4
MMQ_ERR_DEVICE_TIMEOUT = -5
MMQ_ERR_OOM = -6
MMQ_ERR_UNSUPPORTED = -7
MMQ_ERR_NO_DEVICE = -8
MMQ_ERR_SCRATCH_LIMIT = -9

MMQ_Q4_K = 12
MMQ_Q6_K = 14
QTYPES = {"q4_K": MMQ_Q4_K, "q6_K": MMQ_Q6_K}

MMQ_REG_WEXP = 0x1
MMQ_REG_RAW = 0x2
MMQ_ARM_AUTO = 0
MMQ_ARM_F16 = 1
MMQ_ARM_RAW = 2
MMQ_ARM_SPLIT = 3
MMQ_ARM_PAIR = 4
MMQ_OUT_F16 = 1
MMQ_OUT_F32 = 2
ARM_NAMES = {MMQ_ARM_F16: "f16_plane", MMQ_ARM_RAW: "raw_unpack", MMQ_ARM_SPLIT: "split_scale",
             MMQ_ARM_PAIR: "split_scale_sm_pairs"}

Q8_BLOCK_BYTES = 40
BLOCK_BYTES = {MMQ_Q4_K: 144, MMQ_Q6_K: 210}

EXPORTS = [
    "mmq_quantize_act", "mmq_register_weights", "mmq_release_weights", "mmq_weights_wexp",
    "mmq_weights_info", "mmq_gemm", "mmq_gemm_f32", "mmq_gemm_profiled", "mmq_gemm_f32_profiled",
    "mmq_gemm_noalloc", "mmq_debug_chunk_partials", "mmq_dequantize_weights",
    "mmq_last_device_error", "mmq_set_wait_timeout_ns",
    "mmq_selftest_wait_timeout", "mmq_strerror", "mmq_probe_engine_rates",
]

_lock = threading.Lock()
_lib = None


class MMQError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmmq.so (built by quantized_int8_gemm_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libmmq.so not built ({p}); run quantized_int8_gemm_gb300.build.build()")
        L = ctypes.CDLL(p)
        i64, vp, u32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int
        L.mmq_quantize_act.argtypes = [vp, i64, i64, vp, vp]
        L.mmq_register_weights.argtypes = [i32, vp, i64, i64, u32, vp, ctypes.POINTER(vp)]
        L.mmq_release_weights.argtypes = [vp]
        L.mmq_weights_wexp.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(i64)]
        L.mmq_weights_info.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i64),
                                       ctypes.POINTER(i64), ctypes.POINTER(i64),
                                       ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.mmq_gemm.argtypes = [vp, vp, i64, vp, vp, u32, ctypes.POINTER(i32)]
        L.mmq_gemm_f32.argtypes = [vp, vp, i64, vp, vp, u32, ctypes.POINTER(i32)]
        L.mmq_gemm_profiled.argtypes = [vp, vp, i64, vp, vp, u32, ctypes.POINTER(i32), vp, vp]
        L.mmq_gemm_f32_profiled.argtypes = [vp, vp, i64, vp, vp, u32, ctypes.POINTER(i32), vp, vp]
        L.mmq_gemm_noalloc.argtypes = [vp, vp, i64, vp, vp]
        L.mmq_debug_chunk_partials.argtypes = [vp, vp, i64, vp, vp]
        L.mmq_dequantize_weights.argtypes = [i32, vp, i64, i64, vp, i32, vp]
        L.mmq_last_device_error.argtypes = []
        L.mmq_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        L.mmq_set_wait_timeout_ns.restype = None
        L.mmq_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.mmq_probe_engine_rates.argtypes = [vp, vp]
        L.mmq_strerror.argtypes = [i32]
        L.mmq_strerror.restype = ctypes.c_char_p
        for n in EXPORTS:
            f = getattr(L, n)
            if n not in ("mmq_set_wait_timeout_ns", "mmq_strerror"):
                f.restype = ctypes.c_int
        _lib = L
        return L


def strerror(code: int) -> str:
    try:
        return load().mmq_strerror(code).decode()
    except RuntimeError:
        return f"status {code}"


def _check(rc: int, what: str):
    if rc != MMQ_OK:
        raise MMQError(rc, what)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev_ptr(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class Weights:
    """Owning wrapper of an mmq_weights_t handle."""

    def __init__(self, handle: int, qtype: int, od: int, id_: int, flags: int):
        self.handle = ctypes.c_void_p(handle)
        self.qtype, self.od, self.id, self.flags = qtype, od, id_, flags

    def release(self):
        if self.handle:
            _check(load().mmq_release_weights(self.handle), "mmq_release_weights")
            self.handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            if self.handle and _lib is not None:
                _lib.mmq_release_weights(self.handle)
        except Exception:
            pass


def mmq_quantize_act(X: torch.Tensor, Q: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """X (nt, id) fp32 CUDA -> Q (nt, id/32, 40) uint8 pad40 blocks."""
    if X.dtype != torch.float32 or X.dim() != 2:
        raise ValueError("X must be a 2-D float32 tensor")
    nt, id_ = X.shape
    if Q is None:
        Q = torch.empty((nt, id_ // 32, Q8_BLOCK_BYTES), dtype=torch.uint8, device=X.device)
    if Q.numel() != nt * (id_ // 32) * Q8_BLOCK_BYTES:
        raise ValueError("Q has the wrong size")
    _check(load().mmq_quantize_act(_dev_ptr(X, "X"), nt, id_, _dev_ptr(Q, "Q"), _stream(stream)),
           "mmq_quantize_act")
    return Q


def mmq_register_weights(qtype, W: torch.Tensor, od: int, id_: int, flags: int = 0,
                         stream=None) -> Weights:
    """Packed k-quant rows (uint8 CUDA tensor) -> registered Weights."""
    qt = QTYPES.get(qtype, qtype)
    h = ctypes.c_void_p()
    _check(load().mmq_register_weights(int(qt), _dev_ptr(W, "W"), od, id_, flags, _stream(stream),
                                       ctypes.byref(h)), "mmq_register_weights")
    return Weights(h.value, int(qt), od, id_, flags)


def mmq_dequantize_weights(qtype, W: torch.Tensor, od: int, id_: int, dtype=torch.float16,
                           stream=None) -> torch.Tensor:
    """Packed k-quant rows -> dense (od, id) fp16 or fp32 weights (the fallback plane)."""
    qt = QTYPES.get(qtype, qtype)
    out_type = {torch.float16: MMQ_OUT_F16, torch.float32: MMQ_OUT_F32}[dtype]
    out = torch.empty((od, id_), dtype=dtype, device=W.device)
    _check(load().mmq_dequantize_weights(int(qt), _dev_ptr(W, "W"), od, id_, _dev_ptr(out, "out"),
                                         out_type, _stream(stream)), "mmq_dequantize_weights")
    return out


def mmq_weights_wexp(w: Weights) -> torch.Tensor:
    """Zero-copy int8 (od, id) view of the handle's dense W_exp plane."""
    p, pitch = ctypes.c_void_p(), ctypes.c_int64()
    _check(load().mmq_weights_wexp(w.handle, ctypes.byref(p), ctypes.byref(pitch)),
           "mmq_weights_wexp")

    class _Plane:
        __cuda_array_interface__ = {
            "shape": (w.od, w.id), "typestr": "|i1", "data": (p.value, False),
            "strides": (pitch.value, 1), "version": 3,
        }

    return torch.as_tensor(_Plane(), device="cuda")


def mmq_weights_info(w: Weights) -> dict:
    t, od, id_, ob, sb, wb = (ctypes.c_int(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(),
                              ctypes.c_int64(), ctypes.c_int64())
    _check(load().mmq_weights_info(w.handle, *(ctypes.byref(v) for v in (t, od, id_, ob, sb, wb))),
           "mmq_weights_info")
    return {"type": t.value, "od": od.value, "id": id_.value, "operand_bytes": ob.value,
            "scale_bytes": sb.value, "wexp_bytes": wb.value}


def mmq_gemm(w: Weights, Q: torch.Tensor, nt: int, Y: torch.Tensor | None = None, stream=None,
             flags: int = MMQ_ARM_AUTO, return_arm: bool = False):
    """Y (nt, od) fp32 = dequant(Q) . dequant(W)^T."""
    if Y is None:
        Y = torch.empty((nt, w.od), dtype=torch.float32, device=Q.device)
    if Y.dtype != torch.float32 or Y.numel() != nt * w.od:
        raise ValueError("Y must be float32 with nt*od elements")
    arm = ctypes.c_int(0)
    _check(load().mmq_gemm(w.handle, _dev_ptr(Q, "Q"), nt, _dev_ptr(Y, "Y"), _stream(stream), flags,
                           ctypes.byref(arm)), "mmq_gemm")
    return (Y, arm.value) if return_arm else Y


def mmq_gemm_f32(w: Weights, X: torch.Tensor, Y: torch.Tensor | None = None, stream=None,
                 flags: int = MMQ_ARM_AUTO, return_arm: bool = False):
    """Y (nt, od) fp32 from fp32 activations X (nt, id), quantized on the fly."""
    if X.dtype != torch.float32 or X.dim() != 2 or X.shape[1] != w.id:
        raise ValueError("X must be float32 (nt, id)")
    nt = X.shape[0]
    if Y is None:
        Y = torch.empty((nt, w.od), dtype=torch.float32, device=X.device)
    if Y.dtype != torch.float32 or Y.numel() != nt * w.od:
        raise ValueError("Y must be float32 with nt*od elements")
    arm = ctypes.c_int(0)
    _check(load().mmq_gemm_f32(w.handle, _dev_ptr(X, "X"), nt, _dev_ptr(Y, "Y"), _stream(stream),
                               flags, ctypes.byref(arm)), "mmq_gemm_f32")
    return (Y, arm.value) if return_arm else Y


def mmq_gemm_profiled(w: Weights, Q: torch.Tensor, nt: int, Y: torch.Tensor,
                      ev_start: torch.cuda.Event, ev_stop: torch.cuda.Event, stream=None,
                      flags: int = MMQ_ARM_AUTO) -> int:
    """mmq_gemm that records ev_start / ev_stop around the main GEMM kernel.
    The events must already exist (torch creates them lazily: record once)."""
    arm = ctypes.c_int(0)
    _check(load().mmq_gemm_profiled(w.handle, _dev_ptr(Q, "Q"), nt, _dev_ptr(Y, "Y"),
                                    _stream(stream), flags, ctypes.byref(arm),
                                    ctypes.c_void_p(ev_start.cuda_event),
                                    ctypes.c_void_p(ev_stop.cuda_event)), "mmq_gemm_profiled")
    return arm.value


def mmq_gemm_f32_profiled(w: Weights, X: torch.Tensor, Y: torch.Tensor,
                          ev_start: torch.cuda.Event, ev_stop: torch.cuda.Event, stream=None,
                          flags: int = MMQ_ARM_AUTO) -> int:
    """mmq_gemm_f32 that records ev_start / ev_stop around the main GEMM kernel."""
    arm = ctypes.c_int(0)
    _check(load().mmq_gemm_f32_profiled(w.handle, _dev_ptr(X, "X"), X.shape[0], _dev_ptr(Y, "Y"),
                                        _stream(stream), flags, ctypes.byref(arm),
                                        ctypes.c_void_p(ev_start.cuda_event),
                                        ctypes.c_void_p(ev_stop.cuda_event)),
           "mmq_gemm_f32_profiled")
    return arm.value


def mmq_debug_chunk_partials(w: Weights, Q: torch.Tensor, nt: int, stream=None) -> torch.Tensor:
    """Test hook: the fp16-plane arm's raw per-chunk TMEM partials, fp32
    (nt, id/32, od): exact integers, before any float scale."""
    P = torch.empty((nt, w.id // 32, w.od), dtype=torch.float32, device=Q.device)
    _check(load().mmq_debug_chunk_partials(w.handle, _dev_ptr(Q, "Q"), nt, _dev_ptr(P, "P"), _stream(stream)),
           "mmq_debug_chunk_partials")
    return P


def mmq_gemm_noalloc(w: Weights, Q: torch.Tensor, nt: int, Y: torch.Tensor, stream=None):
    """mmq_gemm that allocates no device memory (fixed 16 MiB library scratch);
    for callers that cannot allocate.  Y must be preallocated."""
    _check(load().mmq_gemm_noalloc(w.handle, _dev_ptr(Q, "Q"), nt, _dev_ptr(Y, "Y"), _stream(stream)),
           "mmq_gemm_noalloc")
    return Y


def mmq_last_device_error() -> int:
    return load().mmq_last_device_error()


def mmq_set_wait_timeout_ns(ns: int):
    load().mmq_set_wait_timeout_ns(int(ns))


def mmq_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return load().mmq_selftest_wait_timeout(int(timeout_ns), _stream(stream))


def mmq_strerror(code: int) -> str:
    return strerror(code)


def mmq_probe_engine_rates(stream=None) -> dict:
    """Rates of the tensor engines on the current device (a measurement hook):
    tcgen05 kind::f16 MACs per clock per SM, M = 128 (cta_group::1) and
    M = 256 over an SM pair (cta_group::2), at several N; the whole-GPU
    mma.sync s8 TOPS and f16 TFLOP/s."""
    out = (ctypes.c_double * 12)()
    rc = load().mmq_probe_engine_rates(ctypes.cast(out, ctypes.c_void_p), _stream(stream))
    if rc != MMQ_OK:
        raise MMQError(rc, "mmq_probe_engine_rates")
    return {"umma_f16_mac_per_clk_per_sm": {"N64": out[0], "N96": out[5], "N112": out[6], "N128": out[1],
                                            "N256": out[2]},
            "umma_pair_f16_mac_per_clk_per_sm": {"N64": out[7], "N96": out[8], "N112": out[9], "N128": out[10],
                                                 "N256": out[11]},
            "mma_sync_s8_tops": out[3], "mma_sync_f16_tflops": out[4]}
