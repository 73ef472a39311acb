"""GB300 (sm_103a) k-quant x q8_0 prefill GEMM: Python binding of libmmq.so.

The package holds the CUDA sources (csrc/), their build script (build.py) and
the ctypes binding (mmq.py); the C ABI is declared in include/mmq.h.
"""
from .mmq import (  # noqa: F401
    ARM_NAMES,
    MMQ_ARM_AUTO,
    MMQ_ARM_F16,
    MMQ_ARM_PAIR,
    MMQ_ARM_RAW,
    MMQ_ARM_SPLIT,
    MMQ_OUT_F16,
    MMQ_OUT_F32,
    MMQ_Q4_K,
    MMQ_Q6_K,
    MMQ_REG_RAW,
    MMQ_REG_WEXP,
    MMQError,
    Weights,
    load,
    mmq_dequantize_weights,
    mmq_gemm,
    mmq_gemm_f32,
    mmq_gemm_f32_profiled,
    mmq_gemm_noalloc,
    mmq_debug_chunk_partials,
    mmq_gemm_profiled,
    mmq_last_device_error,
    mmq_probe_engine_rates,
    mmq_quantize_act,
    mmq_register_weights,
    mmq_selftest_wait_timeout,
    mmq_set_wait_timeout_ns,
    mmq_strerror,
    mmq_weights_info,
    mmq_weights_wexp,
)
