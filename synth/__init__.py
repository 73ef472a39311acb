"""Seeded synthetic inputs for the k-quant x q8_0 GEMM (shared by the oracle
side and the CUDA side of every test and benchmark).

This package holds no arithmetic of the method: it draws random bytes and
normal fp32 activations and lays random fields into the packed block formats
by byte offset.  It never quantizes, dequantizes or multiplies.
"""
from .gen import (  # noqa: F401
    CONFIGS,
    Config,
    activations,
    config_by_name,
    config_inputs,
    f16_uniform,
    normal,
    q4k_blocks,
    q6k_blocks,
    splitmix64,
    uniform01,
    uniform_bytes,
    weights,
)
