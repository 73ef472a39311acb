"""CPU oracle for the k-quant x q8_0 MMQ GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or runs anything here, and
shares no code with it.

The arithmetic lives in ``mmq_oracle.c`` (plain C, fp64 accumulation); this
module only builds it with gcc and marshals numpy arrays through ctypes.
"""
from .oracle import (  # noqa: F401
    Q4_K,
    Q6_K,
    build,
    chunk_partials,
    dequant_act,
    dequant_weights,
    expand_q4k_dense,
    expand_q6k_dense,
    f16_to_f64,
    f32_to_f16,
    gemm,
    gemm_entries,
    gemm_entries_int,
    gemm_mt,
    host_threads,
    lib,
    q4k_quant,
    q4k_scale_min,
    q6k_centered,
    quantize_q8_0,
    weight,
)
