"""ctypes marshalling for the C oracle in ``mmq_oracle.c`` (test infrastructure).

``build()`` compiles the C file with gcc into ``oracle/_build/liboracle.so``
(strict ISO C, ``-ffp-contract=off``, no fast-math).  Every function below is
argument marshalling only; the arithmetic is in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_K = 12
Q6_K = 14

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mmq_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            L.mmq_oracle_f32_to_f16.argtypes = [_ptr, _ptr, _i64]
            L.mmq_oracle_f16_to_f64.argtypes = [_ptr, _ptr, _i64]
            L.mmq_oracle_quantize_q8_0.argtypes = [_ptr, _i64, _i64, _ptr]
            L.mmq_oracle_quantize_q8_0.restype = ctypes.c_int
            L.mmq_oracle_dequant_act.argtypes = [_ptr, _i64, _i64, _ptr]
            L.mmq_oracle_q6k_centered.argtypes = [_ptr, ctypes.c_int]
            L.mmq_oracle_q6k_centered.restype = ctypes.c_int
            L.mmq_oracle_q4k_quant.argtypes = [_ptr, ctypes.c_int]
            L.mmq_oracle_q4k_quant.restype = ctypes.c_int
            L.mmq_oracle_q4k_scale_min.argtypes = [_ptr, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_int),
                                                   ctypes.POINTER(ctypes.c_int)]
            L.mmq_oracle_weight.argtypes = [ctypes.c_int, _ptr, ctypes.c_int]
            L.mmq_oracle_weight.restype = ctypes.c_double
            L.mmq_oracle_dequant_weights.argtypes = [ctypes.c_int, _ptr, _i64, _i64,
                                                     _i64, _i64, _ptr]
            L.mmq_oracle_dequant_weights.restype = ctypes.c_int
            L.mmq_oracle_expand_q6k_dense.argtypes = [_ptr, _i64, _i64, _ptr]
            L.mmq_oracle_expand_q6k_dense.restype = ctypes.c_int
            L.mmq_oracle_expand_q4k_dense.argtypes = [_ptr, _i64, _i64, _ptr]
            L.mmq_oracle_expand_q4k_dense.restype = ctypes.c_int
            for fn in (L.mmq_oracle_gemm_entries, L.mmq_oracle_gemm_entries_int):
                fn.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr, _i64, _ptr, _ptr,
                               _i64, _ptr]
                fn.restype = ctypes.c_int
            L.mmq_oracle_gemm.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr, _i64, _ptr]
            L.mmq_oracle_gemm.restype = ctypes.c_int
            L.mmq_oracle_gemm_mt.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr, _i64, _ptr,
                                             ctypes.c_int]
            L.mmq_oracle_gemm_mt.restype = ctypes.c_int
            L.mmq_oracle_chunk_partials.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr, _i64, _ptr]
            L.mmq_oracle_chunk_partials.restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _block_bytes(qtype: int) -> int:
    return {Q6_K: 210, Q4_K: 144}[qtype]


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().mmq_oracle_f32_to_f16(_p(x), _p(out), x.size)
    return out


def f16_to_f64(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().mmq_oracle_f16_to_f64(_p(h), _p(out), h.size)
    return out


def quantize_q8_0(X: np.ndarray) -> np.ndarray:
    """X (nt, id) fp32 -> Q (nt, id/32, 40) uint8 pad40 blocks."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    nt, id_ = X.shape
    Q = np.empty((nt, id_ // 32, 40), dtype=np.uint8)
    rc = lib().mmq_oracle_quantize_q8_0(_p(X), nt, id_, _p(Q))
    if rc != 0:
        raise ValueError(f"oracle quantize_q8_0 failed rc={rc}")
    return Q


def dequant_act(Q: np.ndarray, nt: int, id_: int) -> np.ndarray:
    Q = np.ascontiguousarray(Q, dtype=np.uint8)
    assert Q.size == nt * (id_ // 32) * 40
    out = np.empty((nt, id_), dtype=np.float64)
    lib().mmq_oracle_dequant_act(_p(Q), nt, id_, _p(out))
    return out


def q6k_centered(blk: np.ndarray, e: int) -> int:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size >= 210
    return lib().mmq_oracle_q6k_centered(_p(blk), int(e))


def q4k_quant(blk: np.ndarray, e: int) -> int:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size >= 144
    return lib().mmq_oracle_q4k_quant(_p(blk), int(e))


def q4k_scale_min(blk: np.ndarray, j: int) -> tuple[int, int]:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size >= 144
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().mmq_oracle_q4k_scale_min(_p(blk), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def weight(qtype: int, blk: np.ndarray, e: int) -> float:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size >= _block_bytes(qtype)
    return lib().mmq_oracle_weight(qtype, _p(blk), int(e))


def dequant_weights(qtype: int, W: np.ndarray, od: int, id_: int, o0: int = 0,
                    o1: int | None = None) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == od * (id_ // 256) * _block_bytes(qtype)
    o1 = od if o1 is None else o1
    out = np.empty((o1 - o0, id_), dtype=np.float64)
    rc = lib().mmq_oracle_dequant_weights(qtype, _p(W), od, id_, o0, o1, _p(out))
    if rc != 0:
        raise ValueError(f"oracle dequant_weights failed rc={rc}")
    return out


def expand_q6k_dense(W: np.ndarray, od: int, id_: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == od * (id_ // 256) * 210
    out = np.empty((od, id_), dtype=np.int8)
    rc = lib().mmq_oracle_expand_q6k_dense(_p(W), od, id_, _p(out))
    if rc != 0:
        raise ValueError(f"oracle expand_q6k_dense failed rc={rc}")
    return out


def expand_q4k_dense(W: np.ndarray, od: int, id_: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == od * (id_ // 256) * 144
    out = np.empty((od, id_), dtype=np.int8)
    rc = lib().mmq_oracle_expand_q4k_dense(_p(W), od, id_, _p(out))
    if rc != 0:
        raise ValueError(f"oracle expand_q4k_dense failed rc={rc}")
    return out


def _entries(fn, qtype, W, od, id_, Q, nt, ts, os_):
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Q = np.ascontiguousarray(Q, dtype=np.uint8)
    ts = np.ascontiguousarray(ts, dtype=np.int64)
    os_ = np.ascontiguousarray(os_, dtype=np.int64)
    assert ts.shape == os_.shape
    assert W.size == od * (id_ // 256) * _block_bytes(qtype)
    assert Q.size == nt * (id_ // 32) * 40
    y = np.empty(ts.shape, dtype=np.float64)
    rc = fn(qtype, _p(W), od, id_, _p(Q), nt, _p(ts), _p(os_), ts.size, _p(y))
    if rc != 0:
        raise ValueError(f"oracle gemm entries failed rc={rc}")
    return y


def gemm_entries(qtype, W, od, id_, Q, nt, ts, os_) -> np.ndarray:
    """Y[ts[i], os[i]] in fp64: dot of dequantized weights and activations."""
    return _entries(lib().mmq_oracle_gemm_entries, qtype, W, od, id_, Q, nt, ts, os_)


def gemm_entries_int(qtype, W, od, id_, Q, nt, ts, os_) -> np.ndarray:
    """Same entries via exact int64 sub-block partials, then the scales."""
    return _entries(lib().mmq_oracle_gemm_entries_int, qtype, W, od, id_, Q, nt, ts, os_)


def chunk_partials(qtype: int, W: np.ndarray, od: int, id_: int, Q: np.ndarray, nt: int) -> np.ndarray:
    """Exact int64 partial of every 32-element chunk, sub-block scales applied,
    d and the activation scale not: S (nt, id/32, od)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Q = np.ascontiguousarray(Q, dtype=np.uint8)
    assert W.size == od * (id_ // 256) * _block_bytes(qtype)
    assert Q.size == nt * (id_ // 32) * 40
    S = np.empty((nt, id_ // 32, od), dtype=np.int64)
    rc = lib().mmq_oracle_chunk_partials(qtype, _p(W), od, id_, _p(Q), nt, _p(S))
    if rc != 0:
        raise ValueError(f"oracle chunk_partials failed rc={rc}")
    return S


def gemm(qtype: int, W: np.ndarray, od: int, id_: int, Q: np.ndarray, nt: int) -> np.ndarray:
    """Full (nt, od) output in fp64 (small problems)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Q = np.ascontiguousarray(Q, dtype=np.uint8)
    assert W.size == od * (id_ // 256) * _block_bytes(qtype)
    assert Q.size == nt * (id_ // 32) * 40
    Y = np.empty((nt, od), dtype=np.float64)
    rc = lib().mmq_oracle_gemm(qtype, _p(W), od, id_, _p(Q), nt, _p(Y))
    if rc != 0:
        raise ValueError(f"oracle gemm failed rc={rc}")
    return Y


def host_threads() -> int:
    """Threads the host can run at once (the CPU baseline uses all of them)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def gemm_mt(qtype: int, W: np.ndarray, od: int, id_: int, Q: np.ndarray, nt: int,
            threads: int | None = None) -> np.ndarray:
    """gemm() with the weight rows shared out over `threads` host threads
    (default: all of them); the same values bit for bit."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Q = np.ascontiguousarray(Q, dtype=np.uint8)
    assert W.size == od * (id_ // 256) * _block_bytes(qtype)
    assert Q.size == nt * (id_ // 32) * 40
    Y = np.empty((nt, od), dtype=np.float64)
    n = host_threads() if threads is None else int(threads)
    rc = lib().mmq_oracle_gemm_mt(qtype, _p(W), od, id_, _p(Q), nt, _p(Y), n)
    if rc != 0:
        raise ValueError(f"oracle gemm_mt failed rc={rc}")
    return Y
