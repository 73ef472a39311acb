"""The C-ABI library builds, loads without a GPU and exports every symbol
include/mmq.h declares (no compute calls are made here)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "mmq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mmq_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from quantized_int8_gemm_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for n in ("mmq_quantize_act", "mmq_register_weights", "mmq_gemm", "mmq_weights_wexp",
              "mmq_release_weights", "mmq_last_device_error", "mmq_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_names_match_header():
    from quantized_int8_gemm_gb300 import mmq
    assert sorted(mmq.EXPORTS) == _declared_symbols()


def test_binding_flag_values_match_header():
    """The flag and arm constants the binding passes are the header's."""
    from quantized_int8_gemm_gb300 import mmq
    src = open(os.path.join(ROOT, "include", "mmq.h")).read()
    defs = {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define\s+(MMQ_(?:ARM|REG)_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|[0-9]+)u?\b", src)}
    assert {"MMQ_ARM_PAIR", "MMQ_ARM_SPLIT", "MMQ_REG_RAW"} <= set(defs)
    for name, value in defs.items():
        assert getattr(mmq, name) == value, name


def test_strerror_and_argument_checks_without_gpu(lib):
    lib.mmq_strerror.restype = ctypes.c_char_p
    assert lib.mmq_strerror(0) == b"ok"
    assert b"argument" in lib.mmq_strerror(-1)
    # host-side validation runs before any device call
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.mmq_quantize_act.argtypes = [vp, i64, i64, vp, vp]
    assert lib.mmq_quantize_act(None, 4, 33, None, None) == -1          # id % 32 != 0
    assert lib.mmq_quantize_act(None, 0, 64, None, None) == 0           # nt == 0: no-op
    lib.mmq_register_weights.argtypes = [ctypes.c_int, vp, i64, i64, ctypes.c_uint32, vp,
                                         ctypes.POINTER(vp)]
    h = vp()
    assert lib.mmq_register_weights(7, vp(16), 4, 256, 0, None, ctypes.byref(h)) == -3
    assert lib.mmq_register_weights(14, vp(16), 4, 300, 0, None, ctypes.byref(h)) == -1
    assert lib.mmq_register_weights(12, vp(16), 4, 256, 0x80, None, ctypes.byref(h)) == -1  # unknown flag
    lib.mmq_gemm.argtypes = [vp, vp, i64, vp, vp, ctypes.c_uint32, ctypes.POINTER(ctypes.c_int)]
    assert lib.mmq_gemm(None, None, 4, None, None, 0, None) == -1


def test_oracle_and_product_share_no_code():
    """The product sources never include, import or name the oracle."""
    pkg = os.path.join(ROOT, "quantized_int8_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f
    for f in os.listdir(os.path.join(ROOT, "include")):
        assert "oracle" not in open(os.path.join(ROOT, "include", f)).read().lower()
