"""The engine-rate probe behind the choice of tensor-core kind: it runs, and
its numbers are the ones the design relies on (the fp16 UMMA at its nominal
4096 MACs per clock per SM for N >= 128, the int8 warp-level MMA far below)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_engine_rates():
    from quantized_int8_gemm_gb300 import build
    build.build()
    import quantized_int8_gemm_gb300 as mmq
    r = mmq.mmq_probe_engine_rates()
    assert mmq.mmq_last_device_error() == 0
    umma = r["umma_f16_mac_per_clk_per_sm"]
    assert 3600 <= umma["N128"] <= 4200, umma
    assert 3600 <= umma["N256"] <= 4200, umma
    assert 0 < umma["N64"] < umma["N128"], umma
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # even at 2.1 GHz the whole GPU's fp16 UMMA rate is > 10x the int8 mma.sync rate measured here
    assert r["mma_sync_s8_tops"] > 0 and 10 * r["mma_sync_s8_tops"] < 2 * umma["N128"] * sms * 1.0e9 / 1e12, r
    assert r["mma_sync_f16_tflops"] > 0, r
