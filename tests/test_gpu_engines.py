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
    assert 0 < umma["N64"] < umma["N96"] < umma["N112"] <= umma["N128"], umma
    # on an SM pair (M = 256) the pair arm's 112-token tiles run at the full rate
    pair = r["umma_pair_f16_mac_per_clk_per_sm"]
    for n in ("N112", "N128", "N256"):
        assert 3600 <= pair[n] <= 4200, pair
    assert 0 < pair["N64"] < pair["N112"], pair
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # even at a 1.5 GHz SM clock the whole GPU's fp16 UMMA rate is > 10x the int8 mma.sync rate measured here
    umma_tflops_at_1p5ghz = 2 * umma["N128"] * sms * 1.5e9 / 1e12
    assert 0 < 10 * r["mma_sync_s8_tops"] < umma_tflops_at_1p5ghz, r
    # the warp-level f16 MMA stays below the fp16 UMMA as well
    assert 0 < r["mma_sync_f16_tflops"] < umma_tflops_at_1p5ghz * 2070 / 1500, r
