"""The rate probes: gemm_tc_rate_probe, the dense kind::f16 rate per SM that
the FP16 path's nominal peak is built from, gemm_fma_rate_probe, the FP32
FMA throughput per SM of the packed (FFMA2) and scalar instruction forms, and
gemm_tma_read_probe, the bytes per SM clock a CTA receives through TMA."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402


def test_rate_is_plausible_and_stable():
    # issue-limited tensor pipe: the same FLOP per clock whatever the length
    r1 = g.tc_rate_probe(2048)
    r2 = g.tc_rate_probe(4096)
    assert 2048 <= r1 <= 32768, r1
    assert abs(r1 - r2) / r2 < 0.05, (r1, r2)


def test_nominal_peak_is_at_least_the_measured_one():
    # #SM x rate x max clock bounds what any kernel (cuBLAS included) reaches
    import json
    import os
    rate = g.tc_rate_probe()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nominal = rate * sms * 2070e6 / 1e12
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    if os.path.exists(path):
        measured = json.load(open(path)).get("bf16_tflops")
        if measured:
            assert nominal >= 0.9 * measured, (nominal, measured)


def test_bad_arguments():
    with pytest.raises(g.GemmError) as e:
        g.tc_rate_probe(0)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG


def test_fma_rate_probe_is_plausible():
    # 128 FP32 FMAs per clock per SM is the nominal peak; neither form can pass
    # it, and both reach a large part of it with independent chains
    packed = g.fma_rate_probe(True, 2048)
    scalar = g.fma_rate_probe(False, 2048)
    assert 40.0 <= packed <= 128.5, packed
    assert 40.0 <= scalar <= 128.5, scalar
    again = g.fma_rate_probe(True, 4096)
    assert abs(again - packed) / packed < 0.05, (packed, again)


def test_fma_rate_probe_bad_arguments():
    import ctypes
    out = ctypes.c_double(0.0)
    assert g.fma_rate_probe_raw(2, 1024, ctypes.addressof(out)) == g.GEMM_ERR_INVALID_ARG
    assert g.fma_rate_probe_raw(1, 0, ctypes.addressof(out)) == g.GEMM_ERR_INVALID_ARG
    assert g.fma_rate_probe_raw(1, 1024, 0) == g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("multicast", [False, True])
@pytest.mark.parametrize("region_mb", [24, 1024])
def test_tma_read_probe_is_plausible(multicast, region_mb):
    # a CTA cannot receive more than a few hundred bytes per SM clock; the
    # figure is stable from one launch to the next
    r = g.tma_read_probe(8, multicast=multicast, stages=4, kblocks=256, region_mb=region_mb)
    assert 4.0 <= r["bytes_per_clock_per_sm"] <= 512.0, r
    assert r["total_gbs"] > 0.0, r
    again = g.tma_read_probe(8, multicast=multicast, stages=4, kblocks=256, region_mb=region_mb)
    assert abs(again["bytes_per_clock_per_sm"] - r["bytes_per_clock_per_sm"]) <= 0.15 * r["bytes_per_clock_per_sm"], \
        (r, again)


def test_tma_read_probe_every_sm():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    r = g.tma_read_probe(sms // 2, stages=6, kblocks=512, region_mb=24)
    assert r["bytes_per_clock_per_sm"] > 0.0 and r["total_gbs"] > 0.0, r
    with pytest.raises(g.GemmError) as e:
        g.tma_read_probe(sms // 2 + 1)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
