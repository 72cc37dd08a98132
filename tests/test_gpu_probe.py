"""The tensor-core rate probe (gemm_tc_rate_probe): the dense kind::f16 rate
per SM that the FP16 path's nominal peak is built from."""
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
