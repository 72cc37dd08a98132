"""The roofline accounting reproduces the figures the pages print for 4096^3."""
import os

import pytest

from dense_gemm_11_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accounting_4096.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, value, _unit = line.split(None, 2)
        vals[key] = float(value)
    return vals


def _close(x, printed):
    # The pages round or truncate to the digits they print: allow one unit there.
    digits = len(repr(printed).split(".")[1]) if "." in repr(printed) and not repr(printed).endswith(".0") else 0
    return abs(x - printed) <= 10 ** (-digits) + 1e-9


def test_pages_accounting_4096():
    g = _golden()
    n = 4096
    f = roofline.gemm_flops(n, n, n)
    assert _close(f / 1e9, g["flops_fp32_4096"])
    b = roofline.gemm_bytes(n, n, n, in_bytes=4, beta_nonzero=True)
    assert _close(b / 1e6, g["bytes_fp32_4096_beta"])
    assert _close(f / b, g["ai_fp32_4096_beta"])
    b0 = roofline.gemm_bytes(n, n, n, in_bytes=4, beta_nonzero=False)
    assert _close(b0 / 1e6, g["bytes_fp32_4096_nobeta"])
    assert _close(f / b0, g["ai_fp32_4096_nobeta"])
    bin16 = roofline.gemm_bytes(n, n, n, in_bytes=2, beta_nonzero=False, out_bytes=0)
    assert _close(bin16 / 1e6, g["bytes_fp16_inputs_4096"])
    assert _close(f / bin16, g["ai_fp16_inputs_4096"])


def test_roofline_min():
    # A GEMV-like shape is HBM-bound, a large square is compute-bound.
    t, bound = roofline.roofline_tflops(roofline.gemm_flops(1, 4096, 4096),
                                        roofline.gemm_bytes(1, 4096, 4096, in_bytes=4, beta_nonzero=False),
                                        80.0, 6698.2)
    assert bound == "hbm" and t < 5
    t, bound = roofline.roofline_tflops(roofline.gemm_flops(4096, 4096, 4096),
                                        roofline.gemm_bytes(4096, 4096, 4096, in_bytes=4, beta_nonzero=True),
                                        80.0, 6698.2)
    assert bound == "compute" and t == 80.0
    assert roofline.fp32_fma_peak_tflops(152, 2070.0) == pytest.approx(80.55, abs=0.01)
