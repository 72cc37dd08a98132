"""The bounded-wait watchdog: a wait that can never complete gives up after its
limit, the kernel returns, gemm_check reports GEMM_ERR_TIMEOUT once, and the
context stays usable for the next GEMM.  No fault, trap or hang is involved."""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F32, assert_within

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402


def test_watchdog_timeout_is_reported_and_cleared():
    assert g.check() == g.GEMM_OK
    assert g.watchdog_selftest(20) == g.GEMM_OK
    assert g.check() == g.GEMM_ERR_TIMEOUT
    assert g.check() == g.GEMM_OK  # cleared by the first check
    # the context is still usable
    d = inputs.make(130, 140, 150, kind="f32", dist="uniform", seed=21, beta=0.5)
    A, B, C = (torch.from_numpy(d[k]).cuda() for k in ("A", "B", "C"))
    g.gemm_f32(A, B, C, alpha=1.0, beta=0.5)
    assert g.check() == g.GEMM_OK
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=0.5)
    assert_within(C.cpu().numpy(), ref, S, TOL_F32, "after watchdog")


def test_watchdog_selftest_rejects_bad_limits():
    assert g.watchdog_selftest(0) == g.GEMM_ERR_INVALID_ARG
    assert g.watchdog_selftest(5000) == g.GEMM_ERR_INVALID_ARG

