"""The bounded-wait watchdog: a wait that can never complete gives up after its
limit, the kernel returns, gemm_check reports GEMM_ERR_TIMEOUT once, and the
context stays usable for the next GEMM.  No fault, trap or hang is involved."""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F16, TOL_F32, assert_within

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



@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (300, 1000, 512)])
def test_stalled_gemm_pipeline_times_out_and_recovers(M, N, K):
    """The single-CTA tensor-core GEMM with its producer switched off: the MMA
    and epilogue waits give up after a few ms, the kernel returns without
    writing C, gemm_check reports the timeout once, and the same buffers then
    give the right product."""
    import time
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=M + K, bias=True)
    A = torch.from_numpy(d["A"]).cuda()
    B = torch.from_numpy(d["B"]).cuda()
    C = torch.full((M, N), 1234.5, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert g.check() == g.GEMM_OK
    t0 = time.perf_counter()
    st = g.pipeline_stall_selftest_raw(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), 5, stream)
    assert st == g.GEMM_OK, g.status_string(st)
    assert g.last_plan() == "tc_128x128_stalled_producer"
    assert g.check() == g.GEMM_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.0  # two 5 ms waits in a row, not the 2 s default
    assert g.check() == g.GEMM_OK  # cleared
    assert (C == 1234.5).all()     # nothing was stored
    # the same buffers through the ordinary path
    bias = torch.from_numpy(d["bias"]).cuda()
    g.gemm_f16_f32acc_epilogue(A, B, C, alpha=0.5, beta=0.0, bias=bias, act=1)
    assert g.check() == g.GEMM_OK
    ref, S = oracle.gemm(d["A"], d["B"], None, alpha=0.5, bias=d["bias"], act=1)
    assert_within(C.cpu().numpy(), ref, S, TOL_F16, f"after the stalled pipeline [{g.last_plan()}]", bias=d["bias"])


def test_stalled_pipeline_selftest_rejects_bad_arguments():
    A = torch.zeros(128, 256, dtype=torch.float16, device="cuda")
    B = torch.zeros(256, 128, dtype=torch.float16, device="cuda")
    C = torch.zeros(128, 128, device="cuda")
    f = g.pipeline_stall_selftest_raw
    assert f(128, 128, 256, A.data_ptr(), B.data_ptr(), C.data_ptr(), 0) == g.GEMM_ERR_INVALID_ARG
    assert f(128, 128, 256, A.data_ptr(), B.data_ptr(), C.data_ptr(), 2001) == g.GEMM_ERR_INVALID_ARG
    assert f(0, 128, 256, A.data_ptr(), B.data_ptr(), C.data_ptr(), 5) == g.GEMM_ERR_INVALID_ARG
    assert f(128, 128, 256, 0, B.data_ptr(), C.data_ptr(), 5) == g.GEMM_ERR_INVALID_ARG
    assert f(128, 128, 252, A.data_ptr(), B.data_ptr(), C.data_ptr(), 5) == g.GEMM_ERR_UNSUPPORTED
    assert f(128, 128, 256, A.data_ptr() + 2, B.data_ptr(), C.data_ptr(), 5) == g.GEMM_ERR_UNSUPPORTED
