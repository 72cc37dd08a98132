"""The no-allocation entry point gemm_f16_f32acc_epilogue_noalloc.

It exists for callers that cannot let the library allocate device memory
(for example a serving loop that reserved its whole memory budget up front,
where a cudaMalloc can fail or stall every stream of the device).  Its
split-K scratch is a fixed array inside the library, shared by every call.

Checked here, through the C ABI: two calls in a row give the same output as
the allocating entry point gemm_f16_f32acc_epilogue on the same inputs,
within the FP16 tolerance of the other tests; shapes beyond the fixed scratch
or beyond M <= 64 are rejected with their status codes.  This file is named
so that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F16, assert_within

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402

DEV = torch.device("cuda:0")
STATIC_PARTIAL_FLOATS = 1 << 20  # the fixed scratch: 4 MiB of fp32 partial tiles


def _ptr(t):
    return 0 if t is None else t.data_ptr()


@pytest.mark.parametrize("M,N,K,beta,with_bias,act", [
    (16, 4096, 4096, 0.0, True, 1),     # the M = 16 inference shape, GELU epilogue
    (5, 1024, 512, 0.5, False, 0),      # beta != 0 reads C
    (64, 2048, 1024, 0.0, True, 0),
])
def test_noalloc_matches_allocating_entry_point(M, N, K, beta, with_bias, act):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=77 + M, beta=beta, bias=with_bias)
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    C0 = torch.from_numpy(d["C"]).to(DEV)
    bias = torch.from_numpy(d["bias"]).to(DEV) if with_bias else None
    stream = torch.cuda.current_stream().cuda_stream
    alpha = 0.5

    C_ref = C0.clone()
    st = g.gemm_f16_raw(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C_ref.data_ptr(), _ptr(bias), act, stream)
    assert st == g.GEMM_OK, g.status_string(st)
    ref_plan = g.last_plan()
    torch.cuda.synchronize()

    _, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=alpha, beta=beta, bias=d.get("bias"), act=act)
    ref = C_ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        C = C0.clone()
        st = g.gemm_f16_noalloc_raw(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), _ptr(bias),
                                    act, stream)
        assert st == g.GEMM_OK, g.status_string(st)
        plan = g.last_plan()
        assert g.check() == g.GEMM_OK
        assert_within(C.cpu().numpy(), ref, S, TOL_F16, f"call {call} [{plan} vs {ref_plan}]")


def test_noalloc_rejects_shapes_beyond_its_limits():
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    K = 4096
    stream = torch.cuda.current_stream().cuda_stream
    # M > 64 is not this kernel's shape.
    A = torch.zeros(65, K, dtype=torch.float16, device=DEV)
    B = torch.zeros(K, 256, dtype=torch.float16, device=DEV)
    C = torch.zeros(65, 256, device=DEV)
    assert g.gemm_f16_noalloc_raw(65, 256, K, 1.0, A.data_ptr(), B.data_ptr(), 0.0, C.data_ptr(), 0, 0,
                                  stream) == g.GEMM_ERR_UNSUPPORTED
    # A split-K plan whose partial tiles exceed the fixed scratch: M = 64 gives
    # 128 x 64 fp32 partial tiles; the plan splits K min(SMs // tiles,
    # k-blocks // 2, 32) ways.
    kb = K // 64

    def splits(t):
        return min(sms // t, kb // 2, 32)

    tiles = next((t for t in range(1, sms) if splits(t) > 1 and t * splits(t) * 128 * 64 > STATIC_PARTIAL_FLOATS),
                 None)
    if tiles is None:
        pytest.skip("this GPU has too few SMs for any split-K plan to exceed the fixed scratch")
    N = tiles * 128
    A = torch.zeros(64, K, dtype=torch.float16, device=DEV)
    B = torch.zeros(K, N, dtype=torch.float16, device=DEV)
    C = torch.full((64, N), 7.0, device=DEV)
    st = g.gemm_f16_noalloc_raw(64, N, K, 1.0, A.data_ptr(), B.data_ptr(), 0.0, C.data_ptr(), 0, 0, stream)
    assert st == g.GEMM_ERR_SCRATCH_LIMIT, g.status_string(st)
    assert "scratch" in g.status_string(st)
    torch.cuda.synchronize()
    assert (C == 7.0).all()  # nothing was launched
