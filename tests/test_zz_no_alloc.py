"""The no-allocation entry point gemm_f16_f32acc_epilogue_noalloc.

It exists for callers that cannot let the library allocate device memory:
for example a serving loop that reserved its whole memory budget up front,
where a cudaMalloc can fail or stall every stream of the device.  Its split-K
scratch is a fixed array inside the library, shared by every call.

Checked here, through the C ABI:
  * two calls in a row agree with the oracle (FP16 tolerance) and with the
    allocating entry point gemm_f16_f32acc_epilogue on the same inputs, and
    small-integer inputs give the oracle's exact value on both calls;
  * the split-K shapes really run the plan that uses the fixed array;
  * after one warm-up call, further calls leave the device's free memory
    unchanged;
  * a shape whose partials do not fit even at two K splits is rejected
    without launching anything.
This file is named so that pytest collects it last.
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
KBM = 128                        # rows of B^T per tile of the transposed small-M plan


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _splits(sms, M, N, K):
    """The split count the entry point uses: the planner's count, lowered
    until the partial tiles fit in the fixed array."""
    tiles = -(-N // KBM)
    bn = 32 if M <= 32 else 64
    s = min(sms // tiles, (K // 64) // 2, 32) if tiles < sms else 1
    if s > 1:
        s = min(s, STATIC_PARTIAL_FLOATS // (tiles * KBM * bn))
    return s


def _noalloc(M, N, K, alpha, A, B, beta, C, bias, act, stream):
    st = g.gemm_f16_noalloc_raw(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), _ptr(bias), act,
                                stream)
    assert st == g.GEMM_OK, g.status_string(st)
    return g.last_plan()


@pytest.mark.parametrize("M,N,K,beta,with_bias,act", [
    (16, 4096, 4096, 0.0, True, 1),     # the M = 16 inference shape, GELU epilogue
    (5, 1024, 512, 0.5, False, 0),      # beta != 0 reads C
    (64, 2048, 1024, 0.0, True, 0),
    (64, 4864, 4096, 0.0, True, 3),     # 38 tiles: 4 splits would overflow the array, 3 fit
])
def test_noalloc_matches_oracle_and_allocating_entry_point(M, N, K, beta, with_bias, act):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=77 + M, beta=beta, bias=with_bias)
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    C0 = torch.from_numpy(d["C"]).to(DEV)
    bias = torch.from_numpy(d["bias"]).to(DEV) if with_bias else None
    stream = torch.cuda.current_stream().cuda_stream
    alpha = 0.5
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count

    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=alpha, beta=beta, bias=d.get("bias"), act=act)

    C_alloc = C0.clone()
    st = g.gemm_f16_raw(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C_alloc.data_ptr(), _ptr(bias), act,
                        stream)
    assert st == g.GEMM_OK, g.status_string(st)
    alloc_plan = g.last_plan()
    torch.cuda.synchronize()
    got_alloc = C_alloc.cpu().numpy().astype(np.float64)
    assert_within(got_alloc, ref, S, TOL_F16, f"allocating entry point [{alloc_plan}]", bias=d.get("bias"))

    for call in range(2):
        C = C0.clone()
        plan = _noalloc(M, N, K, alpha, A, B, beta, C, bias, act, stream)
        assert g.check() == g.GEMM_OK
        if _splits(sms, M, N, K) > 1:
            assert plan.endswith("splitk_static"), plan
        got = C.cpu().numpy()
        assert_within(got, ref, S, TOL_F16, f"call {call} vs oracle [{plan}]", bias=d.get("bias"))
        # and against the allocating entry point, within the same tolerance
        assert_within(got, got_alloc, S, TOL_F16, f"call {call} vs {alloc_plan} [{plan}]", bias=d.get("bias"))


@pytest.mark.parametrize("M,N,K", [(16, 2048, 1024), (64, 4864, 4096)])
def test_noalloc_small_integers_exact(M, N, K):
    # |sum| <= 16 K + 2 * 4 < 2^24: every partial sum is exact in FP32, so the
    # split-K reduction through the fixed array must give the exact value.
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=5 + M, beta=2.0)
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    C0 = torch.from_numpy(d["C"]).to(DEV)
    stream = torch.cuda.current_stream().cuda_stream
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    for call in range(2):
        C = C0.clone()
        plan = _noalloc(M, N, K, 1.0, A, B, 2.0, C, None, 0, stream)
        assert plan.endswith("splitk_static"), plan
        assert g.check() == g.GEMM_OK
        np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref, err_msg=f"call {call} [{plan}]")


def test_noalloc_calls_leave_free_device_memory_unchanged():
    M, N, K, n = 16, 4096, 4096, 5
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=3, beta=0.0, bias=True)
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    bias = torch.from_numpy(d["bias"]).to(DEV)
    outs = [torch.empty(M, N, device=DEV) for _ in range(n)]  # every buffer exists before the first call
    stream = torch.cuda.current_stream().cuda_stream
    # Call 1 is the warm-up: under lazy module loading it may be the call that
    # places the library's kernels (and the fixed array) on the device.
    _noalloc(M, N, K, 0.5, A, B, 0.0, outs[0], bias, 1, stream)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(DEV)
    for i in range(1, n):
        plan = _noalloc(M, N, K, 0.5, A, B, 0.0, outs[i], bias, 1, stream)
        assert plan.endswith("splitk_static"), plan
        torch.cuda.synchronize()
        free_i, _ = torch.cuda.mem_get_info(DEV)
        assert free_i == free0, f"call {i + 1}: free device memory {free0} -> {free_i}"
    assert g.check() == g.GEMM_OK
    ref, S = oracle.gemm(d["A"], d["B"], None, alpha=0.5, bias=d["bias"], act=1)
    for i in range(n):
        assert_within(outs[i].cpu().numpy(), ref, S, TOL_F16, f"call {i + 1}", bias=d["bias"])


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
    # M = 64 gives 128 x 64 fp32 partial tiles; a plan that splits K but
    # cannot keep even two splits' partials in the fixed array is rejected.
    kb = K // 64

    def planner_splits(t):
        return min(sms // t, kb // 2, 32)

    tiles = next((t for t in range(1, sms) if planner_splits(t) > 1 and STATIC_PARTIAL_FLOATS // (t * 128 * 64) < 2),
                 None)
    if tiles is None:
        pytest.skip("on this GPU every split-K plan fits the fixed scratch at two splits")
    N = tiles * 128
    A = torch.zeros(64, K, dtype=torch.float16, device=DEV)
    B = torch.zeros(K, N, dtype=torch.float16, device=DEV)
    C = torch.full((64, N), 7.0, device=DEV)
    st = g.gemm_f16_noalloc_raw(64, N, K, 1.0, A.data_ptr(), B.data_ptr(), 0.0, C.data_ptr(), 0, 0, stream)
    assert st == g.GEMM_ERR_SCRATCH_LIMIT, g.status_string(st)
    assert "scratch" in g.status_string(st)
    torch.cuda.synchronize()
    assert (C == 7.0).all()  # nothing was launched
