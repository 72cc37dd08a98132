"""BF16-input / FP32-accumulate GEMM (tcgen05, the FP16 kernels with BF16
operand formats) parity against the CPU oracle, elementwise within
|C - C_ref| <= 2e-3 * S + 1e-6, exact for small integers.  Called through the
C ABI (ctypes binding).  Products of two BF16 values are exact in FP32, so the
bound is the FP16 path's."""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F16, assert_within, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402

DEV = torch.device("cuda:0")


def to_bf16(x):
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), x), "input is not bf16-exact"
    return t.to(DEV)


def run_bf16(d, alpha, beta, bias=None, act=0):
    A = to_bf16(d["A"])
    B = to_bf16(d["B"])
    C = torch.from_numpy(d["C"]).to(DEV)
    b = torch.from_numpy(bias).to(DEV) if bias is not None else None
    g.gemm_bf16_f32acc_epilogue(A, B, C, alpha=alpha, beta=beta, bias=b, act=act)
    st = g.check()
    assert st == g.GEMM_OK, g.status_string(st)
    return C.cpu().numpy(), g.last_plan()


def check_workload(name, rows=None, exact=False):
    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(w)
    bias = d.get("bias")
    got, plan = run_bf16(d, w.alpha, w.beta, bias, w.act)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=w.alpha, beta=w.beta, bias=bias, act=w.act, rows=rows)
    sel = got if rows is None else got[rows]
    if exact:
        np.testing.assert_array_equal(sel.astype(np.float64), ref, err_msg=f"{name} [{plan}]")
        return plan
    assert_within(sel, ref, S, TOL_F16, f"{name} [{plan}]", bias=bias)
    return plan


def test_bf16_4096_sampled():
    check_workload("bf16_4096", rows=sample_rows(4096, seed=13))


def test_bf16_4096_small_integers_exact():
    check_workload("bf16_4096_int", rows=sample_rows(4096, seed=14), exact=True)


@pytest.mark.parametrize("i", [0, 1, 2, 3])
def test_bf16_epilogue_shapes(i):
    w = inputs.WORKLOADS[f"bf16_epi{i}"]
    rows = None if w.M <= 128 else sample_rows(w.M, seed=15 + i)
    check_workload(f"bf16_epi{i}", rows=rows)


@pytest.mark.parametrize("M", [1, 17, 64, 65, 128, 129, 300])
@pytest.mark.parametrize("N,K", [(8, 8), (264, 136), (520, 1032)])
@pytest.mark.parametrize("act", [0, 3])
def test_bf16_ragged_shapes(M, N, K, act):
    d = inputs.make(M, N, K, kind="bf16", dist="normal_k", seed=M * 7 + N + K, beta=0.0, bias=True)
    got, plan = run_bf16(d, 1.5, 0.0, d["bias"], act)
    ref, S = oracle.gemm(d["A"], d["B"], None, alpha=1.5, beta=0.0, bias=d["bias"], act=act)
    assert_within(got, ref, S, TOL_F16, f"{M}x{N}x{K} act={act} [{plan}]", bias=d["bias"])


@pytest.mark.parametrize("M,N,K", [(16, 4096, 1024), (128, 1024, 4096), (384, 512, 640), (5, 64, 4096),
                                   (2048, 4096, 512), (2000, 4000, 1032)])
def test_bf16_small_integers_exact_paths(M, N, K):
    d = inputs.make(M, N, K, kind="bf16", dist="smallint", seed=16, beta=2.0)
    got, plan = run_bf16(d, 1.0, 2.0)
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)


@pytest.mark.parametrize("M,N,K", [(129, 9728, 128), (1000, 4000, 520), (4100, 4104, 64)])
@pytest.mark.parametrize("act", [2, 3])
def test_bf16_cta_pair_ragged(M, N, K, act):
    d = inputs.make(M, N, K, kind="bf16", dist="normal_k", seed=M + N + K + 1, beta=0.25, bias=True)
    got, plan = run_bf16(d, -0.75, 0.25, d["bias"], act)
    assert "pair" in plan
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=-0.75, beta=0.25, bias=d["bias"], act=act)
    assert_within(got, ref, S, TOL_F16, f"{M}x{N}x{K} act={act} [{plan}]", bias=d["bias"])


def test_bf16_values_outside_fp16_range():
    # Entries near 2**20 overflow FP16 but are ordinary BF16 numbers; a kernel
    # that read the operands as FP16 would produce inf or garbage here.
    rng = np.random.default_rng(17)
    M, N, K = 256, 512, 256
    A = inputs.round_to_bf16(rng.uniform(-1, 1, (M, K)) * 2.0 ** 20)
    B = inputs.round_to_bf16(rng.uniform(-1, 1, (K, N)) * 2.0 ** -12)
    d = {"A": A, "B": B, "C": np.full((M, N), np.nan, dtype=np.float32)}
    got, plan = run_bf16(d, 1.0, 0.0)
    ref, S = oracle.gemm(A, B, None, alpha=1.0, beta=0.0)
    assert np.isfinite(got).all(), plan
    assert_within(got, ref, S, TOL_F16, f"wide range [{plan}]")


def test_bf16_and_f16_paths_agree_on_shared_values():
    # Small integers are exact in both formats: the two entry points must give
    # bit-identical results (same kernels, same summation order).
    d = inputs.make(512, 1024, 768, kind="bf16", dist="smallint", seed=18)
    got_bf, plan = run_bf16(d, 1.0, 0.0)
    A = torch.from_numpy(d["A"].astype(np.float16)).to(DEV)
    B = torch.from_numpy(d["B"].astype(np.float16)).to(DEV)
    C = torch.empty(512, 1024, device=DEV)
    g.gemm_f16_f32acc_epilogue(A, B, C)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got_bf, C.cpu().numpy(), err_msg=plan)


def test_bf16_rejects_fp16_tensors():
    A = torch.zeros(8, 8, dtype=torch.float16, device=DEV)
    C = torch.zeros(8, 8, device=DEV)
    with pytest.raises(TypeError):
        g.gemm_bf16_f32acc_epilogue(A, A, C)
