"""FP32 GEMM on the tensor cores through three TF32 products
(gemm_f32_3xtf32) against the CPU oracle, with the FP32 path's bound
|C - C_ref| <= 1e-5 * S + 1e-6.  Called through the C ABI."""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F32, assert_within, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402

DEV = torch.device("cuda:0")


def run(d, alpha, beta):
    A, B, C = (torch.from_numpy(d[k]).to(DEV) for k in ("A", "B", "C"))
    g.gemm_f32_3xtf32(A, B, C, alpha=alpha, beta=beta)
    st = g.check()
    assert st == g.GEMM_OK, g.status_string(st)
    return C.cpu().numpy(), g.last_plan()


@pytest.mark.parametrize("name", ["f32_512", "f32_sq128", "f32_sq1024", "f32_irr0"])
def test_3xtf32_workloads(name):
    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(w)
    got, plan = run(d, w.alpha, w.beta)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=w.alpha, beta=w.beta)
    err = assert_within(got, ref, S, TOL_F32, f"{name} [{plan}]")
    assert plan.startswith("tf32x3")
    assert err < 2e-6, f"{name}: max |err|/S {err:.2e}"  # the method's own level, well inside 1e-5


def test_3xtf32_4096_sampled():
    w = inputs.WORKLOADS["f32_sq4096"]
    d = inputs.make_workload(w)
    got, plan = run(d, w.alpha, w.beta)
    rows = sample_rows(4096, seed=41)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=w.alpha, beta=w.beta, rows=rows)
    assert_within(got[rows], ref, S, TOL_F32, f"4096^3 [{plan}]")


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (129, 260, 33), (300, 516, 1000), (257, 4, 129), (1000, 3000, 777),
                                   (64, 1024, 4099)])
def test_3xtf32_ragged(M, N, K):
    ldc = (N + 3) // 4 * 4 + 4
    d = inputs.make(M, N, K, kind="f32", dist="normal", seed=M + N + K, beta=-0.5, ldc=ldc)
    A, B = torch.from_numpy(d["A"]).to(DEV), torch.from_numpy(d["B"]).to(DEV)
    Cfull = torch.from_numpy(d["C"]).to(DEV)
    g.gemm_f32_3xtf32(A, B, Cfull[:, :N], alpha=0.7, beta=-0.5)
    assert g.check() == g.GEMM_OK
    got, plan = Cfull.cpu().numpy(), g.last_plan()
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=0.7, beta=-0.5, K=K, N=N)
    assert_within(got[:, :N], ref, S, TOL_F32, f"{M}x{N}x{K} [{plan}]")
    # the padding columns of C beyond N are not written
    np.testing.assert_array_equal(got[:, N:], d["C"][:, N:])


def test_3xtf32_unaligned_operands_and_strides():
    # A and B with odd leading dimensions and offsets: the split pass reads any layout.
    M, N, K = 200, 264, 300
    rng = np.random.default_rng(42)
    Abuf = torch.from_numpy(rng.normal(size=(M * 301 + 1,)).astype(np.float32)).to(DEV)
    Bbuf = torch.from_numpy(rng.normal(size=(K * 267 + 3,)).astype(np.float32)).to(DEV)
    A = Abuf[1:1 + M * 301].view(M, 301)[:, :K]
    B = Bbuf[3:3 + K * 267].view(K, 267)[:, :N]
    C = torch.empty(M, N, device=DEV)
    g.gemm_f32_3xtf32(A, B, C)
    torch.cuda.synchronize()
    ref, S = oracle.gemm(A.cpu().numpy(), B.cpu().numpy())
    assert_within(C.cpu().numpy(), ref, S, TOL_F32, g.last_plan())


def test_3xtf32_small_integers_exact():
    # Integers in [-4, 4] are TF32 values with a zero low part: every product
    # and partial sum is exact, so the result equals the oracle bit for bit.
    d = inputs.make(512, 768, 1024, kind="f32", dist="smallint", seed=43, beta=2.0)
    got, plan = run(d, 1.0, 2.0)
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)


def test_3xtf32_needs_the_low_parts():
    # Values with mantissa bits below TF32's 10: a single TF32 product would be
    # off by ~2^-11 relative; the three-product form must stay at FP32 level.
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(44)
    A = (1.0 + rng.integers(1, 2 ** 12, (M, K)) * 2.0 ** -23).astype(np.float32)
    B = (1.0 + rng.integers(1, 2 ** 12, (K, N)) * 2.0 ** -23).astype(np.float32)
    d = {"A": A, "B": B, "C": np.full((M, N), np.nan, np.float32)}
    got, plan = run(d, 1.0, 0.0)
    ref, S = oracle.gemm(A, B)
    err = np.max(np.abs(got - ref) / S)
    assert err < 2e-6, f"max |err|/S {err:.2e} [{plan}]"


def test_3xtf32_alpha_zero_and_unsupported_c():
    C0 = torch.randn(33, 24, device=DEV)
    C = C0.clone()
    A = torch.full((33, 16), float("nan"), device=DEV)
    B = torch.full((16, 24), float("nan"), device=DEV)
    g.gemm_f32_3xtf32(A, B, C, alpha=0.0, beta=2.0)
    torch.cuda.synchronize()
    assert torch.equal(C, 2.0 * C0)
    Cbuf = torch.zeros(33 * 24 + 1, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32_3xtf32(torch.ones(33, 16, device=DEV), torch.ones(16, 24, device=DEV),
                          Cbuf[1:].view(33, 24))
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED
