"""Tensor-core GEMM with a 16-bit C (FP16 or BF16 output, FP32 accumulate and
epilogue, one round-to-nearest-even at the end) against the CPU oracle.
Called through the C ABI (gemm_tc_f32acc_epilogue).  Tolerance: the FP16
path's 2e-3 * S + 1e-6 plus one rounding to the output format; small-integer
inputs are compared bit for bit with the oracle's exact value rounded once."""
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
TORCH_T = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def c_initial(C32, out):
    """The C0 the GPU starts from: C rounded to the output type (as float64)."""
    if np.isnan(C32).all():
        return C32
    return oracle.round_to(out, C32.astype(np.float64))


def run_tc(d, in_kind, out, alpha, beta, bias=None, act=0):
    A = torch.from_numpy(np.asarray(d["A"], dtype=np.float32)).to(TORCH_T[in_kind]).to(DEV)
    B = torch.from_numpy(np.asarray(d["B"], dtype=np.float32)).to(TORCH_T[in_kind]).to(DEV)
    C0 = c_initial(d["C"], out)
    C = torch.from_numpy(C0.astype(np.float32)).to(TORCH_T[out]).to(DEV)
    b = torch.from_numpy(bias).to(DEV) if bias is not None else None
    g.gemm_tc(A, B, C, alpha=alpha, beta=beta, bias=b, act=act)
    st = g.check()
    assert st == g.GEMM_OK, g.status_string(st)
    return C.float().cpu().numpy().astype(np.float64), C0, g.last_plan()


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("in_kind", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 1024), (16, 4096, 4096), (128, 11008, 1024), (200, 520, 264),
                                   (1, 8, 8), (65, 264, 136), (1000, 4000, 520)])
def test_out16_parity(in_kind, out, M, N, K):
    d = inputs.make(M, N, K, kind=in_kind, dist="normal_k", seed=M + N + K, beta=0.5, bias=True)
    act = (M + N) % 4
    got, C0, plan = run_tc(d, in_kind, out, 0.75, 0.5, d["bias"], act)
    rows = sample_rows(M, seed=19) if M > 512 else None
    ref, S = oracle.gemm(d["A"], d["B"], C0, alpha=0.75, beta=0.5, bias=d["bias"], act=act, rows=rows)
    sel = got if rows is None else got[rows]
    assert_within(sel, ref, S, TOL_F16, f"{in_kind}->{out} {M}x{N}x{K} act={act} [{plan}]", out=out, bias=d["bias"])


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 1024), (16, 1024, 2048), (128, 1024, 4096), (5, 64, 512),
                                   (384, 512, 640)])
def test_out16_small_integers_round_once(out, M, N, K):
    # The FP32 accumulation of small integers is exact, so the GPU's single
    # rounding to the output type must give the oracle's exact value rounded
    # once -- including the ties of values beyond 2**11 (FP16) or 2**8 (BF16).
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=20, beta=2.0)
    got, C0, plan = run_tc(d, "f16", out, 1.0, 2.0)
    ref, _ = oracle.gemm(d["A"], d["B"], C0, alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got, oracle.round_to(out, ref), err_msg=f"{out} [{plan}]")


def test_out16_f16_overflow_gives_inf():
    d = inputs.make(256, 256, 512, kind="f16", dist="smallint", seed=21)
    got, _, plan = run_tc(d, "f16", "f16", 256.0, 0.0)
    ref, _ = oracle.gemm(d["A"], d["B"], None, alpha=256.0, with_scale=False)
    want = oracle.round_to("f16", ref)
    assert np.isinf(want).any() and np.isfinite(want).any()
    np.testing.assert_array_equal(got, want, err_msg=plan)


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("act", [0, 2, 3])
def test_out16_alpha_zero_epilogue_only(out, act):
    rng = np.random.default_rng(22)
    C32 = rng.uniform(-2, 2, (33, 24)).astype(np.float32)
    C0 = c_initial(C32, out)
    bias = rng.normal(0, 0.1, 24).astype(np.float32)
    A = torch.full((33, 16), float("nan"), dtype=torch.float16, device=DEV)
    B = torch.full((16, 24), float("nan"), dtype=torch.float16, device=DEV)
    C = torch.from_numpy(C0.astype(np.float32)).to(TORCH_T[out]).to(DEV)
    g.gemm_tc(A, B, C, alpha=0.0, beta=-1.5, bias=torch.from_numpy(bias).to(DEV), act=act)
    torch.cuda.synchronize()
    assert g.last_plan() == "scale_c_batched"
    ref, S = oracle.gemm(np.zeros((33, 16)), np.zeros((16, 24)), C0, alpha=0.0, beta=-1.5, bias=bias, act=act)
    assert_within(C.float().cpu().numpy(), ref, S, 1e-6, f"alpha=0 {out} act={act}", out=out, bias=bias)


def test_out16_beta_zero_does_not_read_c():
    d = inputs.make(300, 264, 128, kind="bf16", dist="normal_k", seed=23, beta=0.0)
    A = torch.from_numpy(d["A"]).to(torch.bfloat16).to(DEV)
    B = torch.from_numpy(d["B"]).to(torch.bfloat16).to(DEV)
    C = torch.full((300, 264), float("nan"), dtype=torch.bfloat16, device=DEV)
    g.gemm_tc(A, B, C)
    torch.cuda.synchronize()
    assert torch.isfinite(C).all(), g.last_plan()


def test_out16_matches_f32_output_rounded():
    # Same inputs, same kernels: the 16-bit result is the FP32 result rounded
    # once (the FP32 path's value is exactly what the 16-bit store rounds).
    d = inputs.make(1024, 2048, 1024, kind="f16", dist="normal_k", seed=24, beta=0.0, bias=True)
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    bias = torch.from_numpy(d["bias"]).to(DEV)
    C32 = torch.empty(1024, 2048, device=DEV)
    g.gemm_tc(A, B, C32, alpha=0.5, bias=bias, act=1)
    for out in ("f16", "bf16"):
        C16 = torch.empty(1024, 2048, dtype=TORCH_T[out], device=DEV)
        g.gemm_tc(A, B, C16, alpha=0.5, bias=bias, act=1)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(C16.float().cpu().numpy().astype(np.float64),
                                      oracle.round_to(out, C32.cpu().numpy().astype(np.float64)),
                                      err_msg=f"{out} [{g.last_plan()}]")


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 512), (1024, 3072, 256), (4096, 11008, 512)])
def test_out16_pair_64_column_stores(out, M, N, K):
    # CTA-pair tiles 256 or 192 wide store a 16-bit C in 32 x 64 boxes.
    d = inputs.make(M, N, K, kind="bf16", dist="normal_k", seed=M + N, beta=0.5, bias=True)
    got, C0, plan = run_tc(d, "bf16", out, 1.25, 0.5, d["bias"], 3)
    assert plan.startswith("tc_pair_256x256") or plan.startswith("tc_pair_256x192"), plan
    rows = sample_rows(M, seed=51)
    ref, S = oracle.gemm(d["A"], d["B"], C0, alpha=1.25, beta=0.5, bias=d["bias"], act=3, rows=rows)
    assert_within(got[rows], ref, S, TOL_F16, f"{out} {M}x{N}x{K} [{plan}]", out=out, bias=d["bias"])


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_out16_pair_64_column_stores_exact(out):
    d = inputs.make(1024, 3072, 256, kind="f16", dist="smallint", seed=52, beta=2.0)
    got, C0, plan = run_tc(d, "f16", out, 1.0, 2.0)
    assert "pair" in plan, plan
    ref, _ = oracle.gemm(d["A"], d["B"], C0, alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got, oracle.round_to(out, ref), err_msg=plan)
