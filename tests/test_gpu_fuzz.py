"""Seeded randomized parity sweep over every GPU entry point: random shapes
(edge sizes included), scalars, activations, element types, batches and B
layouts, each compared with the CPU oracle (row-sampled for large outputs)
under the path's own bound.  Reproducible: every case derives from its index."""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F16, TOL_F32, assert_within, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402

DEV = torch.device("cuda:0")
TORCH_T = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
EDGE = (1, 2, 7, 8, 31, 64, 65, 127, 128, 129, 255, 256, 257)


def _dim(rng, hi, mult=1):
    v = int(rng.choice(EDGE)) if rng.random() < 0.4 else int(rng.integers(1, hi))
    return max(mult, (v + mult - 1) // mult * mult)


def _rows(M, rng):
    return None if M <= 300 else sample_rows(M, seed=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("case", range(40))
def test_fuzz_f32(case):
    rng = np.random.default_rng(1000 + case)
    M, N, K = _dim(rng, 1500), _dim(rng, 1500), _dim(rng, 1200)
    lda, ldb, ldc = K + int(rng.integers(0, 5)), N + int(rng.integers(0, 5)), N + int(rng.integers(0, 5))
    alpha, beta = float(rng.choice([1.0, -0.5, 2.25])), float(rng.choice([0.0, 1.0, -1.5]))
    d = inputs.make(M, N, K, kind="f32", dist="normal", seed=case, beta=beta, lda=lda, ldb=ldb, ldc=ldc)
    A, B, C = (torch.from_numpy(d[k]).to(DEV) for k in ("A", "B", "C"))
    g.gemm_f32(A[:, :K], B[:, :N], C[:, :N], alpha=alpha, beta=beta)
    assert g.check() == g.GEMM_OK
    plan = g.last_plan()
    got = C.cpu().numpy()
    rows = _rows(M, rng)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=alpha, beta=beta, K=K, N=N, rows=rows)
    sel = got[:, :N] if rows is None else got[rows, :N]
    assert_within(sel, ref, S, TOL_F32, f"case {case}: {M}x{N}x{K} ld {lda},{ldb},{ldc} [{plan}]")
    np.testing.assert_array_equal(got[:, N:], d["C"][:, N:])  # padding untouched


@pytest.mark.parametrize("case", range(40))
def test_fuzz_tensor_core(case):
    rng = np.random.default_rng(2000 + case)
    batch = int(rng.choice([1, 1, 2, 3]))
    M, N, K = _dim(rng, 1200), _dim(rng, 2000, 8), _dim(rng, 2000, 8)
    in_kind = str(rng.choice(["f16", "bf16"]))
    out = str(rng.choice(["f32", "f32", "f16", "bf16"]))
    b_trans = bool(rng.random() < 0.35)
    act = int(rng.integers(0, 4))
    alpha, beta = float(rng.choice([1.0, 0.5, -1.25])), float(rng.choice([0.0, 0.0, 1.0, -0.75]))
    bias = bool(rng.random() < 0.5)
    d = inputs.make_batched(batch, M, N, K, kind=in_kind, dist="normal_k", seed=case, beta=beta, bias=bias,
                            b_trans=b_trans)
    C0 = d["C"].astype(np.float64) if (out == "f32" or beta == 0.0) else oracle.round_to(out, d["C"])
    A = torch.from_numpy(d["A"]).to(TORCH_T[in_kind]).to(DEV)
    B = torch.from_numpy(d["B"]).to(TORCH_T[in_kind]).to(DEV)
    C = torch.from_numpy(C0.astype(np.float32)).to(TORCH_T[out]).to(DEV)
    b = torch.from_numpy(d["bias"]).to(DEV) if bias else None
    g.gemm_tc_batched(A, B, C, alpha=alpha, beta=beta, bias=b, act=act, b_trans=b_trans)
    assert g.check() == g.GEMM_OK
    plan = g.last_plan()
    got = C.float().cpu().numpy().astype(np.float64)
    for z in range(batch):
        rows = _rows(M, rng)
        Bz = d["B"][z].T if b_trans else d["B"][z]
        ref, S = oracle.gemm(d["A"][z], Bz, C0[z] if beta != 0.0 else None, alpha=alpha, beta=beta,
                             bias=d.get("bias"), act=act, rows=rows)
        sel = got[z] if rows is None else got[z][rows]
        assert_within(sel, ref, S, TOL_F16,
                      f"case {case}: {batch}x{M}x{N}x{K} {in_kind}->{out} trans={b_trans} act={act} [{plan}]", out=out, bias=d.get("bias"))


@pytest.mark.parametrize("case", range(12))
def test_fuzz_3xtf32(case):
    rng = np.random.default_rng(3000 + case)
    M, N, K = _dim(rng, 1500), _dim(rng, 1500), _dim(rng, 1500)
    ldc = (N + 3) // 4 * 4
    alpha, beta = float(rng.choice([1.0, -0.5])), float(rng.choice([0.0, 1.0]))
    d = inputs.make(M, N, K, kind="f32", dist="uniform", seed=case, beta=beta, ldc=ldc)
    A, B = torch.from_numpy(d["A"]).to(DEV), torch.from_numpy(d["B"]).to(DEV)
    C = torch.from_numpy(d["C"]).to(DEV)
    g.gemm_f32_3xtf32(A, B, C[:, :N], alpha=alpha, beta=beta)
    assert g.check() == g.GEMM_OK
    plan = g.last_plan()
    rows = _rows(M, rng)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=alpha, beta=beta, N=N, rows=rows)
    got = C.cpu().numpy()
    sel = got[:, :N] if rows is None else got[rows, :N]
    assert_within(sel, ref, S, TOL_F32, f"case {case}: {M}x{N}x{K} [{plan}]")
