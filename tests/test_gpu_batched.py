"""Strided-batched tensor-core GEMM (gemm_tc_strided_batched) against the CPU
oracle applied to each matrix of the batch: op(B) = B or B^T (attention's
Q K^T has the keys stored N x K), shared operands (batch stride 0), padded
output strides, every output type, every plan (transposed small-M, 1-CTA,
CTA pair, split-K).  Tolerance 2e-3 * S + 1e-6 (+ one output rounding for a
16-bit C); small integers bit-exact."""
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
TORCH_T = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def dev16(x, kind):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(TORCH_T[kind]).to(DEV)


def c_start(C32, out):
    if np.isnan(C32).all() or out == "f32":
        return C32.astype(np.float64)
    return oracle.round_to(out, C32.astype(np.float64))


def oracle_batch(d, C0, alpha, beta, b_trans, act=0, rows=None, with_scale=True):
    refs, scales = [], []
    for z in range(d["A"].shape[0]):
        Bz = d["B"][z].T if b_trans else d["B"][z]
        r, S = oracle.gemm(d["A"][z], Bz, C0[z] if beta != 0.0 else None, alpha=alpha, beta=beta,
                           bias=d.get("bias"), act=act, rows=rows, with_scale=with_scale)
        refs.append(r)
        scales.append(S)
    return np.stack(refs), (np.stack(scales) if with_scale else None)


def run_batched(d, in_kind, out, alpha, beta, b_trans, act=0):
    C0 = c_start(d["C"], out)
    A, B = dev16(d["A"], in_kind), dev16(d["B"], in_kind)
    C = torch.from_numpy(C0.astype(np.float32)).to(TORCH_T[out]).to(DEV)
    bias = torch.from_numpy(d["bias"]).to(DEV) if "bias" in d else None
    g.gemm_tc_batched(A, B, C, alpha=alpha, beta=beta, bias=bias, act=act, b_trans=b_trans)
    st = g.check()
    assert st == g.GEMM_OK, g.status_string(st)
    return C.float().cpu().numpy().astype(np.float64), C0, g.last_plan()


# (batch, M, N, K): attention Q K^T (S x S x d) and P V (S x d x S) per head,
# small-M decode shapes, and a shape whose tiles need split-K.
SHAPES = [(8, 512, 512, 128), (8, 512, 128, 512), (12, 1, 256, 128), (6, 40, 264, 520), (4, 128, 512, 256),
          (3, 300, 136, 64), (2, 128, 128, 4096), (10, 128, 2048, 128)]


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("batch,M,N,K", SHAPES)
def test_batched_parity(batch, M, N, K, b_trans):
    d = inputs.make_batched(batch, M, N, K, kind="f16", seed=batch * 7 + M + N + K, beta=0.5, bias=True,
                            b_trans=b_trans)
    act = (M + K) % 4
    got, C0, plan = run_batched(d, "f16", "f32", 0.75, 0.5, b_trans, act)
    ref, S = oracle_batch(d, C0, 0.75, 0.5, b_trans, act)
    assert_within(got, ref, S, TOL_F16, f"{batch}x{M}x{N}x{K} trans={b_trans} [{plan}]", bias=d.get("bias"))


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("batch,M,N,K", [(4, 256, 512, 192), (5, 16, 1024, 2048), (3, 128, 384, 640),
                                         (2, 1024, 2048, 256), (7, 64, 136, 64)])
def test_batched_small_integers_exact(batch, M, N, K, b_trans):
    d = inputs.make_batched(batch, M, N, K, kind="bf16", dist="smallint", seed=31, beta=2.0, b_trans=b_trans)
    got, C0, plan = run_batched(d, "bf16", "f32", 1.0, 2.0, b_trans)
    ref, _ = oracle_batch(d, C0, 1.0, 2.0, b_trans, with_scale=False)
    np.testing.assert_array_equal(got, ref, err_msg=f"trans={b_trans} [{plan}]")


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("b_trans", [False, True])
def test_batched_out16_attention_scores(out, b_trans):
    # Q K^T scores of 16 heads, S = 256, d = 64, written as 16-bit.
    d = inputs.make_batched(16, 256, 256, 64, kind="bf16", seed=32, b_trans=b_trans)
    got, C0, plan = run_batched(d, "bf16", out, 0.125, 0.0, b_trans)
    ref, S = oracle_batch(d, C0, 0.125, 0.0, b_trans)
    assert_within(got, ref, S, TOL_F16, f"{out} trans={b_trans} [{plan}]", out=out)


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("M", [16, 128, 512])
def test_batched_shared_weight(M, b_trans):
    # One B for the whole batch (stride 0, a 2-D tensor): batched activations
    # times a shared weight matrix.
    batch, N, K = 6, 384, 256
    d = inputs.make_batched(batch, M, N, K, kind="f16", seed=33 + M, b_trans=b_trans)
    Bshared = d["B"][0]
    A = dev16(d["A"], "f16")
    C = torch.empty(batch, M, N, device=DEV)
    g.gemm_tc_batched(A, dev16(Bshared, "f16"), C, b_trans=b_trans)
    torch.cuda.synchronize()
    plan = g.last_plan()
    for z in range(batch):
        ref, S = oracle.gemm(d["A"][z], Bshared.T if b_trans else Bshared)
        assert_within(C[z].cpu().numpy(), ref, S, TOL_F16, f"z={z} trans={b_trans} [{plan}]")


def test_batched_expanded_a_and_padded_c():
    # A broadcast with torch.expand (batch stride 0) and C matrices separated
    # by padding that must stay untouched.
    batch, M, N, K = 5, 200, 136, 96
    d = inputs.make_batched(batch, M, N, K, kind="f16", seed=34)
    A1 = dev16(d["A"][0], "f16")
    A = A1.unsqueeze(0).expand(batch, M, K)
    assert A.stride(0) == 0
    pad = 8 * 11
    Cbuf = torch.full((batch, M * N + pad), 7.0, device=DEV)
    C = Cbuf[:, :M * N].view(batch, M, N)
    g.gemm_tc_batched(A, dev16(d["B"], "f16"), C)
    torch.cuda.synchronize()
    assert torch.all(Cbuf[:, M * N:] == 7.0)
    for z in range(batch):
        ref, S = oracle.gemm(d["A"][0], d["B"][z])
        assert_within(C[z].cpu().numpy(), ref, S, TOL_F16, f"z={z} [{g.last_plan()}]")


def test_single_gemm_with_transposed_b_matches_batched_of_one():
    d = inputs.make_batched(1, 1000, 4000, 264, kind="f16", seed=35, b_trans=True)
    got, C0, plan = run_batched(d, "f16", "f32", 1.0, 0.0, True)
    ref, S = oracle_batch(d, C0, 1.0, 0.0, True)
    assert "pair" in plan
    assert_within(got, ref, S, TOL_F16, f"[{plan}]")


def test_batched_alpha_zero_scales_every_matrix():
    batch, M, N = 4, 33, 24
    rng = np.random.default_rng(36)
    C0 = rng.uniform(-1, 1, (batch, M, N)).astype(np.float32)
    C = torch.from_numpy(C0).to(DEV)
    A = torch.zeros(batch, M, 16, dtype=torch.float16, device=DEV)
    B = torch.zeros(batch, 16, N, dtype=torch.float16, device=DEV)
    g.gemm_tc_batched(A, B, C, alpha=0.0, beta=-2.0, act=2)
    torch.cuda.synchronize()
    assert g.last_plan() == "scale_c_batched"
    np.testing.assert_array_equal(C.cpu().numpy(), np.maximum(-2.0 * C0, 0.0))


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("b_trans", [False, True])
def test_batched_small_m_cluster_split(out, b_trans):
    # Decode-like batch: 4 matrices of 8 x 2048 x 4096 -> 64 tiles, K split
    # over clusters; 16-bit or FP32 C with beta and bias.
    batch, M, N, K = 4, 8, 2048, 4096
    d = inputs.make_batched(batch, M, N, K, kind="bf16", seed=37, beta=1.5, bias=True, b_trans=b_trans)
    got, C0, plan = run_batched(d, "bf16", out, 0.5, 1.5, b_trans, act=3)
    assert "clusterk" in plan, plan
    ref, S = oracle_batch(d, C0, 0.5, 1.5, b_trans, act=3)
    assert_within(got, ref, S, TOL_F16, f"{out} trans={b_trans} [{plan}]", out=out, bias=d.get("bias"))
