"""Tensor-core GEMM with K split over the CTAs of a thread-block cluster, not
transposed (few 128-row tiles: M <= 256 with a moderate N): each CTA computes
one K slice of a tile, the partials are added in split order through
distributed shared memory and the fused epilogue writes C.  Against the CPU
oracle: small integers bit-exact for every tile width and cluster size a
tuning table can force, random data within 2e-3 * S + 1e-6 (+ one output
rounding for a 16-bit C)."""
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


def run(d, alpha, beta, act=0, in_kind="f16", out="f32", b_trans=False):
    C0 = d["C"].astype(np.float64) if (out == "f32" or beta == 0.0) else oracle.round_to(out, d["C"])
    A = torch.from_numpy(np.asarray(d["A"], dtype=np.float32)).to(TORCH_T[in_kind]).to(DEV)
    B = torch.from_numpy(np.asarray(d["B"], dtype=np.float32)).to(TORCH_T[in_kind]).to(DEV)
    C = torch.from_numpy(C0.astype(np.float32)).to(TORCH_T[out]).to(DEV)
    bias = torch.from_numpy(d["bias"]).to(DEV) if "bias" in d else None
    g.gemm_tc_batched(A, B, C, alpha=alpha, beta=beta, bias=bias, act=act, b_trans=b_trans)
    st = g.check()
    assert st == g.GEMM_OK, g.status_string(st)
    return C.float().cpu().numpy().astype(np.float64), C0, g.last_plan()


@pytest.mark.parametrize("M,N,K,split", [(128, 4096, 4096, True), (256, 4096, 4096, True), (128, 2048, 8192, True),
                                         (100, 3000, 1000, False), (96, 8192, 2048, False),
                                         (128, 11008, 4096, False)])
def test_planner_splits_few_tiles_over_a_cluster(M, N, K, split):
    # split while whole 128 x 128 tiles would leave half the SMs idle and each
    # would stream long enough to repay the hand-over (K = 1000 / 2048: no)
    d = inputs.make_batched(1, M, N, K, kind="f16", seed=M + N, beta=0.0, bias=True)
    got, _, plan = run(d, 0.5, 0.0, act=1)
    assert ("clusterk" in plan) == split, plan
    rows = sample_rows(M, seed=60)
    ref, S = oracle.gemm(d["A"][0], d["B"][0], None, alpha=0.5, bias=d["bias"], act=1, rows=rows)
    assert_within(got[0][rows], ref, S, TOL_F16, f"{M}x{N}x{K} [{plan}]", bias=d["bias"])


@pytest.mark.parametrize("bn,cs", [(256, 2), (256, 3), (256, 8), (192, 2), (192, 5), (128, 4), (128, 3), (256, 0)])
def test_every_width_and_cluster_size_is_exact(bn, cs):
    # 2 tile rows (M = 200, the second ragged), a ragged last tile column and
    # 17 k blocks (uneven k slices); small integers are exact in any order.
    M, N, K = 200, 1000, 1088
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=61, beta=1.0)
    A, B, C = (torch.from_numpy(d[k]).to(DEV) for k in ("A", "B", "C"))
    try:
        g.tune_set([dict(path=g.GEMM_PATH_TC, M=M, N=N, K=K, variant=4, bn=bn, splits=cs)])
        g.gemm_f16_f32acc_epilogue(A, B, C, alpha=1.0, beta=1.0)
        assert g.check() == g.GEMM_OK
        plan = g.last_plan()
    finally:
        g.tune_set([])
    assert plan == f"tc_128x{bn}_clusterk+tuned" or (cs == 0 and plan.endswith("clusterk+tuned")), plan
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=1.0, with_scale=False)
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref, err_msg=plan)


def test_tuned_cluster_split_ignored_when_too_many_ctas():
    # 2048 x 4096 in 128 x 256 tiles split 8 ways would need 16 x 16 x 8 CTAs at once:
    # the entry is dropped and the planner's own plan (CTA pairs) runs
    M, N, K = 2048, 4096, 512
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=62)
    A, B, C = (torch.from_numpy(d[k]).to(DEV) for k in ("A", "B", "C"))
    try:
        g.tune_set([dict(path=g.GEMM_PATH_TC, M=M, N=N, K=K, variant=4, bn=256, splits=8)])
        g.gemm_f16_f32acc_epilogue(A, B, C, alpha=1.0, beta=0.0)
        assert g.check() == g.GEMM_OK
        plan = g.last_plan()
    finally:
        g.tune_set([])
    assert "pair" in plan and "+tuned" not in plan, plan
    rows = sample_rows(M, seed=63)
    ref, _ = oracle.gemm(d["A"], d["B"], None, with_scale=False, rows=rows)
    np.testing.assert_array_equal(C.cpu().numpy()[rows].astype(np.float64), ref, err_msg=plan)


@pytest.mark.parametrize("in_kind,out", [("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("b_trans", [False, True])
def test_batched_16bit_output_and_transposed_b(in_kind, out, b_trans):
    batch, M, N, K = 3, 96, 776, 2048
    d = inputs.make_batched(batch, M, N, K, kind=in_kind, seed=64, beta=-0.75, bias=True, b_trans=b_trans)
    got, C0, plan = run(d, 1.25, -0.75, act=3, in_kind=in_kind, out=out, b_trans=b_trans)
    assert "clusterk" in plan and "swap" not in plan, plan
    for z in range(batch):
        Bz = d["B"][z].T if b_trans else d["B"][z]
        ref, S = oracle.gemm(d["A"][z], Bz, C0[z], alpha=1.25, beta=-0.75, bias=d["bias"], act=3)
        assert_within(got[z], ref, S, TOL_F16, f"z={z} {in_kind}->{out} trans={b_trans} [{plan}]", out=out, bias=d["bias"])


def test_deterministic_across_calls():
    d = inputs.make(128, 4096, 4096, kind="f16", seed=65)
    A, B = torch.from_numpy(d["A"]).to(DEV), torch.from_numpy(d["B"]).to(DEV)
    C1 = torch.empty(128, 4096, device=DEV)
    C2 = torch.empty(128, 4096, device=DEV)
    g.gemm_f16_f32acc_epilogue(A, B, C1)
    g.gemm_f16_f32acc_epilogue(A, B, C2)
    torch.cuda.synchronize()
    assert "clusterk" in g.last_plan()
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("M,N,K,b_trans,out", [(128, 11008, 1024, False, "f32"), (100, 3000, 1000, False, "f32"),
                                               (100, 3000, 1000, True, "f32"), (96, 8192, 2048, True, "bf16"),
                                               (120, 9000, 1040, False, "f16")])
def test_96_wide_whole_tiles(M, N, K, b_trans, out):
    # fewer 128-wide tiles than SMs, 16 k blocks or more and no cluster split:
    # 96-wide tiles, one per SM.  Stored K x N, B's second 64-column box reaches 32 columns past
    # the tile (past N on the last one); stored N x K, the box is 96 rows.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    in_kind = "bf16" if out == "bf16" else "f16"
    # small integers: exact sums, one rounding to a 16-bit C
    d = inputs.make_batched(1, M, N, K, kind=in_kind, dist="smallint", seed=M + N, beta=1.0, b_trans=b_trans)
    got, C0, plan = run(d, 1.0, 1.0, in_kind=in_kind, out=out, b_trans=b_trans)
    if sms == 152:
        assert plan == "tc_128x96_epi8", plan
    B = d["B"][0].T if b_trans else d["B"][0]
    ref, _ = oracle.gemm(d["A"][0], B, C0[0], alpha=1.0, beta=1.0, with_scale=False)
    if out != "f32":
        ref = oracle.round_to(out, ref)
    np.testing.assert_array_equal(got[0], ref, err_msg=plan)
    # normal data with bias and an activation
    d = inputs.make_batched(1, M, N, K, kind=in_kind, seed=M + N + 1, beta=-0.5, bias=True, b_trans=b_trans)
    got, C0, plan = run(d, 0.75, -0.5, act=1, in_kind=in_kind, out=out, b_trans=b_trans)
    B = d["B"][0].T if b_trans else d["B"][0]
    ref, S = oracle.gemm(d["A"][0], B, C0[0], alpha=0.75, beta=-0.5, bias=d["bias"], act=1)
    assert_within(got[0], ref, S, TOL_F16, f"{M}x{N}x{K} {out} trans={b_trans} [{plan}]", out=out, bias=d["bias"])


def test_short_k_keeps_128_wide_tiles():
    # 9 k blocks: 128-wide whole tiles (96-wide measured slower there)
    d = inputs.make_batched(1, 120, 9000, 520, kind="f16", dist="smallint", seed=66, beta=0.0)
    got, C0, plan = run(d, 1.0, 0.0)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert plan == "tc_128x128_epi8", plan
    ref, _ = oracle.gemm(d["A"][0], d["B"][0], None, with_scale=False)
    np.testing.assert_array_equal(got[0], ref, err_msg=plan)
