"""FP16-input / FP32-accumulate GEMM (tcgen05) parity against the CPU oracle,
elementwise within |C - C_ref| <= 2e-3 * S + 1e-6, exact for small integers.
Called through the C ABI (ctypes binding)."""
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


def run_f16(d, alpha, beta, bias=None, act=0):
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    C = torch.from_numpy(d["C"]).to(DEV)
    b = torch.from_numpy(bias).to(DEV) if bias is not None else None
    g.gemm_f16_f32acc_epilogue(A, B, C, alpha=alpha, beta=beta, bias=b, act=act)
    st = g.check()
    assert st == g.GEMM_OK, g.status_string(st)
    return C.cpu().numpy(), g.last_plan()


def check_workload(name, rows=None, exact=False):
    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(w)
    bias = d.get("bias")
    got, plan = run_f16(d, w.alpha, w.beta, bias, w.act)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=w.alpha, beta=w.beta, bias=bias, act=w.act, rows=rows)
    sel = got if rows is None else got[rows]
    if exact:
        np.testing.assert_array_equal(sel.astype(np.float64), ref, err_msg=f"{name} [{plan}]")
        return plan
    assert_within(sel, ref, S, TOL_F16, f"{name} [{plan}]", bias=bias)
    return plan


def test_f16_4096_sampled():
    check_workload("f16_4096", rows=sample_rows(4096, seed=3))


def test_f16_4096_small_integers_exact():
    check_workload("f16_4096_int", rows=sample_rows(4096, seed=4), exact=True)


@pytest.mark.parametrize("i", [0, 1, 2, 3])
def test_f16_epilogue_shapes(i):
    w = inputs.WORKLOADS[f"f16_epi{i}"]
    rows = None if w.M <= 128 else sample_rows(w.M, seed=5 + i)
    check_workload(f"f16_epi{i}", rows=rows)


@pytest.mark.parametrize("M", [1, 3, 16, 17, 32, 33, 64, 65, 127, 128, 129, 200, 300])
@pytest.mark.parametrize("N,K", [(8, 8), (136, 72), (264, 136), (520, 1032)])
def test_f16_ragged_shapes(M, N, K):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=M * 131 + N + K, beta=0.0, bias=True)
    got, plan = run_f16(d, 1.5, 0.0, d["bias"], 0)
    ref, S = oracle.gemm(d["A"], d["B"], None, alpha=1.5, beta=0.0, bias=d["bias"])
    assert_within(got, ref, S, TOL_F16, f"{M}x{N}x{K} [{plan}]", bias=d["bias"])


@pytest.mark.parametrize("M,N,K", [(16, 4096, 1024), (128, 1024, 4096), (384, 512, 640), (5, 64, 4096),
                                   (2048, 4096, 512), (2000, 4000, 1032)])
def test_f16_small_integers_exact_paths(M, N, K):
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=6, beta=2.0)
    got, plan = run_f16(d, 1.0, 2.0)
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (16, 1024, 2048), (2048, 4096, 1024)])
@pytest.mark.parametrize("act", [0, 1, 2, 3])
def test_f16_beta_and_bias_epilogue(M, N, K, act):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=7, beta=-0.5, bias=True)
    got, plan = run_f16(d, 0.5, -0.5, d["bias"], act)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=0.5, beta=-0.5, bias=d["bias"], act=act)
    assert_within(got, ref, S, TOL_F16, f"beta/bias act={act} [{plan}]", bias=d["bias"])


@pytest.mark.parametrize("M,N,K", [(129, 9728, 128), (300, 8448, 200), (1000, 4000, 520), (4100, 4104, 64)])
def test_f16_cta_pair_ragged(M, N, K):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=M + N + K, beta=0.25, bias=True)
    got, plan = run_f16(d, -0.75, 0.25, d["bias"], 1)
    assert "pair" in plan
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=-0.75, beta=0.25, bias=d["bias"], act=1)
    assert_within(got, ref, S, TOL_F16, f"{M}x{N}x{K} [{plan}]", bias=d["bias"])


def test_f16_beta_zero_does_not_read_c():
    d = inputs.make(300, 264, 128, kind="f16", dist="normal_k", seed=8, beta=0.0)
    got, plan = run_f16(d, 1.0, 0.0)
    assert np.isfinite(got).all(), plan


@pytest.mark.parametrize("act", [1, 2, 3])
def test_f16_alpha_zero_epilogue_only(act):
    rng = np.random.default_rng(9)
    C0 = rng.uniform(-1, 1, (33, 24)).astype(np.float32)
    bias = rng.normal(0, 0.1, 24).astype(np.float32)
    A = torch.full((33, 16), float("nan"), dtype=torch.float16, device=DEV)
    B = torch.full((16, 24), float("nan"), dtype=torch.float16, device=DEV)
    C = torch.from_numpy(C0).to(DEV)
    g.gemm_f16_f32acc_epilogue(A, B, C, alpha=0.0, beta=2.0, bias=torch.from_numpy(bias).to(DEV), act=act)
    torch.cuda.synchronize()
    ref, S = oracle.gemm(np.zeros((33, 16)), np.zeros((16, 24)), C0, alpha=0.0, beta=2.0, bias=bias, act=act)
    assert_within(C.cpu().numpy(), ref, S, 1e-6, f"alpha=0 act={act}", bias=bias)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (16, 4096, 4096), (128, 11008, 4096)])
def test_f16_deterministic(M, N, K):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=10, beta=0.0)
    a, plan = run_f16(d, 1.0, 0.0)
    b, _ = run_f16(d, 1.0, 0.0)
    np.testing.assert_array_equal(a, b, err_msg=plan)


def test_f16_unsupported_is_reported():
    A = torch.zeros(8, 12, dtype=torch.float16, device=DEV)
    B = torch.zeros(12, 8, dtype=torch.float16, device=DEV)
    C = torch.zeros(8, 8, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_f32acc_epilogue(A, B, C)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,N,K", [(256, 520, 128), (2048, 4096, 256), (40, 264, 64)])
def test_f16_unaligned_bias_pointer(M, N, K):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=31, beta=0.0, bias=True)
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    C = torch.from_numpy(d["C"]).to(DEV)
    buf = torch.zeros(N + 1, device=DEV)
    buf[1:] = torch.from_numpy(d["bias"]).to(DEV)
    bias = buf[1:]  # 4-byte aligned only
    assert bias.data_ptr() % 16 != 0
    g.gemm_f16_f32acc_epilogue(A, B, C, alpha=0.5, beta=0.0, bias=bias, act=1)
    assert g.check() == g.GEMM_OK
    ref, S = oracle.gemm(d["A"], d["B"], None, alpha=0.5, beta=0.0, bias=d["bias"], act=1)
    assert_within(C.cpu().numpy(), ref, S, TOL_F16, f"unaligned bias [{g.last_plan()}]", bias=d["bias"])


@pytest.mark.parametrize("act", [1, 2, 3])
def test_activation_accuracy_on_exact_preactivations(act):
    # Small-integer operands and a dyadic alpha make every pre-activation
    # exact in FP32 (x = k / 32, |x| up to about 7.6), so the only error left
    # is the activation's own: held to 1e-6 |x| + 1e-7, far inside the GEMM
    # bound.
    M, N, K = 256, 1024, 64
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=40)
    got, plan = run_f16(d, 1.0 / 32, 0.0, None, act)
    ref, _ = oracle.gemm(d["A"], d["B"], None, alpha=1.0 / 32, act=act, with_scale=False)
    x, _ = oracle.gemm(d["A"], d["B"], None, alpha=1.0 / 32, with_scale=False)
    assert np.unique(x).size > 400  # a dense sweep of the range
    err = np.abs(got.astype(np.float64) - ref)
    bound = 1e-6 * np.abs(x) + 1e-7 if act != 2 else np.zeros_like(x)
    assert np.all(err <= bound), f"act {act} [{plan}]: max err {err.max():.3e} at x={x.flat[np.argmax(err - bound)]}"


@pytest.mark.parametrize("variant,bn,splits", [(1, 256, 0), (1, 224, 0), (1, 192, 0), (2, 256, 1), (2, 128, 3),
                                               (2, 256, 5), (3, 32, 1), (3, 64, 4), (3, 32, 2), (3, 64, 8),
                                               (3, 32, 3)])
def test_tuned_plans_are_exact(variant, bn, splits):
    # Every plan a tuning table can force computes the same exact result on
    # small integers (M = 24 fits every family, including the transposed one).
    M, N, K = 24, 1000, 1024
    d = inputs.make(M, N, K, kind="f16", dist="smallint", seed=45, beta=1.0)
    try:
        g.tune_set([dict(path=g.GEMM_PATH_TC, M=M, N=N, K=K, variant=variant, bn=bn, splits=splits)])
        got, plan = run_f16(d, 1.0, 1.0)
    finally:
        g.tune_set([])
    assert plan.endswith("+tuned"), plan
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=1.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)


def test_tuned_plan_ignored_when_it_cannot_run():
    M, N, K = 100, 264, 128  # M > 64: the transposed family cannot hold it
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=46)
    try:
        g.tune_set([dict(path=g.GEMM_PATH_TC, M=M, N=N, K=K, variant=3, bn=64, splits=2)])
        got, plan = run_f16(d, 1.0, 0.0)
    finally:
        g.tune_set([])
    assert "+tuned" not in plan
    ref, S = oracle.gemm(d["A"], d["B"], None)
    assert_within(got, ref, S, TOL_F16, plan)


def test_autotune_writes_a_usable_table(tmp_path):
    from dense_gemm_11_gb300 import autotune
    out = tmp_path / "table.json"
    doc = autotune.main(["--shape", "tc:48x2048x1024", "--shape", "f32:192x320x256", "--min-gain", "-1",
                         "--out", str(out)])
    assert len(doc["entries"]) == 2 and len(doc["reports"]) == 2
    try:
        assert g.load_tuning(str(out)) == 2
        d = inputs.make(48, 2048, 1024, kind="f16", dist="smallint", seed=47)
        got, plan = run_f16(d, 1.0, 0.0)
        assert plan.endswith("+tuned")
        ref, _ = oracle.gemm(d["A"], d["B"], None, with_scale=False)
        np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)
    finally:
        g.tune_set([])


@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (1, 4096, 2048), (64, 1000, 3000), (33, 136, 8192)])
def test_f16_cluster_split_k(M, N, K):
    # Small M with few tiles: K is split over the CTAs of a cluster and the
    # partials are added through distributed shared memory.
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=M + N + K, beta=0.5, bias=True)
    got, plan = run_f16(d, 1.25, 0.5, d["bias"], 1)
    assert "clusterk" in plan, plan
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.25, beta=0.5, bias=d["bias"], act=1)
    assert_within(got, ref, S, TOL_F16, f"{M}x{N}x{K} [{plan}]", bias=d["bias"])


@pytest.mark.parametrize("M,N,K,act", [(2048, 4096, 256, 1), (1000, 4000, 512, 3), (4100, 4104, 64, 0), (513, 4104, 128, 2)])
def test_f16_short_k_pair_eight_epilogue_warps(M, N, K, act):
    d = inputs.make(M, N, K, kind="f16", dist="normal_k", seed=M + K, beta=-0.5, bias=True)
    got, plan = run_f16(d, 0.75, -0.5, d["bias"], act)
    assert "pair" in plan and plan.endswith("epi8"), plan
    rows = sample_rows(M, seed=49)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=0.75, beta=-0.5, bias=d["bias"], act=act, rows=rows)
    assert_within(got[rows], ref, S, TOL_F16, f"{M}x{N}x{K} [{plan}]", bias=d["bias"])


def test_f16_short_k_pair_exact():
    d = inputs.make(1024, 2048, 512, kind="f16", dist="smallint", seed=50, beta=1.0)
    got, plan = run_f16(d, 1.0, 1.0)
    assert plan.endswith("epi8"), plan
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=1.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)
