"""FP32 SGEMM parity: the CUDA path against the CPU oracle on the same seeded
inputs, elementwise within |C - C_ref| <= 1e-5 * S + 1e-6 (exact for small
integers).  Called through the C ABI (ctypes binding)."""
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


def run_f32(d, alpha, beta, K=None, N=None, M=None, offset=0):
    """Copy the arrays to the GPU (optionally at an element offset) and run gemm_f32 on views."""
    A, B, C = d["A"], d["B"], d["C"]
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[1] if N is None else N

    def dev(x):
        flat = torch.empty(x.size + offset + 8, dtype=torch.float32, device=DEV)
        flat[offset:offset + x.size] = torch.from_numpy(np.ascontiguousarray(x)).reshape(-1).to(DEV)
        return flat, flat[offset:offset + x.size].view(x.shape)

    _, Ad = dev(A)
    _, Bd = dev(B)
    Cflat, Cd = dev(C)
    g.gemm_f32(Ad[:, :K], Bd[:K, :N], Cd[:, :N], alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    return Cd.cpu().numpy(), g.last_plan()


def check_workload(name, rows=None):
    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(w)
    got, plan = run_f32(d, w.alpha, w.beta)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=w.alpha, beta=w.beta, rows=rows)
    sel = got if rows is None else got[rows]
    return assert_within(sel, ref, S, TOL_F32, f"{name} [{plan}]"), plan


def test_f32_512_full():
    check_workload("f32_512")


@pytest.mark.parametrize("s", [128, 256, 512, 1024, 2048])
def test_f32_square_sweep_full(s):
    check_workload(f"f32_sq{s}")


def test_f32_square_4096_sampled():
    check_workload("f32_sq4096", rows=sample_rows(4096, seed=1))


@pytest.mark.parametrize("i", [0, 2, 3])
def test_f32_irregular_full(i):
    check_workload(f"f32_irr{i}")


def test_f32_irregular_4095_4097_4099_sampled():
    _, plan = check_workload("f32_irr1", rows=sample_rows(4095, seed=2))
    # lda = 4099: rows are not 16-byte aligned; large problems are repacked
    assert "repack" in plan or "vec4b" in plan


SHAPES = [1, 3, 17, 32, 64, 128, 129]


@pytest.mark.parametrize("M", SHAPES)
@pytest.mark.parametrize("N", [1, 17, 129])
@pytest.mark.parametrize("K", [1, 32, 129])
def test_f32_small_shape_grid(M, N, K):
    d = inputs.make(M, N, K, kind="f32", dist="uniform", seed=M * 10007 + N * 101 + K, beta=0.75)
    got, plan = run_f32(d, -1.25, 0.75)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=-1.25, beta=0.75)
    assert_within(got, ref, S, TOL_F32, f"{M}x{N}x{K} [{plan}]")


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (3, 1024, 1024), (1024, 3, 17)])
def test_f32_p3_shape_list_large(M, N, K):
    d = inputs.make(M, N, K, kind="f32", dist="normal", seed=5, beta=0.0)
    got, plan = run_f32(d, 1.0, 0.0)
    ref, S = oracle.gemm(d["A"], d["B"], None, alpha=1.0, beta=0.0)
    assert_within(got, ref, S, TOL_F32, f"{M}x{N}x{K} [{plan}]")


@pytest.mark.parametrize("lds", [(300, 260, 270), (301, 263, 259), (1040, 1032, 1036)])
def test_f32_leading_dims_larger_than_width(lds):
    M, N, K = 250, 257, 299
    lda, ldb, ldc = lds
    if lda < K:
        lda = K + (lda % 7) + 1
    d = inputs.make(M, N, K, kind="f32", dist="uniform", seed=11, beta=0.5, lda=lda, ldb=ldb, ldc=ldc)
    got, plan = run_f32(d, 1.0, 0.5, K=K, N=N)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=0.5, K=K, N=N)
    assert_within(got[:, :N], ref, S, TOL_F32, f"ld {lds} [{plan}]")
    # columns past N in C are untouched
    np.testing.assert_array_equal(got[:, N:], d["C"][:, N:])


@pytest.mark.parametrize("M,N,K,lda,ldb", [(1300, 1500, 1100, 1101, 1500), (1024, 2050, 1031, 1031, 2053)])
def test_f32_repacked_unaligned_large(M, N, K, lda, ldb):
    d = inputs.make(M, N, K, kind="f32", dist="normal", seed=23, beta=0.25, lda=lda, ldb=ldb)
    got, plan = run_f32(d, 1.0, 0.25, K=K, N=N)
    assert "repack" in plan
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=0.25, K=K, N=N, rows=sample_rows(M, seed=3))
    assert_within(got[sample_rows(M, seed=3)], ref, S, TOL_F32, f"repacked [{plan}]")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_f32_unaligned_base_pointers(offset):
    M, N, K = 300, 260, 200
    d = inputs.make(M, N, K, kind="f32", dist="uniform", seed=12, beta=1.5)
    got, plan = run_f32(d, 0.5, 1.5, offset=offset)
    assert "vec4b" in plan or "sgemv" in plan
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=0.5, beta=1.5)
    assert_within(got, ref, S, TOL_F32, f"offset {offset} [{plan}]")


def test_f32_beta_zero_does_not_read_c():
    d = inputs.make(513, 515, 257, kind="f32", dist="normal", seed=13, beta=0.0)
    assert np.isnan(d["C"]).all()
    got, plan = run_f32(d, 0.7, 0.0)
    assert np.isfinite(got).all(), plan


@pytest.mark.parametrize("M,N,K", [(200, 300, 400), (1, 4096, 4096), (4096, 1, 4096), (64, 64, 8192)])
def test_f32_small_integers_exact(M, N, K):
    d = inputs.make(M, N, K, kind="f32", dist="smallint", seed=14, beta=2.0)
    got, plan = run_f32(d, 1.0, 2.0)
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)


def test_f32_alpha_zero_and_k_zero():
    rng = np.random.default_rng(15)
    C0 = rng.uniform(-1, 1, (77, 65)).astype(np.float32)
    Cd = torch.from_numpy(C0).to(DEV)
    An = torch.full((77, 33), float("nan"), device=DEV)
    Bn = torch.full((33, 65), float("nan"), device=DEV)
    g.gemm_f32(An, Bn, Cd, alpha=0.0, beta=-2.0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Cd.cpu().numpy(), (-2.0 * C0.astype(np.float64)).astype(np.float32))
    g.gemm_f32(torch.empty(77, 0, device=DEV), torch.empty(0, 65, device=DEV), Cd, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert (Cd == 0).all()


def test_f32_guard_band_untouched():
    M, N, K = 129, 131, 67
    d = inputs.make(M, N, K, kind="f32", dist="uniform", seed=16, beta=1.0)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), 12345.0, device=DEV)
    Cd = buf[pad:pad + M * N].view(M, N)
    Cd.copy_(torch.from_numpy(d["C"]).to(DEV))
    A = torch.from_numpy(d["A"]).to(DEV)
    B = torch.from_numpy(d["B"]).to(DEV)
    g.gemm_f32(A, B, Cd, alpha=1.0, beta=1.0)
    torch.cuda.synchronize()
    assert (buf[:pad] == 12345.0).all() and (buf[pad + M * N:] == 12345.0).all()


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (1, 4096, 4096), (256, 384, 2048)])
def test_f32_deterministic(M, N, K):
    d = inputs.make(M, N, K, kind="f32", dist="normal", seed=17, beta=0.0)
    a, plan = run_f32(d, 1.0, 0.0)
    b, _ = run_f32(d, 1.0, 0.0)
    np.testing.assert_array_equal(a, b, err_msg=plan)


def test_f32_two_streams():
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    d1 = inputs.make(640, 700, 512, kind="f32", dist="normal", seed=18, beta=0.0)
    d2 = inputs.make(300, 900, 1024, kind="f32", dist="normal", seed=19, beta=0.0)
    t1 = [torch.from_numpy(d1[k]).to(DEV) for k in ("A", "B", "C")]
    t2 = [torch.from_numpy(d2[k]).to(DEV) for k in ("A", "B", "C")]
    torch.cuda.synchronize()
    for _ in range(3):
        g.gemm_f32(*t1, alpha=1.0, beta=0.0, stream=s1)
        g.gemm_f32(*t2, alpha=1.0, beta=0.0, stream=s2)
    torch.cuda.synchronize()
    for d, t in ((d1, t1), (d2, t2)):
        ref, S = oracle.gemm(d["A"], d["B"], None, alpha=1.0, beta=0.0)
        assert_within(t[2].cpu().numpy(), ref, S, TOL_F32, "two streams")


@pytest.mark.parametrize("variant,splits", [(1, 0), (2, 1), (2, 4), (2, 16)])
def test_tuned_f32_plans_are_exact(variant, splits):
    M, N, K = 300, 520, 1000
    d = inputs.make(M, N, K, kind="f32", dist="smallint", seed=48, beta=1.0)
    A, B, C = (torch.from_numpy(d[k]).to(DEV) for k in ("A", "B", "C"))
    try:
        g.tune_set([dict(path=g.GEMM_PATH_F32, M=M, N=N, K=K, variant=variant, bn=0, splits=splits)])
        g.gemm_f32(A, B, C, alpha=1.0, beta=1.0)
        torch.cuda.synchronize()
        plan = g.last_plan()
    finally:
        g.tune_set([])
    assert plan.endswith("+tuned"), plan
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=1.0, with_scale=False)
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref, err_msg=plan)


@pytest.mark.parametrize("M,N,K,strip", [(2048, 2049, 1024, 1), (2048, 2088, 512, 40), (1800, 2305, 700, 1)])
def test_f32_column_edge_strip_exact(M, N, K, strip):
    # Big tiles cover the first N - r columns and the r-column edge strip runs
    # on its own (a matrix-vector product for r = 1); C's padding (ldc > N)
    # stays untouched.  Small integers: exact whatever the summation order.
    ldc = N + 5
    d = inputs.make(M, N, K, kind="f32", dist="smallint", seed=N + K, beta=1.0, ldc=ldc)
    got, plan = run_f32(d, 1.0, 1.0, N=N)
    assert plan.endswith("+colstrip1" if strip == 1 else "+colstrip"), plan
    N0 = N - strip
    rows = sample_rows(M, seed=5)
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=1.0, N=N, rows=rows, with_scale=False)
    np.testing.assert_array_equal(got[rows, :N].astype(np.float64), ref, err_msg=plan)
    # every row of the strip
    ref_s, _ = oracle.gemm(d["A"], np.ascontiguousarray(d["B"][:, N0:N]), np.ascontiguousarray(d["C"][:, N0:N]),
                           alpha=1.0, beta=1.0, with_scale=False)
    np.testing.assert_array_equal(got[:, N0:N].astype(np.float64), ref_s, err_msg=plan)
    np.testing.assert_array_equal(got[:, N:], d["C"][:, N:])


@pytest.mark.parametrize("M,N,K", [(300, 200, 500), (33, 129, 257), (100, 64, 2048), (512, 512, 512), (256, 256, 256)])
@pytest.mark.parametrize("offset", [0, 1])
def test_f32_k_group_plan(M, N, K, offset):
    # Few tiles, short K: 32x64 tiles whose K is split among four warp groups
    # of the CTA (ragged K leaves some groups a zero-filled last slice);
    # offset 1 puts every row off 16-byte alignment (the 4-byte copy path).
    d = inputs.make(M, N, K, kind="f32", dist="normal", seed=M + N + K, beta=0.75)
    got, plan = run_f32(d, -1.25, 0.75, offset=offset)
    assert "kg4" in plan, plan
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=-1.25, beta=0.75)
    assert_within(got, ref, S, TOL_F32, f"{M}x{N}x{K} [{plan}]")


@pytest.mark.parametrize("M,N,K", [(300, 200, 500), (64, 640, 1024)])
def test_f32_k_group_plan_small_integers_exact(M, N, K):
    d = inputs.make(M, N, K, kind="f32", dist="smallint", seed=7, beta=2.0)
    got, plan = run_f32(d, 1.0, 2.0)
    assert "kg4" in plan, plan
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=plan)


# M == 1 (a row vector times B): ragged N and K, a leading dimension past N,
# beta != 0; every column against the oracle.
@pytest.mark.parametrize("N,K,ldb", [(4000, 3001, None), (6000, 2048, 6004), (11008, 4096, None),
                                     (12345, 1500, 12352), (2000, 4096, None), (20000, 1024, None)])
def test_f32_m1_shapes(N, K, ldb):
    d = inputs.make(1, N, K, kind="f32", dist="uniform", seed=60, beta=0.5, ldb=ldb)
    got, p = run_f32(d, 0.7, 0.5, K=K, N=N)
    ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=0.7, beta=0.5, K=K, N=N)
    assert_within(got[:, :N], ref, S, TOL_F32, f"1 x {N} x {K} [{p}]")


@pytest.mark.parametrize("N,K", [(6000, 2048), (11008, 4099)])
def test_f32_m1_exact_and_beta_zero(N, K):
    d = inputs.make(1, N, K, kind="f32", dist="smallint", seed=61, beta=2.0)
    got, p = run_f32(d, 1.0, 2.0)
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=2.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=p)
    # beta == 0 never reads C (NaN there stays out of the result)
    d0 = inputs.make(1, N, K, kind="f32", dist="normal", seed=62, beta=0.0)
    assert np.isnan(d0["C"]).all()
    got0, p0 = run_f32(d0, 0.5, 0.0)
    assert np.isfinite(got0).all(), p0


@pytest.mark.parametrize("N,K,plan", [(4096, 4096, "sgemv_cols_clusterk"), (11008, 4096, "sgemv_cols_clusterk"),
                                      (3000, 4097, "sgemv_cols_clusterk"), (2000, 4096, "sgemv_cols_splitk"),
                                      (4096, 100, "sgemv_cols")])
def test_f32_m1_plans_exact(N, K, plan):
    # K split over a cluster (up to 8 CTAs, sums through distributed shared
    # memory) while every SM still gets a CTA; otherwise the global split-K
    # kernel, or no split for short K
    d = inputs.make(1, N, K, kind="f32", dist="smallint", seed=63, beta=-1.0)
    got, p = run_f32(d, 1.0, -1.0)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert p == plan, p
    ref, _ = oracle.gemm(d["A"], d["B"], d["C"], alpha=1.0, beta=-1.0, with_scale=False)
    np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=p)
