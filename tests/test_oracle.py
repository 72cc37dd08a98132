"""Pins for the CPU oracle: closed forms, exact brute force and textbook values.

None of these re-types the oracle's formula in floating point.  The reference
values come from exact rational arithmetic (fractions.Fraction), exact integer
arithmetic, closed forms of special matrices (identity, permutation, rank-1,
zero), and the tabulated standard normal CDF for GELU(x) = x * Phi(x).

Each case is chosen so that a plausible slip in the oracle fails at least one
of them: a transposed operand (non-square brute force), a wrong leading
dimension (views with ld > width), a dropped beta*C or bias term (identity,
beta-only, brute force with bias), bias indexed by row (M != N with bias), a
tanh-approximate GELU (Phi(1) to 1e-15), a missing |beta||C| in the error
scale (exact S check).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _exact(A, B, C0, alpha, beta, bias, K, N):
    """Exact rational evaluation of alpha*A@B + beta*C0 + bias, of the error
    scale S = |alpha| sum|a||b| + |beta||c| (the bias is not part of it) and of
    the magnitude S + |bias| that bounds the double rounding of the value."""
    M = A.shape[0]
    out = [[None] * N for _ in range(M)]
    sc = [[None] * N for _ in range(M)]
    mag = [[None] * N for _ in range(M)]
    fa, fb = Fraction(float(alpha)), Fraction(float(beta))
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            sa = Fraction(0)
            for k in range(K):
                a, b = Fraction(float(A[i, k])), Fraction(float(B[k, j]))
                s += a * b
                sa += abs(a) * abs(b)
            v = fa * s
            e = abs(fa) * sa
            if beta != 0.0:
                c = Fraction(float(C0[i, j]))
                v += fb * c
                e += abs(fb) * abs(c)
            m = e
            if bias is not None:
                v += Fraction(float(bias[j]))
                m += abs(Fraction(float(bias[j])))
            out[i][j] = v
            sc[i][j] = e
            mag[i][j] = m
    return out, sc, mag


TINY = [(1, 1, 1), (1, 5, 3), (3, 1, 7), (2, 3, 5), (7, 5, 3), (5, 7, 2), (8, 8, 8), (3, 11, 13)]


@pytest.mark.parametrize("shape", TINY)
@pytest.mark.parametrize("with_bias", [False, True])
def test_bruteforce_fraction(shape, with_bias):
    M, N, K = shape
    rng = np.random.default_rng(1000 + M * 100 + N * 10 + K)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    bias = rng.normal(0, 0.1, N).astype(np.float32) if with_bias else None
    alpha, beta = 0.7, -1.3
    out, S = oracle.gemm(A, B, C0, alpha=alpha, beta=beta, bias=bias)
    ex, exS, mag = _exact(A, B, C0, alpha, beta, bias, K, N)
    eps = np.finfo(np.float64).eps
    for i in range(M):
        for j in range(N):
            ref = ex[i][j]
            bound = (K + 4) * eps * float(mag[i][j]) + 1e-300
            assert abs(Fraction(out[i, j]) - ref) <= Fraction(bound), (i, j)
            assert abs(S[i, j] - float(exS[i][j])) <= (K + 4) * eps * float(exS[i][j])


def test_bruteforce_with_leading_dims():
    """A (M x lda), B (K x ldb), C (M x ldc) with ld > width: only the window counts."""
    M, N, K = 5, 6, 7
    lda, ldb, ldc = 9, 11, 8
    rng = np.random.default_rng(7)
    A = rng.uniform(-1, 1, (M, lda)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, ldb)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, ldc)).astype(np.float32)
    out, _ = oracle.gemm(A, B, C0, alpha=1.5, beta=0.5, K=K, N=N)
    ex, exS, _ = _exact(A[:, :K], B[:, :N], C0[:, :N], 1.5, 0.5, None, K, N)
    eps = np.finfo(np.float64).eps
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(out[i, j]) - ex[i][j]) <= Fraction((K + 4) * eps * float(exS[i][j]))


def test_identity_left_and_right():
    rng = np.random.default_rng(3)
    n, N = 37, 23
    B = rng.uniform(-1, 1, (n, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (n, N)).astype(np.float32)
    I = np.eye(n, dtype=np.float32)
    out, _ = oracle.gemm(I, B, C0, alpha=2.0, beta=0.5)
    # I @ B = B exactly; 2*B and 0.5*C0 are exact, their sum is one rounding.
    np.testing.assert_array_equal(out, 2.0 * B.astype(np.float64) + 0.5 * C0.astype(np.float64))
    A = rng.uniform(-1, 1, (N, n)).astype(np.float32)
    C1 = rng.uniform(-1, 1, (N, n)).astype(np.float32)
    out2, _ = oracle.gemm(A, I, C1, alpha=1.0, beta=-0.25)
    np.testing.assert_array_equal(out2, A.astype(np.float64) - 0.25 * C1.astype(np.float64))


def test_permutation_rows():
    rng = np.random.default_rng(4)
    n, N = 29, 17
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float32)
    P[np.arange(n), perm] = 1.0
    B = rng.normal(0, 1, (n, N)).astype(np.float32)
    out, _ = oracle.gemm(P, B)
    np.testing.assert_array_equal(out, B[perm].astype(np.float64))


def test_rank1_closed_form():
    """a_ik = u_i, b_kj = v_j  =>  C_ij = alpha*K*u_i*v_j + beta*c_ij (dyadic, exact)."""
    rng = np.random.default_rng(5)
    M, N, K = 19, 13, 64
    u = rng.integers(-8, 9, M) / 8.0
    v = rng.integers(-8, 9, N) / 4.0
    c = rng.integers(-16, 17, (M, N)) / 16.0
    A = np.repeat(u[:, None], K, axis=1).astype(np.float32)
    B = np.repeat(v[None, :], K, axis=0).astype(np.float32)
    out, _ = oracle.gemm(A, B, c.astype(np.float32), alpha=0.5, beta=0.25)
    expect = 0.5 * K * np.outer(u, v) + 0.25 * c
    np.testing.assert_array_equal(out, expect)


def test_smallint_exact_against_integer_product():
    rng = np.random.default_rng(6)
    M, N, K = 33, 41, 300
    A = rng.integers(-4, 5, (M, K))
    B = rng.integers(-4, 5, (K, N))
    C0 = rng.integers(-4, 5, (M, N))
    out, _ = oracle.gemm(A.astype(np.float16), B.astype(np.float16), C0.astype(np.float32),
                         alpha=1.0, beta=2.0)
    exact = A.astype(np.int64) @ B.astype(np.int64) + 2 * C0.astype(np.int64)
    np.testing.assert_array_equal(out, exact.astype(np.float64))


def test_beta_only_and_degenerate():
    rng = np.random.default_rng(8)
    M, N, K = 12, 9, 5
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    Z = np.zeros((M, K), dtype=np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    out, _ = oracle.gemm(Z, B, C0, alpha=1.0, beta=0.75)
    np.testing.assert_array_equal(out, 0.75 * C0.astype(np.float64))
    # alpha == 0: A and B are not read (NaN inside them must not show).
    An = np.full((M, K), np.nan, dtype=np.float32)
    Bn = np.full((K, N), np.nan, dtype=np.float32)
    out, S = oracle.gemm(An, Bn, C0, alpha=0.0, beta=-2.0)
    np.testing.assert_array_equal(out, -2.0 * C0.astype(np.float64))
    np.testing.assert_array_equal(S, 2.0 * np.abs(C0.astype(np.float64)))
    # K == 0: the product is empty.
    out, _ = oracle.gemm(np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), C0,
                         alpha=1.0, beta=3.0)
    np.testing.assert_array_equal(out, 3.0 * C0.astype(np.float64))
    # beta == 0: C is not read.
    Cn = np.full((M, N), np.nan, dtype=np.float32)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    out, _ = oracle.gemm(A, B, Cn, alpha=1.0, beta=0.0)
    assert np.isfinite(out).all()


# Standard normal CDF, tabulated values: Phi(1), Phi(-1), Phi(2), Phi(0.5).
PHI = {1.0: 0.8413447460685429, -1.0: 0.15865525393145707, 2.0: 0.9772498680518208,
       0.5: 0.6914624612740131, -3.0: 0.0013498980316300946}


def test_gelu_special_values():
    assert oracle.gelu(0.0) == 0.0
    for x, phi in PHI.items():
        assert abs(oracle.gelu(x) - x * phi) <= 4e-16 * max(1.0, abs(x))
    assert oracle.gelu(12.0) == 12.0
    assert abs(oracle.gelu(-12.0)) < 1e-30
    # act=1 is applied to the complete pre-activation (product + beta*C + bias).
    C0 = np.array([[1.0, -1.0]], dtype=np.float32)
    bias = np.array([1.0, 0.5], dtype=np.float32)
    out, _ = oracle.gemm(np.zeros((1, 3), np.float32), np.zeros((3, 2), np.float32), C0,
                         alpha=1.0, beta=1.0, bias=bias, act=1)
    assert abs(out[0, 0] - 2.0 * PHI[2.0]) < 1e-15
    assert abs(out[0, 1] - (-0.5) * (1.0 - PHI[0.5])) < 1e-15


def test_numpy_blas_crosscheck():
    rng = np.random.default_rng(9)
    M, N, K = 64, 48, 80
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    B = rng.normal(0, 1, (K, N)).astype(np.float32)
    C0 = rng.normal(0, 1, (M, N)).astype(np.float32)
    out, S = oracle.gemm(A, B, C0, alpha=0.7, beta=-0.3)
    ref = 0.7 * (A.astype(np.float64) @ B.astype(np.float64)) - 0.3 * C0.astype(np.float64)
    assert np.all(np.abs(out - ref) <= 1e-13 * S)


def test_row_subset_and_threads_are_consistent():
    rng = np.random.default_rng(10)
    M, N, K = 50, 31, 70
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    B = rng.normal(0, 1, (K, N)).astype(np.float32)
    C0 = rng.normal(0, 1, (M, N)).astype(np.float32)
    full, Sf = oracle.gemm(A, B, C0, alpha=1.0, beta=0.5, threads=1)
    many, Sm = oracle.gemm(A, B, C0, alpha=1.0, beta=0.5, threads=7)
    np.testing.assert_array_equal(full, many)
    np.testing.assert_array_equal(Sf, Sm)
    rows = [49, 0, 17, 17, 3]
    sub, Ss = oracle.gemm(A, B, C0, alpha=1.0, beta=0.5, rows=rows, threads=3)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(Ss, Sf[rows])


def test_rejects_bad_arguments():
    A = np.zeros((2, 3), np.float32)
    B = np.zeros((3, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.gemm(A, B, None, beta=1.0)
    with pytest.raises(ValueError):
        oracle.gemm(A, B, rows=[2])
    with pytest.raises(ValueError):
        oracle.gemm(A, B, act=5)


def test_relu_and_tanh_gelu():
    # ReLU
    assert oracle.act(2, 3.5) == 3.5 and oracle.act(2, -2.0) == 0.0 and oracle.act(2, 0.0) == 0.0
    # tanh-GELU: f(x) - f(-x) = x for any odd inner function (tanh is odd)
    for x in (0.1, 0.5, 1.0, 2.0, 3.7):
        assert abs((oracle.act(3, x) - oracle.act(3, -x)) - x) < 1e-15 * max(1.0, x)
    assert oracle.act(3, 0.0) == 0.0
    assert oracle.act(3, 20.0) == 20.0 and abs(oracle.act(3, -20.0)) < 1e-30
    # it approximates the exact GELU to better than 1e-3 everywhere (x * Phi(x))
    for x, phi in PHI.items():
        assert abs(oracle.act(3, x) - x * phi) < 1e-3 * max(1.0, abs(x))
        assert oracle.act(3, x) != oracle.act(1, x)  # and it is not the exact form
    # identity / exact GELU dispatch
    assert oracle.act(0, -1.25) == -1.25
    assert oracle.act(1, 1.0) == oracle.gelu(1.0)
    # act applies after bias inside the GEMM
    out, _ = oracle.gemm(np.zeros((1, 2), np.float32), np.zeros((2, 3), np.float32),
                         bias=np.array([-1.0, 0.0, 2.0], np.float32), act=2)
    np.testing.assert_array_equal(out, [[0.0, 0.0, 2.0]])


def test_tanh_gelu_matches_an_independent_implementation():
    """The tanh form of GELU against PyTorch's own CPU implementation in double
    (a test-only library cross-check; nothing in the product calls it).  Its
    coefficients (sqrt(2/pi) and 0.044715, Hendrycks and Gimpel) decide the
    value at every |x| of order one, so a slip in either fails here."""
    torch = pytest.importorskip("torch")
    xs = [-6.0, -3.0, -1.5, -0.5, 0.25, 1.0, 2.5, 6.0]
    ref = torch.nn.functional.gelu(torch.tensor(xs, dtype=torch.float64), approximate="tanh").tolist()
    for x, r in zip(xs, ref):
        assert abs(oracle.act(3, x) - r) <= 1e-15 * max(1.0, abs(x)), x


def test_tanh_gelu_quartic_series_coefficient():
    """Near 0, 0.5 x (1 + tanh(c (x + a x^3))) = x/2 + (c/2) x^2 + (c a / 2 - c^3 / 6) x^4 + O(x^6)
    (tanh t = t - t^3/3 + ...), with c = sqrt(2/pi) and the cubic coefficient
    a = 0.044715 of Hendrycks and Gimpel: the x^4 term is the only place a
    enters at this order, so it pins a independently of any other evaluation.
    At x = 2^-8 the O(x^6) remainder is 2.3e-6 of that term; a = 0.0447
    instead of 0.044715 moves it by 9e-5."""
    import math
    c = math.sqrt(2.0 / math.pi)
    x = 2.0 ** -8
    quartic = (oracle.act(3, x) - x / 2 - c * x * x / 2) / x ** 4
    want = c * 0.044715 / 2 - c ** 3 / 6
    assert abs(quartic / want - 1.0) < 2e-5


def test_round_to_f16_matches_numpy_binary16():
    # numpy converts float64 to IEEE binary16 directly with round-to-nearest-
    # even, including subnormals and overflow: an independent implementation.
    rng = np.random.default_rng(11)
    x = rng.uniform(1.0, 2.0, 40000) * np.exp2(rng.integers(-28, 18, 40000)) * rng.choice([-1.0, 1.0], 40000)
    # exact ties and just-past-tie values at several binades
    ties = np.array([(1 + (2 * k + 1) * 2.0 ** -11) * 2.0 ** e for k in range(8) for e in (-20, -14, -3, 0, 9, 15)])
    x = np.concatenate([x, ties, -ties, ties + np.spacing(ties), [65504.0, 65519.0, 65520.0, 1e6, 2.0 ** -25,
                                                                 3 * 2.0 ** -26, 2.0 ** -24, 0.0, -0.0]])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    got = oracle.round_to("f16", x)
    np.testing.assert_array_equal(got, ref)
    assert np.signbit(got[-1])


def test_round_to_f32_matches_numpy_binary32():
    rng = np.random.default_rng(12)
    x = rng.normal(size=40000) * np.exp2(rng.integers(-140, 128, 40000).astype(np.float64))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(oracle.round_to("f32", x), ref)


def test_round_to_bf16_special_cases():
    u = 2.0 ** -7  # spacing of bfloat16 in [1, 2)
    cases = {
        1.0: 1.0,
        1.0 + u / 2: 1.0,                      # tie -> even (1.0)
        1.0 + 3 * u / 2: 1.0 + 2 * u,          # tie -> even (1 + 2u)
        1.0 + u / 2 + 2.0 ** -40: 1.0 + u,     # just past the tie: up (rounding through
                                               # binary32 first would give 1.0)
        -(1.0 + u / 2 + 2.0 ** -40): -(1.0 + u),
        3.0 * 2.0 ** 100: 3.0 * 2.0 ** 100,
        2.0 ** -133: 2.0 ** -133,              # smallest subnormal
        2.0 ** -134: 0.0,                      # half of it: tie -> even (0)
        1.5 * 2.0 ** -134: 2.0 ** -133,
        (2.0 - 2.0 ** -7) * 2.0 ** 127: (2.0 - 2.0 ** -7) * 2.0 ** 127,  # largest finite
        (2.0 - 2.0 ** -8) * 2.0 ** 127: np.inf,                          # its tie: to inf
    }
    x = np.array(list(cases.keys()))
    np.testing.assert_array_equal(oracle.round_to("bf16", x), np.array(list(cases.values())))


def test_round_to_bf16_matches_bit_rounding_of_binary32_values():
    # For values that are already binary32 numbers the result must equal the
    # round-to-nearest-even of the float32 bit pattern's top 16 bits.
    from dense_gemm_11_gb300 import inputs
    rng = np.random.default_rng(13)
    x = (rng.normal(size=40000) * np.exp2(rng.integers(-120, 120, 40000))).astype(np.float32)
    np.testing.assert_array_equal(oracle.round_to("bf16", x.astype(np.float64)),
                                  inputs.round_to_bf16(x).astype(np.float64))
