"""Shared helpers for the parity tests: row sampling and the tolerance check."""
import numpy as np

# Tolerances of the acceptance rule |C - C_ref| <= tol * S + 1e-6, S the
# per-element error scale |alpha| sum_k |a_ik||b_kj| + |beta||c_ij|.
TOL_F32 = 1e-5
TOL_F16 = 2e-3
ABS_FLOOR = 1e-6
# The bias is not part of S.  Adding it to the FP32 pre-activation is one
# rounding (at most half an FP32 ulp of |v|, |v| <= S + |bias_j|); the
# activation after it has slope at most 1.13 (GELU) and its FP32 evaluation
# errs by a few ulps of its argument.  Together that is under four FP32 ulps
# (2^-21) of |bias_j| on top of the tol * S part.
BIAS_ALLOWANCE = 2.0 ** -21
# Unit roundoff of a 16-bit result: rounding the FP32 epilogue value v once to
# the output format adds at most u * |v| <= u * (|ref| + tol * S).
UNIT_ROUNDOFF = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def sample_rows(M, seed=0, n_random=24, tile=128):
    """Rows on both sides of every 4th tile boundary, the first/last rows and random rows."""
    rows = {0, 1, M - 1, M - 2}
    for b in range(0, M, tile * 4):
        rows.update({b - 1, b, b + 1, b + tile - 1, b + tile})
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, M, size=n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < M), dtype=np.int64)


def assert_within(got, ref, S, tol, what="", out="f32", bias=None):
    """|got - ref| <= tol * S + 1e-6 (+ BIAS_ALLOWANCE |bias_j| when a bias
    vector was added), widened by one output rounding for a 16-bit result
    (out = "f16" or "bf16")."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = tol * S + ABS_FLOOR
    if bias is not None:
        bound = bound + BIAS_ALLOWANCE * np.abs(np.asarray(bias, dtype=np.float64))[: got.shape[-1]]
    if out != "f32":
        bound = bound + UNIT_ROUNDOFF[out] * (np.abs(ref) + tol * S)
    bad = ~(err <= bound)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; first {idx}; "
            f"max |err| {np.nanmax(err):.3e}, max |err|/S {np.nanmax(err / np.maximum(S, 1e-30)):.3e}")
    return float(np.max(err / np.maximum(S, 1e-30))) if err.size else 0.0
