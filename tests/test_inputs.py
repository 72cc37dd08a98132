"""The seeded input generators (no GPU): reproducibility and the bfloat16
rounding that the BF16 workloads use."""
import numpy as np
import pytest

from dense_gemm_11_gb300 import inputs


def test_same_seed_same_arrays():
    a = inputs.make(7, 9, 5, kind="f16", dist="normal_k", seed=3, beta=1.0, bias=True)
    b = inputs.make(7, 9, 5, kind="f16", dist="normal_k", seed=3, beta=1.0, bias=True)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_bf16_rounding_special_cases():
    # Spacing of bfloat16 in [1, 2) is 2**-7.  Halfway cases go to the even
    # neighbour, anything past halfway rounds up, and values already on the
    # grid are unchanged.
    ulp = 2.0 ** -7
    x = np.array([1.0, 1.0 + ulp / 2, 1.0 + 3 * ulp / 2, 1.0 + ulp / 2 + 2.0 ** -20,
                  -(1.0 + ulp / 2), 3.0, -4.0, 0.0, 2.0 ** -130, 65504.0])
    want = np.array([1.0, 1.0, 1.0 + 2 * ulp, 1.0 + ulp, -1.0, 3.0, -4.0, 0.0, 2.0 ** -130, 65536.0])
    got = inputs.round_to_bf16(x)
    assert got.dtype == np.float32
    np.testing.assert_array_equal(got.astype(np.float64), want)


def test_bf16_rounding_agrees_with_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = rng.normal(size=20000) * np.exp(rng.uniform(-30, 30, 20000))
    got = inputs.round_to_bf16(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(got, ref)
    assert (got.view(np.uint32) & 0xFFFF).max() == 0


def test_bf16_workloads_hold_bf16_values():
    d = inputs.make(16, 24, 40, kind="bf16", dist="normal_k", seed=1, beta=0.5, bias=True)
    for k in ("A", "B"):
        assert d[k].dtype == np.float32
        assert (d[k].view(np.uint32) & 0xFFFF).max() == 0
    d = inputs.make(8, 8, 8, kind="bf16", dist="smallint", seed=2)
    assert set(np.unique(d["A"])).issubset(set(range(-4, 5)))
