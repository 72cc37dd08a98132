"""The GEMM11_DEBUG build (libgemm11_debug.so) on the GPU.

The debug build keeps one operand stage in flight, checks the index of every
store to C and of every access to library scratch on the device, guards the
scratch with filled bands, and synchronises at the end of every call.  Which
library a process uses is fixed when it first loads one (environment variable
GEMM11_DEBUG), so each check runs in a child process:

  * a parity subset of the other GPU tests passes against the oracle with the
    debug library (the synchronous pipelines compute the same results);
  * a test-only shrink of the C extent the FP32 path checks against
    (GEMM11_DEBUG_SHRINK_C) makes the device-side check fire: the call
    returns GEMM_ERR_DEBUG_CHECK, the stores past the extent are skipped and
    the rest of C is right.  The real buffer is larger than the shrunk extent,
    so no access leaves it either way;
  * a test-only overwrite of one guard-band word (GEMM11_DEBUG_POKE_CANARY;
    memory the library allocated) is caught by the band check after the call.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(args, extra_env, timeout=900):
    env = dict(os.environ)
    env.update({"GEMM11_DEBUG": "1", **extra_env})
    r = subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    return r.returncode, r.stdout + r.stderr


def test_parity_subset_with_the_debug_library():
    rc, out = _child(["-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                      "tests/test_gpu_f32.py", "tests/test_gpu_f16.py", "tests/test_gpu_batched.py",
                      "tests/test_gpu_clusterk.py",
                      "-k", "small_shape_grid or k_group or leading_dims or unaligned or small_integers or tuned "
                            "or ragged or beta or cluster or batched_parity or p3_shape or column_edge"], {})
    assert rc == 0, out[-3000:]
    assert " passed" in out


SHRINK_SCRIPT = r"""
import numpy as np, torch
import dense_gemm_11_gb300 as g
assert g.debug_build()
M = N = K = 64
rng = np.random.default_rng(1)
A = torch.from_numpy(rng.integers(-4, 5, (M, K)).astype(np.float32)).cuda()
B = torch.from_numpy(rng.integers(-4, 5, (K, N)).astype(np.float32)).cuda()
C = torch.full((M, N), 1234.0, device="cuda")
st = g.gemm_f32_raw(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N,
                    torch.cuda.current_stream().cuda_stream)
assert st == g.GEMM_ERR_DEBUG_CHECK, g.status_string(st)
got = C.cpu().numpy().reshape(-1)
ref = (A.cpu().numpy().astype(np.float64) @ B.cpu().numpy().astype(np.float64)).reshape(-1)
assert (got[-8:] == 1234.0).all(), got[-8:]             # past the shrunk extent: not stored
np.testing.assert_array_equal(got[:-8], ref[:-8])      # the rest: exact small-integer products
assert g.check() == g.GEMM_OK                          # the fault was reported once, by the call
print("shrink ok")
"""

POKE_SCRIPT = r"""
import numpy as np, torch
import dense_gemm_11_gb300 as g
assert g.debug_build()
M, N, K = 256, 256, 4096   # few tiles, long K: the FP32 plan splits K through library scratch
A = torch.randn(M, K, device="cuda")
B = torch.randn(K, N, device="cuda")
C = torch.zeros(M, N, device="cuda")
stream = torch.cuda.current_stream().cuda_stream
st = g.gemm_f32_raw(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N, stream)
assert "splitk" in g.last_plan(), g.last_plan()
assert st == g.GEMM_ERR_DEBUG_CHECK, g.status_string(st)
print("poke ok")
"""


def test_device_side_bounds_check_fires_and_skips_the_store():
    rc, out = _child(["-c", SHRINK_SCRIPT], {"GEMM11_DEBUG_SHRINK_C": "8"})
    assert rc == 0 and "shrink ok" in out, out[-3000:]


def test_scratch_guard_band_check_catches_an_overwrite():
    rc, out = _child(["-c", POKE_SCRIPT], {"GEMM11_DEBUG_POKE_CANARY": "1"})
    assert rc == 0 and "poke ok" in out, out[-3000:]


def test_release_library_is_the_default():
    import dense_gemm_11_gb300 as g
    if os.environ.get("GEMM11_DEBUG", "0") != "1":
        assert not g.debug_build()
