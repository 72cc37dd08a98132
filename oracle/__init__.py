"""CPU oracle for the dense GEMM library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding in ``dense_gemm_11_gb300``) never imports, loads or calls
it, and the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (plain C, double accumulation, k
ascending) and follows the GEMM definition C = alpha*A*B + beta*C of
"SGEMM优化，从naive到warptiling" (section 项目概况 / 问题与估算), with the
bias/scale/GELU epilogue of the DeepGEMM essay "企业官网建设流程全解析"
(sections 1.3 and 3.2), and the rounding of a 16-bit output.  This module
only compiles that file and marshals numpy arrays into it.

Every oracle function is pinned by ``tests/test_oracle.py`` against closed
forms, exact brute force and textbook values (none is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgemm_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into a shared library (gcc, -O2, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_gemm_f64.restype = ctypes.c_int
            lib.oracle_gemm_f64.argtypes = [
                ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_long, ctypes.c_void_p, ctypes.c_long,
                ctypes.c_double, ctypes.c_void_p, ctypes.c_long,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_long,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_gelu_f64.restype = ctypes.c_double
            lib.oracle_gelu_f64.argtypes = [ctypes.c_double]
            lib.oracle_round_f64.restype = ctypes.c_int
            lib.oracle_round_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long]
            lib.oracle_act_f64.restype = ctypes.c_double
            lib.oracle_act_f64.argtypes = [ctypes.c_int, ctypes.c_double]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _as_f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x), dtype=np.float64)


def gemm(A, B, C0=None, *, alpha=1.0, beta=0.0, bias=None, act=0, rows=None,
         K=None, N=None, threads=None, with_scale=True):
    """Evaluate out = act(alpha*A[:, :K] @ B[:K, :N] + beta*C0[:, :N] + bias).

    ``A`` is an (M, lda) array (lda >= K), ``B`` (K, ldb) with ldb >= N and
    ``C0`` (M, ldc) with ldc >= N; any dtype whose values are exact in double
    (float32, float16, small integers).  ``rows`` selects output rows (default:
    all).  Returns ``(out, scale)``, both float64 of shape (len(rows), N);
    ``scale`` is the per-element error scale S (None if ``with_scale`` is
    False).
    """
    lib = _load()
    A64 = _as_f64(A)
    B64 = _as_f64(B)
    M = A64.shape[0]
    K = A64.shape[1] if K is None else int(K)
    N = B64.shape[1] if N is None else int(N)
    if B64.shape[0] < K:
        raise ValueError("B has fewer than K rows")
    C64 = _as_f64(C0) if (C0 is not None and beta != 0.0) else None
    if beta != 0.0 and C64 is None:
        raise ValueError("beta != 0 needs C0")
    b64 = _as_f64(bias)
    if b64 is not None and b64.shape[0] < N:
        raise ValueError("bias shorter than N")
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    out = np.empty((nrows, N), dtype=np.float64)
    scale = np.empty((nrows, N), dtype=np.float64) if with_scale else None
    nthreads = default_threads() if threads is None else int(threads)

    def ptr(a):
        return None if a is None else a.ctypes.data

    rc = lib.oracle_gemm_f64(
        M, N, K, float(alpha),
        ptr(A64), A64.shape[1] if A64.ndim == 2 else 0,
        ptr(B64), B64.shape[1] if B64.ndim == 2 else 0,
        float(beta), ptr(C64), C64.shape[1] if C64 is not None else 0,
        ptr(b64), int(act), ptr(rows_arr), nrows, ptr(out), ptr(scale), nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm_f64 rejected its arguments")
    return out, scale


OUT_TYPES = {"f32": 0, "f16": 1, "bf16": 2}


def round_to(out_type: str, x):
    """Round each value of x once, to nearest (ties to even), to the output
    type "f32", "f16" or "bf16"; overflow gives +-inf.  Returns float64."""
    x64 = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(x64)
    rc = _load().oracle_round_f64(OUT_TYPES[out_type], x64.ctypes.data, out.ctypes.data, x64.size)
    if rc != 0:
        raise ValueError("oracle_round_f64 rejected its arguments")
    return out


def gelu(x: float) -> float:
    """Exact-erf GELU in double (the oracle's activation)."""
    return float(_load().oracle_gelu_f64(float(x)))


def act(kind: int, x: float) -> float:
    """Activation `kind` (0 identity, 1 exact GELU, 2 ReLU, 3 tanh GELU) in double."""
    return float(_load().oracle_act_f64(int(kind), float(x)))
