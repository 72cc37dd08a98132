"""Python binding of libgemm11.so, the GB300 (sm_103a) dense GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/gemm11.h``.  There is no
fallback: if the shared library is missing, every call raises.

    gemm_f32(A, B, C, alpha=1.0, beta=0.0)            C = alpha*A@B + beta*C (fp32)
    gemm_f32_3xtf32(A, B, C, alpha=1.0, beta=0.0)     the same on the tensor cores (3 TF32 products)
    gemm_f16_f32acc_epilogue(A, B, C, alpha=1.0, beta=0.0, bias=None, act=0)
                                                      C = act(alpha*A@B + beta*C + bias)
    gemm_bf16_f32acc_epilogue(...)                    the same with bf16 A and B
    gemm_tc(A, B, C, ...)                             the same for fp16/bf16 A, B and fp32/fp16/bf16 C
    gemm_tc_batched(A, B, C, ..., b_trans=False)      a strided batch of those (3-D tensors), op(B) = B or B^T

Tensors are torch CUDA tensors on the current device; A and B may be 2-D
views with a leading dimension larger than their width (unit column stride).
Calls are asynchronous on the current torch stream (or ``stream=``).
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import DEBUG_LIB_PATH, LIB_PATH, build  # noqa: F401  (build() is part of the public API)

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_UNSUPPORTED = -2
GEMM_ERR_CUDA = -3
GEMM_ERR_TIMEOUT = -4
GEMM_ERR_SCRATCH_LIMIT = -5
GEMM_ERR_DEBUG_CHECK = -6
GEMM_ACT_NONE = 0
GEMM_ACT_GELU = 1
GEMM_ACT_RELU = 2
GEMM_ACT_GELU_TANH = 3
GEMM_DTYPE_F32 = 0
GEMM_DTYPE_F16 = 1
GEMM_DTYPE_BF16 = 2
GEMM_PATH_F32 = 0
GEMM_PATH_TC = 1


class TuneEntry(ctypes.Structure):
    """One row of the tuning table (gemm_tune_entry in include/gemm11.h)."""
    _fields_ = [("path", ctypes.c_int), ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("variant", ctypes.c_int), ("bn", ctypes.c_int), ("splits", ctypes.c_int)]

    def as_dict(self):
        return {f: int(getattr(self, f)) for f, _ in self._fields_}

EXPORTED_SYMBOLS = ("gemm_f32", "gemm_f32_3xtf32", "gemm_f16_f32acc_epilogue", "gemm_bf16_f32acc_epilogue",
                    "gemm_tc_f32acc_epilogue", "gemm_tc_strided_batched", "gemm_f16_f32acc_epilogue_noalloc",
                    "gemm_tune_set", "gemm_tune_get",
                    "gemm_status_string", "gemm_last_cuda_error", "gemm_check", "gemm_watchdog_selftest",
                    "gemm_last_plan", "gemm_last_launch_count", "gemm_tc_rate_probe",
                    "gemm_pipeline_stall_selftest", "gemm_fma_rate_probe", "gemm_tma_read_probe",
                    "gemm_debug_build")

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        if status == GEMM_ERR_CUDA and _lib is not None:
            msg += f" (cudaError {_lib.gemm_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")


def library_path() -> str:
    """The library this process uses: the debug build (libgemm11_debug.so)
    when the environment variable GEMM11_DEBUG is 1, else libgemm11.so."""
    return DEBUG_LIB_PATH if os.environ.get("GEMM11_DEBUG", "0") == "1" else LIB_PATH


def lib():
    """The loaded library (ctypes): libgemm11.so, or libgemm11_debug.so with
    GEMM11_DEBUG=1.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); call "
                                   "dense_gemm_11_gb300.build()")
            L = ctypes.CDLL(path)
            c_int, c_float, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
            L.gemm_f32.restype = c_int
            L.gemm_f32.argtypes = [c_int, c_int, c_int, c_float, c_void_p, c_int, c_void_p, c_int, c_float,
                                   c_void_p, c_int, c_void_p]
            L.gemm_f32_3xtf32.restype = c_int
            L.gemm_f32_3xtf32.argtypes = L.gemm_f32.argtypes
            L.gemm_f16_f32acc_epilogue.restype = c_int
            L.gemm_f16_f32acc_epilogue.argtypes = [c_int, c_int, c_int, c_float, c_void_p, c_void_p, c_float,
                                                   c_void_p, c_void_p, c_int, c_void_p]
            L.gemm_bf16_f32acc_epilogue.restype = c_int
            L.gemm_bf16_f32acc_epilogue.argtypes = L.gemm_f16_f32acc_epilogue.argtypes
            L.gemm_tc_f32acc_epilogue.restype = c_int
            L.gemm_tc_f32acc_epilogue.argtypes = [c_int, c_int, c_int, c_float, c_void_p, c_void_p, c_int,
                                                  c_float, c_void_p, c_int, c_void_p, c_int, c_void_p]
            c_ll = ctypes.c_longlong
            L.gemm_tc_strided_batched.restype = c_int
            L.gemm_tc_strided_batched.argtypes = [c_int, c_int, c_int, c_int, c_float, c_void_p, c_ll, c_void_p,
                                                  c_ll, c_int, c_int, c_float, c_void_p, c_ll, c_int, c_void_p,
                                                  c_int, c_void_p]
            L.gemm_f16_f32acc_epilogue_noalloc.restype = c_int
            L.gemm_f16_f32acc_epilogue_noalloc.argtypes = L.gemm_f16_f32acc_epilogue.argtypes
            L.gemm_tune_set.restype = c_int
            L.gemm_tune_set.argtypes = [ctypes.POINTER(TuneEntry), c_int]
            L.gemm_tune_get.restype = c_int
            L.gemm_tune_get.argtypes = [ctypes.POINTER(TuneEntry), c_int]
            L.gemm_status_string.restype = ctypes.c_char_p
            L.gemm_status_string.argtypes = [c_int]
            L.gemm_last_cuda_error.restype = c_int
            L.gemm_last_cuda_error.argtypes = []
            L.gemm_check.restype = c_int
            L.gemm_check.argtypes = [c_void_p]
            L.gemm_watchdog_selftest.restype = c_int
            L.gemm_watchdog_selftest.argtypes = [c_int, c_void_p]
            L.gemm_last_plan.restype = ctypes.c_char_p
            L.gemm_last_plan.argtypes = []
            L.gemm_last_launch_count.restype = c_int
            L.gemm_last_launch_count.argtypes = []
            L.gemm_pipeline_stall_selftest.restype = c_int
            L.gemm_pipeline_stall_selftest.argtypes = [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_int,
                                                       c_void_p]
            L.gemm_debug_build.restype = c_int
            L.gemm_debug_build.argtypes = []
            L.gemm_fma_rate_probe.restype = c_int
            L.gemm_fma_rate_probe.argtypes = [c_int, c_int, ctypes.POINTER(ctypes.c_double), c_void_p]
            L.gemm_tc_rate_probe.restype = c_int
            L.gemm_tc_rate_probe.argtypes = [c_int, ctypes.POINTER(ctypes.c_double), c_void_p]
            L.gemm_tma_read_probe.restype = c_int
            L.gemm_tma_read_probe.argtypes = [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(ctypes.c_double),
                                              ctypes.POINTER(ctypes.c_double), c_void_p]
            _lib = L
    return _lib


def debug_build() -> bool:
    """True when the loaded library is the GEMM11_DEBUG build."""
    return bool(lib().gemm_debug_build())


def status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


def last_plan() -> str:
    return lib().gemm_last_plan().decode()


def last_launch_count() -> int:
    return int(lib().gemm_last_launch_count())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _mat(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} needs unit column stride")
    # a single row has no row stride of its own: report the tensor's when it is
    # a valid one (a view keeps its parent's, which may be 16-byte aligned)
    if t.shape[0] > 1 or t.stride(0) >= t.shape[1]:
        return t.data_ptr(), max(t.stride(0), 1)
    return t.data_ptr(), max(t.shape[1], 1)


def gemm_f32_raw(M, N, K, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, stream_ptr=0) -> int:
    """Direct C-ABI call with integer device pointers; returns the status code."""
    return lib().gemm_f32(int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr), int(lda),
                          ctypes.c_void_p(B_ptr), int(ldb), float(beta), ctypes.c_void_p(C_ptr), int(ldc),
                          ctypes.c_void_p(stream_ptr))


def gemm_f16_raw(M, N, K, alpha, A_ptr, B_ptr, beta, C_ptr, bias_ptr=0, act=0, stream_ptr=0) -> int:
    """Direct C-ABI call with integer device pointers; returns the status code."""
    return lib().gemm_f16_f32acc_epilogue(int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr),
                                          ctypes.c_void_p(B_ptr), float(beta), ctypes.c_void_p(C_ptr),
                                          ctypes.c_void_p(bias_ptr or None), int(act), ctypes.c_void_p(stream_ptr))


def gemm_bf16_raw(M, N, K, alpha, A_ptr, B_ptr, beta, C_ptr, bias_ptr=0, act=0, stream_ptr=0) -> int:
    """Direct C-ABI call of the BF16-input entry point; returns the status code."""
    return lib().gemm_bf16_f32acc_epilogue(int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr),
                                           ctypes.c_void_p(B_ptr), float(beta), ctypes.c_void_p(C_ptr),
                                           ctypes.c_void_p(bias_ptr or None), int(act), ctypes.c_void_p(stream_ptr))


def gemm_tc_raw(M, N, K, alpha, A_ptr, B_ptr, ab_type, beta, C_ptr, c_type, bias_ptr=0, act=0,
                stream_ptr=0) -> int:
    """Direct C-ABI call of the general tensor-core entry point; returns the status code."""
    return lib().gemm_tc_f32acc_epilogue(int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr),
                                         ctypes.c_void_p(B_ptr), int(ab_type), float(beta), ctypes.c_void_p(C_ptr),
                                         int(c_type), ctypes.c_void_p(bias_ptr or None), int(act),
                                         ctypes.c_void_p(stream_ptr))


def gemm_tc_batched_raw(batch, M, N, K, alpha, A_ptr, stride_a, B_ptr, stride_b, ab_type, b_trans, beta, C_ptr,
                        stride_c, c_type, bias_ptr=0, act=0, stream_ptr=0) -> int:
    """Direct C-ABI call of the strided-batched entry point; returns the status code."""
    return lib().gemm_tc_strided_batched(int(batch), int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr),
                                         int(stride_a), ctypes.c_void_p(B_ptr), int(stride_b), int(ab_type),
                                         int(b_trans), float(beta), ctypes.c_void_p(C_ptr), int(stride_c),
                                         int(c_type), ctypes.c_void_p(bias_ptr or None), int(act),
                                         ctypes.c_void_p(stream_ptr))


def gemm_f16_noalloc_raw(M, N, K, alpha, A_ptr, B_ptr, beta, C_ptr, bias_ptr=0, act=0, stream_ptr=0) -> int:
    """C-ABI call of the no-allocation variant (M <= 64); returns the status code.

    For callers that cannot let the library allocate device memory: the
    split-K scratch is a fixed array inside the library.  Calls that overlap
    on the GPU share that array and race; issue them on one stream.
    """
    return lib().gemm_f16_f32acc_epilogue_noalloc(int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr),
                                                  ctypes.c_void_p(B_ptr), float(beta), ctypes.c_void_p(C_ptr),
                                                  ctypes.c_void_p(bias_ptr or None), int(act),
                                                  ctypes.c_void_p(stream_ptr))


def gemm_f32_3xtf32_raw(M, N, K, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, stream_ptr=0) -> int:
    """Direct C-ABI call of the 3xTF32 FP32 GEMM; returns the status code."""
    return lib().gemm_f32_3xtf32(int(M), int(N), int(K), float(alpha), ctypes.c_void_p(A_ptr), int(lda),
                                 ctypes.c_void_p(B_ptr), int(ldb), float(beta), ctypes.c_void_p(C_ptr), int(ldc),
                                 ctypes.c_void_p(stream_ptr))


def gemm_f32_3xtf32(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, stream=None) -> None:
    """C = alpha * A @ B + beta * C, FP32 operands, on the tensor cores (3 TF32 products)."""
    _gemm_f32_like("gemm_f32_3xtf32", A, B, C, alpha, beta, stream)


def gemm_f32(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, stream=None) -> None:
    """C = alpha * A @ B + beta * C in true FP32 (CUDA-core FFMA)."""
    _gemm_f32_like("gemm_f32", A, B, C, alpha, beta, stream)


def _gemm_f32_like(fn_name, A, B, C, alpha, beta, stream) -> None:
    import torch
    a_ptr, lda = _mat(A, "A", torch.float32)
    b_ptr, ldb = _mat(B, "B", torch.float32)
    c_ptr, ldc = _mat(C, "C", torch.float32)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} B{tuple(B.shape)} C{tuple(C.shape)}")
    st = getattr(lib(), fn_name)(M, N, K, float(alpha), ctypes.c_void_p(a_ptr), lda, ctypes.c_void_p(b_ptr), ldb,
                                 float(beta), ctypes.c_void_p(c_ptr), ldc, _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, fn_name)


def _gemm_16bit(fn_name, in_dtype, A, B, C, alpha, beta, bias, act, stream) -> None:
    import torch
    for name, t, dt in (("A", A, in_dtype), ("B", B, in_dtype), ("C", C, torch.float32)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dt or t.dim() != 2:
            raise TypeError(f"{name} must be a 2-D CUDA {dt} tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (leading dimension = width)")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} B{tuple(B.shape)} C{tuple(C.shape)}")
    bias_ptr = None
    if bias is not None:
        if not bias.is_cuda or bias.dtype != torch.float32 or bias.numel() != N or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous CUDA float32 tensor of length N")
        bias_ptr = bias.data_ptr()
    st = getattr(lib(), fn_name)(M, N, K, float(alpha), ctypes.c_void_p(A.data_ptr()),
                                 ctypes.c_void_p(B.data_ptr()), float(beta), ctypes.c_void_p(C.data_ptr()),
                                 ctypes.c_void_p(bias_ptr), int(act), _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, fn_name)


def gemm_f16_f32acc_epilogue(A, B, C, alpha: float = 1.0, beta: float = 0.0, bias=None, act: int = 0, *,
                             stream=None) -> None:
    """C = act(alpha * A @ B + beta * C + bias): fp16 A, B; fp32 accumulate, bias and C."""
    import torch
    _gemm_16bit("gemm_f16_f32acc_epilogue", torch.float16, A, B, C, alpha, beta, bias, act, stream)


def gemm_bf16_f32acc_epilogue(A, B, C, alpha: float = 1.0, beta: float = 0.0, bias=None, act: int = 0, *,
                              stream=None) -> None:
    """C = act(alpha * A @ B + beta * C + bias): bf16 A, B; fp32 accumulate, bias and C."""
    import torch
    _gemm_16bit("gemm_bf16_f32acc_epilogue", torch.bfloat16, A, B, C, alpha, beta, bias, act, stream)


def gemm_tc(A, B, C, alpha: float = 1.0, beta: float = 0.0, bias=None, act: int = 0, *, stream=None) -> None:
    """C = act(alpha * A @ B + beta * C + bias) on the tensor cores, FP32 accumulate.

    A and B: both fp16 or both bf16.  C: fp32, fp16 or bf16 (a 16-bit C is the
    FP32 epilogue value rounded once to nearest even).  bias: fp32 or None.
    """
    import torch
    types = {torch.float32: GEMM_DTYPE_F32, torch.float16: GEMM_DTYPE_F16, torch.bfloat16: GEMM_DTYPE_BF16}
    for name, t in (("A", A), ("B", B), ("C", C)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 2 or t.dtype not in types:
            raise TypeError(f"{name} must be a 2-D CUDA float32/float16/bfloat16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (leading dimension = width)")
    if A.dtype != B.dtype or A.dtype == torch.float32:
        raise TypeError("A and B must both be float16 or both bfloat16")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} B{tuple(B.shape)} C{tuple(C.shape)}")
    bias_ptr = 0
    if bias is not None:
        if not bias.is_cuda or bias.dtype != torch.float32 or bias.numel() != N or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous CUDA float32 tensor of length N")
        bias_ptr = bias.data_ptr()
    st = lib().gemm_tc_f32acc_epilogue(M, N, K, float(alpha), ctypes.c_void_p(A.data_ptr()),
                                       ctypes.c_void_p(B.data_ptr()), types[A.dtype], float(beta),
                                       ctypes.c_void_p(C.data_ptr()), types[C.dtype],
                                       ctypes.c_void_p(bias_ptr or None), int(act), _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tc_f32acc_epilogue")


def _batched_operand(t, name, rows, cols):
    """(pointer, batch stride in elements, batch) of a 2-D (shared) or 3-D operand
    whose matrices are row-major with unit column stride and row stride = cols."""
    if t.dim() == 2:
        if tuple(t.shape) != (rows, cols) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {rows} x {cols} matrix")
        return t.data_ptr(), 0, None
    if t.dim() != 3 or tuple(t.shape[1:]) != (rows, cols) or t.stride(2) != 1 or t.stride(1) != cols:
        raise ValueError(f"{name} must be (batch, {rows}, {cols}) with row-major matrices, got "
                         f"shape {tuple(t.shape)} strides {t.stride()}")
    return t.data_ptr(), t.stride(0), t.shape[0]


def gemm_tc_batched(A, B, C, alpha: float = 1.0, beta: float = 0.0, bias=None, act: int = 0, *,
                    b_trans: bool = False, stream=None) -> None:
    """C[z] = act(alpha * A[z] @ op(B[z]) + beta * C[z] + bias) for every z, one launch.

    C: (batch, M, N) fp32/fp16/bf16.  A: (batch, M, K) or a shared (M, K).
    B: (batch, K, N), or (batch, N, K) with b_trans=True (op(B) = B^T, e.g. the
    keys of Q K^T); a 2-D B is shared by the batch.  A 3-D operand may have
    batch stride 0 (torch.expand).  A and B both fp16 or both bf16.
    """
    import torch
    types = {torch.float32: GEMM_DTYPE_F32, torch.float16: GEMM_DTYPE_F16, torch.bfloat16: GEMM_DTYPE_BF16}
    for name, t in (("A", A), ("B", B), ("C", C)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in types:
            raise TypeError(f"{name} must be a CUDA float32/float16/bfloat16 tensor")
    if A.dtype != B.dtype or A.dtype == torch.float32:
        raise TypeError("A and B must both be float16 or both bfloat16")
    if C.dim() != 3:
        raise ValueError("C must be (batch, M, N)")
    batch, M, N = C.shape
    K = A.shape[-1]
    c_ptr, sc, _ = _batched_operand(C, "C", M, N)
    a_ptr, sa, ba = _batched_operand(A, "A", M, K)
    b_ptr, sb, bb = _batched_operand(B, "B", N if b_trans else K, K if b_trans else N)
    for nb, name in ((ba, "A"), (bb, "B")):
        if nb is not None and nb != batch:
            raise ValueError(f"{name} has batch {nb}, C has {batch}")
    if batch > 1 and sc < M * N:
        raise ValueError("C's matrices overlap (batch stride < M * N)")
    bias_ptr = 0
    if bias is not None:
        if not bias.is_cuda or bias.dtype != torch.float32 or bias.numel() != N or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous CUDA float32 tensor of length N")
        bias_ptr = bias.data_ptr()
    st = lib().gemm_tc_strided_batched(batch, M, N, K, float(alpha), ctypes.c_void_p(a_ptr), sa,
                                       ctypes.c_void_p(b_ptr), sb, types[A.dtype], 1 if b_trans else 0, float(beta),
                                       ctypes.c_void_p(c_ptr), sc if batch > 1 else M * N, types[C.dtype],
                                       ctypes.c_void_p(bias_ptr or None), int(act), _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tc_strided_batched")


def tune_set(entries) -> None:
    """Install a tuning table: an iterable of dicts (or TuneEntry) with keys
    path, M, N, K, variant, bn, splits.  An empty iterable clears the table."""
    rows = [e if isinstance(e, TuneEntry) else TuneEntry(**{k: int(e.get(k, 0)) for k, _ in TuneEntry._fields_})
            for e in entries]
    arr = (TuneEntry * max(1, len(rows)))(*rows)
    st = lib().gemm_tune_set(arr, len(rows))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tune_set")


def tune_get() -> list:
    """The installed tuning table as a list of dicts."""
    n = lib().gemm_tune_get(None, 0)
    arr = (TuneEntry * max(1, n))()
    n = lib().gemm_tune_get(arr, n)
    return [arr[i].as_dict() for i in range(n)]


def default_tuning_path() -> str:
    """The tuning table shipped for GB300 (written by ``autotune`` on one)."""
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "tuning", "gb300.json")


def load_tuning(path: str) -> int:
    """Install the table stored by ``autotune`` in a JSON file; returns the entry count."""
    import json
    with open(path) as f:
        doc = json.load(f)
    tune_set(doc["entries"])
    return len(doc["entries"])


def watchdog_selftest(wait_ms: int = 20, stream=None) -> int:
    """Enqueue the watchdog probe (a wait that must time out after wait_ms); returns the status."""
    return int(lib().gemm_watchdog_selftest(int(wait_ms), _stream_handle(stream)))


def pipeline_stall_selftest_raw(M, N, K, A_ptr, B_ptr, C_ptr, wait_ms=5, stream_ptr=0) -> int:
    """Enqueue the single-CTA tensor-core GEMM with its TMA producer switched off
    and every wait limited to wait_ms (the waits must run out); returns the status."""
    return int(lib().gemm_pipeline_stall_selftest(int(M), int(N), int(K), ctypes.c_void_p(A_ptr),
                                                  ctypes.c_void_p(B_ptr), ctypes.c_void_p(C_ptr), int(wait_ms),
                                                  ctypes.c_void_p(stream_ptr)))


def fma_rate_probe(packed: bool = True, iters: int = 4096, stream=None) -> float:
    """FP32 FMAs per clock per SM of an 8 x 8 outer product in registers,
    measured with the packed two-wide FMA form gemm_f32 uses (packed=True)
    or with scalar FMAs."""
    out = ctypes.c_double(0.0)
    st = lib().gemm_fma_rate_probe(1 if packed else 0, int(iters), ctypes.byref(out), _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_fma_rate_probe")
    return float(out.value)


def tma_read_probe(clusters: int, multicast: bool = False, stages: int = 4, kblocks: int = 512,
                   region_mb: int = 24, stream=None) -> dict:
    """Bytes per SM clock that each CTA receives through TMA (median over the
    CTAs) and the total GB/s, for `clusters` clusters of 2 CTAs streaming
    `kblocks` 32 KB stages (the 64-wide k block of a 256-row panel of a
    K-major FP16 operand with 4096-element rows, two 128-row boxes) from a
    `region_mb` MB region (24 MB stays in L2), each CTA loading its own copy
    or (multicast=True) one box per CTA multicast to both."""
    per_sm, total = ctypes.c_double(0.0), ctypes.c_double(0.0)
    st = lib().gemm_tma_read_probe(int(clusters), 1 if multicast else 0, int(stages), int(kblocks), int(region_mb),
                                   ctypes.byref(per_sm), ctypes.byref(total), _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tma_read_probe")
    return {"bytes_per_clock_per_sm": float(per_sm.value), "total_gbs": float(total.value)}


def tma_read_probe_raw(clusters, multicast, stages, kblocks, region_mb, per_sm_ptr, total_ptr, stream_ptr=0) -> int:
    """Direct C-ABI call of gemm_tma_read_probe (pointers: addresses of doubles, or 0)."""
    dp = ctypes.POINTER(ctypes.c_double)
    return int(lib().gemm_tma_read_probe(int(clusters), int(multicast), int(stages), int(kblocks), int(region_mb),
                                         ctypes.cast(per_sm_ptr, dp), ctypes.cast(total_ptr, dp),
                                         ctypes.c_void_p(stream_ptr)))


def fma_rate_probe_raw(packed, iters, out_ptr, stream_ptr=0) -> int:
    """Direct C-ABI call of gemm_fma_rate_probe (out_ptr: address of a double, or 0)."""
    return int(lib().gemm_fma_rate_probe(int(packed), int(iters), ctypes.cast(out_ptr, ctypes.POINTER(ctypes.c_double)),
                                         ctypes.c_void_p(stream_ptr)))


def tc_rate_probe(iters: int = 4096, stream=None) -> float:
    """The tensor core's dense FP16/BF16 rate per SM in FLOP per clock,
    measured by timing back-to-back MMAs on every SM (median over the SMs)."""
    out = ctypes.c_double(0.0)
    st = lib().gemm_tc_rate_probe(int(iters), ctypes.byref(out), _stream_handle(stream))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tc_rate_probe")
    return float(out.value)


def check(stream=None) -> int:
    """Synchronise the stream and return the watchdog status (GEMM_OK or GEMM_ERR_TIMEOUT)."""
    return int(lib().gemm_check(_stream_handle(stream)))
