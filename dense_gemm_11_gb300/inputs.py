"""Seeded synthetic inputs for the GEMM workloads.

This module draws random numbers and rounds them to the input precision; it
holds none of the GEMM arithmetic.  The CUDA path and the CPU oracle both take
their inputs from here, so both see the identical arrays.

Recipe (the same for every workload):
  * generator ``numpy.random.default_rng(seed)`` (PCG64);
  * draw order A, then B, then C, then bias; each drawn as float64 and then
    cast (float32, or float16 with round-to-nearest-even; bf16 inputs are
    cast to float32 and then rounded to bfloat16, nearest-even on the float32
    bit pattern, and held in float32 arrays whose values are all exact
    bfloat16 numbers -- numpy has no bfloat16 type);
  * ``uniform`` = U[-1, 1]; ``normal`` = N(0, sigma) with sigma the standard
    deviation; ``normal_k`` = N(0, 1/sqrt(K)); ``smallint`` = integers drawn
    uniformly from [-4, 4] (exact in fp16, bf16 and fp32; every partial sum of K
    products stays below 2**24 for K <= 2**20);
  * when beta == 0, C is filled with NaN so that a kernel that reads it fails.

Workloads (the shapes, value distributions, alpha and beta of the pages'
benchmarks; the M=N=K=4096 square is the one "SGEMM优化，从naive到warptiling"
(section 项目概况) and the DeepGEMM essay "企业官网建设流程全解析" (section 5.1)
time):
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "f32", "f16", "bf16", or "f32x3" (FP32 through gemm_f32_3xtf32)
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dist: str            # uniform | normal | normal_k | smallint
    seed: int
    bias: bool = False   # 16-bit inputs only: bias ~ N(0, 0.1), fp32, length N
    act: int = 0         # 0 none, 1 exact GELU, 2 ReLU, 3 tanh GELU
    note: str = ""
    batch: int = 1       # > 1: a strided batch of independent GEMMs
    b_trans: bool = False  # B stored N x K (op(B) = B^T)
    out: str = "f32"     # element type of C: f32, f16 or bf16

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K


SWEEP_SIZES = (128, 256, 512, 1024, 2048, 4096)
IRREGULAR_SHAPES = ((1000, 3000, 777), (4095, 4097, 4099), (1, 4096, 4096), (4096, 1, 4096))
EPILOGUE_SHAPES = ((16, 4096, 4096), (128, 11008, 4096), (4096, 11008, 4096), (4096, 4096, 11008))


def _registry():
    w = {}
    w["f32_512"] = Workload("f32_512", "f32", 512, 512, 512, 1.0, 0.5, "uniform", 0,
                            note="FP32 512^3, alpha 1, beta 0.5, U[-1,1], seed 0")
    for i, s in enumerate(SWEEP_SIZES):
        w[f"f32_sq{s}"] = Workload(f"f32_sq{s}", "f32", s, s, s, 1.0, 3.0, "uniform", i,
                                   note=f"FP32 square sweep {s}^3, beta 3, C reset each run")
    for i, (m, n, k) in enumerate(IRREGULAR_SHAPES):
        w[f"f32_irr{i}"] = Workload(f"f32_irr{i}", "f32", m, n, k, 0.7, 0.0, "normal", i,
                                    note=f"FP32 irregular {m}x{n}x{k}, lda=K ldb=N ldc=N")
    w["f16_4096"] = Workload("f16_4096", "f16", 4096, 4096, 4096, 1.0, 0.0, "normal_k", 0,
                             note="FP16-in FP32-acc 4096^3")
    w["f16_4096_int"] = Workload("f16_4096_int", "f16", 4096, 4096, 4096, 1.0, 0.0, "smallint", 0,
                                 note="FP16-in 4096^3, integers in [-4,4], exact")
    for i, (m, n, k) in enumerate(EPILOGUE_SHAPES):
        w[f"f16_epi{i}"] = Workload(f"f16_epi{i}", "f16", m, n, k, 0.5, 0.0, "normal_k", i,
                                    bias=True, act=1,
                                    note=f"FP16 GELU(0.5*A*B+bias) {m}x{n}x{k}")
    w["bf16_4096"] = Workload("bf16_4096", "bf16", 4096, 4096, 4096, 1.0, 0.0, "normal_k", 10,
                              note="BF16-in FP32-acc 4096^3")
    w["bf16_4096_int"] = Workload("bf16_4096_int", "bf16", 4096, 4096, 4096, 1.0, 0.0, "smallint", 11,
                                  note="BF16-in 4096^3, integers in [-4,4], exact")
    for i, ((m, n, k), act) in enumerate(zip(EPILOGUE_SHAPES, (2, 3, 2, 3))):
        w[f"bf16_epi{i}"] = Workload(f"bf16_epi{i}", "bf16", m, n, k, 0.5, 0.0, "normal_k", 12 + i,
                                     bias=True, act=act,
                                     note=f"BF16 {'ReLU' if act == 2 else 'tanh-GELU'}(0.5*A*B+bias) {m}x{n}x{k}")
    w["f32x3_4096"] = Workload("f32x3_4096", "f32x3", 4096, 4096, 4096, 1.0, 3.0, "uniform", 3,
                               note="FP32 4096^3 on the tensor cores (3 x TF32), beta 3, C reset each run")
    w["f16_4096_out16"] = Workload("f16_4096_out16", "f16", 4096, 4096, 4096, 1.0, 0.0, "normal_k", 16,
                                   out="f16", note="FP16-in FP32-acc 4096^3, FP16 C")
    # Attention products per head (32 = batch 4 x 8 heads, sequence 2048, head
    # dimension 128): scores Q K^T / sqrt(d) with the keys stored S x d, and
    # P V; BF16 in and out.  P is a stand-in drawn like the other operands.
    w["bf16_attn_qk"] = Workload("bf16_attn_qk", "bf16", 2048, 2048, 128, 128 ** -0.5, 0.0, "normal", 17,
                                 batch=32, b_trans=True, out="bf16",
                                 note="32 x (2048x128) (2048x128)^T / sqrt(128), BF16 in/out")
    w["bf16_attn_pv"] = Workload("bf16_attn_pv", "bf16", 2048, 128, 2048, 1.0, 0.0, "normal_k", 18,
                                 batch=32, out="bf16", note="32 x (2048x2048) (2048x128), BF16 in/out")
    return w


WORKLOADS = _registry()


def _draw(rng, dist, shape, K):
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    if dist == "normal":
        return rng.normal(0.0, 1.0, size=shape)
    if dist == "normal_k":
        return rng.normal(0.0, 1.0 / np.sqrt(max(K, 1)), size=shape)
    if dist == "smallint":
        return rng.integers(-4, 5, size=shape).astype(np.float64)
    raise ValueError(f"unknown distribution {dist!r}")


def round_to_bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as float32.

    x is cast to float32 first; the low 16 bits of each float32 pattern are
    then rounded away.  Finite inputs only (the generators draw no inf/NaN).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _cast_input(x, kind):
    if kind in ("f32", "f32x3"):
        return x.astype(np.float32)
    if kind == "f16":
        return x.astype(np.float16)
    if kind == "bf16":
        return round_to_bf16(x)
    raise ValueError(f"unknown input kind {kind!r}")


def make(M, N, K, *, kind="f32", dist="uniform", seed=0, beta=0.0, bias=False,
         lda=None, ldb=None, ldc=None):
    """Draw A (M x lda), B (K x ldb), C (M x ldc) and bias (N) for one GEMM.

    Leading dimensions default to the widths (K, N, N).  Columns past the
    logical width are drawn too (they are part of the buffer but never part of
    the product).  Returns a dict with numpy arrays: A and B are float32
    (kind "f32"), float16 (kind "f16") or float32 holding bfloat16 values
    (kind "bf16"); C and bias are float32.
    """
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    if lda < K or ldb < N or ldc < N:
        raise ValueError("leading dimension smaller than the width")
    rng = np.random.default_rng(seed)
    A = _cast_input(_draw(rng, dist, (M, lda), K), kind)
    B = _cast_input(_draw(rng, dist, (K, ldb), K), kind)
    if beta != 0.0:
        Cdist = "uniform" if dist in ("uniform", "normal_k") else dist
        C = _draw(rng, Cdist, (M, ldc), K).astype(np.float32)
    else:
        C = np.full((M, ldc), np.nan, dtype=np.float32)
    out = {"A": A, "B": B, "C": C}
    if bias:
        out["bias"] = rng.normal(0.0, 0.1, size=(N,)).astype(np.float32)
    return out


def make_batched(batch, M, N, K, *, kind="f16", dist="normal_k", seed=0, beta=0.0, bias=False, b_trans=False):
    """Draw a strided batch: A (batch, M, K), B (batch, K, N) -- or
    (batch, N, K) with b_trans, the layout of attention keys -- C
    (batch, M, N) and bias (N); same recipe and draw order as make()."""
    rng = np.random.default_rng(seed)
    A = _cast_input(_draw(rng, dist, (batch, M, K), K), kind)
    B = _cast_input(_draw(rng, dist, (batch, N, K) if b_trans else (batch, K, N), K), kind)
    if beta != 0.0:
        Cdist = "uniform" if dist in ("uniform", "normal_k") else dist
        C = _draw(rng, Cdist, (batch, M, N), K).astype(np.float32)
    else:
        C = np.full((batch, M, N), np.nan, dtype=np.float32)
    out = {"A": A, "B": B, "C": C}
    if bias:
        out["bias"] = rng.normal(0.0, 0.1, size=(N,)).astype(np.float32)
    return out


def make_workload(w: Workload):
    if w.batch > 1 or w.b_trans:
        return make_batched(w.batch, w.M, w.N, w.K, kind=w.kind, dist=w.dist, seed=w.seed, beta=w.beta,
                            bias=w.bias, b_trans=w.b_trans)
    return make(w.M, w.N, w.K, kind=w.kind, dist=w.dist, seed=w.seed, beta=w.beta, bias=w.bias)
