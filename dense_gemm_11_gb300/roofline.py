"""Work and traffic accounting for the roofline figures.

FLOPs and algorithmic bytes follow the pages' own accounting:
  * "SGEMM优化，从naive到warptiling", section 项目概况 / 问题与估算: 2*M*N*K
    flops; A and B read once, C read once and written once (4 bytes each);
  * "第24讲 ... GEMM 分块与 Tensor Core 思维", section 1.1: the same count
    without the C read when C is only written;
  * the DeepGEMM essay "企业官网建设流程全解析", section 1.2: FP16 inputs are
    2 bytes per element.
The epilogue's O(M*N) operations are not counted as flops, as on the pages.
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int, batch: int = 1) -> int:
    return 2 * batch * M * N * K


def gemm_bytes(M: int, N: int, K: int, *, in_bytes: int, beta_nonzero: bool,
               bias: bool = False, out_bytes: int = 4, batch: int = 1) -> int:
    """Minimum bytes a GEMM (or each of `batch` independent ones) must move:
    A and B once, C written (and read if beta != 0), the bias once."""
    b = batch * (in_bytes * (M * K + K * N) + out_bytes * M * N * (2 if beta_nonzero else 1))
    if bias:
        b += 4 * N
    return b


def fp32_fma_peak_tflops(sm_count: int, sm_mhz: float, lanes_per_sm: int = 128) -> float:
    """CUDA-core FP32 peak: SMs x FP32 lanes per SM x 2 flops per FFMA x clock."""
    return sm_count * lanes_per_sm * 2 * sm_mhz * 1e6 / 1e12


def roofline_tflops(flops: int, nbytes: int, peak_tflops: float, hbm_gbs: float) -> tuple:
    """min(compute peak, HBM bandwidth x arithmetic intensity), and which one binds."""
    ai = flops / nbytes
    mem_bound = hbm_gbs * 1e9 * ai / 1e12
    if mem_bound < peak_tflops:
        return mem_bound, "hbm"
    return peak_tflops, "compute"
