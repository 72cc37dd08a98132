// internal.h -- host-side interfaces shared by the translation units of
// libgemm11.so (not installed, not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gemm11 {

// Scratch for split-K partial tiles and their arrival counters, owned by the
// library, one per (device, stream), grown on demand.  Counters are zero
// between calls: every kernel that increments one resets it.
struct Scratch {
    float *partials = nullptr;
    unsigned *counters = nullptr;
};
// Returns cudaSuccess and fills `out` with at least `partial_floats` floats and
// `ncounters` zeroed counters usable on `stream` (current device).
cudaError_t acquire_scratch(cudaStream_t stream, size_t partial_floats, size_t ncounters, Scratch *out);

// A second per-(device, stream) buffer for repacked operands (used together
// with the partials above), grown on demand.
cudaError_t acquire_operand_scratch(cudaStream_t stream, size_t floats, float **out);

// Device address of the current device's watchdog word.
unsigned *watchdog_word();

// GEMM11_DEBUG builds only: elements by which gemm_f32 shrinks the C extent
// its kernels check stores against (environment GEMM11_DEBUG_SHRINK_C, 0 if
// unset), so that a test can watch a device-side bounds check fire and skip
// the stores past it.  Release builds return 0 and never read it.
size_t debug_shrink_c();

// Plain launch through cudaLaunchKernelEx with an error check.  (The grid
// kernels here are not launched with programmatic stream serialization: their
// CTAs are placed several per SM, and letting the next kernel's CTAs take
// free slots early skewed that placement -- 1024^3 FP32 ran 51 -> 77 us.)
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

// Tuned plan for one exact shape, installed through gemm_tune_set (see the
// header for the meaning of the fields).  path 0: FP32 CUDA-core GEMM,
// path 1: tensor-core GEMM (single matrix).  Returns false when no entry
// matches; the planner then uses its own rules.
struct TunePlan {
    int variant = 0, bn = 0, splits = 0;
};
bool tune_lookup(int path, int M, int N, int K, TunePlan *out);

int device_sm_count();  // multiprocessors of the current device
int current_device_id();  // -1 if none

// Opt `kern` in to `bytes` of dynamic shared memory on the current device,
// once per (kernel, device): `done_mask` is a static owned by the caller's
// launcher instantiation (one per kernel), bit d set once device d is done.
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel kern, int bytes, unsigned long long &done_mask) {
    const int d = current_device_id();
    if (d < 0) return cudaErrorInvalidDevice;
    const unsigned long long bit = d < 64 ? (1ull << d) : 0ull;
    if (bit && (__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) __atomic_fetch_or(&done_mask, bit, __ATOMIC_RELEASE);
    return e;
}

struct CallInfo {
    const char *plan = "none";
    int launches = 0;
    bool tuned = false;  // the plan came from the tuning table
};

// ---- FP32 path (sgemm.cu) ----
cudaError_t run_gemm_f32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                         float beta, float *C, int ldc, cudaStream_t stream, CallInfo *info);

// ---- FP16 tensor-core path (hgemm.cu) ----
// Returns cudaSuccess, or cudaErrorNotSupported when the tensor-map encoder
// is unavailable.
// One tensor-core GEMM or a strided batch of them, every matrix row-major:
//   C_z = act(alpha * A_z * op(B_z) + beta * C_z + bias),  z < batch,
// A_z = A + z * stride_a (M x K), B_z = B + z * stride_b (K x N, or N x K
// with b_trans, op(B) = B^T), C_z = C + z * stride_c (M x N); strides in
// elements, 0 for an operand shared by the whole batch.  A and B are FP16
// (bf16 == false) or BF16 (bf16 == true); C is FP32, FP16 or BF16 (c_type:
// 0, 1, 2 -- the C ABI's gemm_dtype codes).  Every combination uses the same
// kernels and plans.
struct TcGemm {
    int batch = 1, M = 0, N = 0, K = 0;
    float alpha = 1.f, beta = 0.f;
    const void *A = nullptr;
    long long stride_a = 0;
    const void *B = nullptr;
    long long stride_b = 0;
    int b_trans = 0;
    void *C = nullptr;
    long long stride_c = 0;
    int c_type = 0;
    const float *bias = nullptr;
    int act = 0;
    bool bf16 = false;
};
cudaError_t run_gemm_f16(const TcGemm &g, cudaStream_t stream, CallInfo *info);

// FP32 GEMM on the tensor cores with three TF32 products per k step (operands
// split into high and low TF32 parts); C 16-byte aligned with ldc % 4 == 0.
cudaError_t run_gemm_f32_3xtf32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                                float beta, float *C, int ldc, cudaStream_t stream, CallInfo *info);

// The same small-M (M <= 64) transposed split-K plan with its scratch in a
// fixed device array (no allocation).  *reject = 1 if M > 64, 2 if the plan's
// scratch exceeds the array; nothing is launched then.
cudaError_t run_gemm_f16_small_m_noalloc(int M, int N, int K, float alpha, const void *A, const void *B, float beta,
                                         float *C, const float *bias, int act, cudaStream_t stream, CallInfo *info,
                                         int *reject);

// Diagnostic: the single-CTA tensor-core plan for C = A x B (FP16, 128 x 128
// tiles, no K split) with its TMA producer issuing nothing and every bounded
// wait of the kernel limited to wait_ns: the waits run out, the kernel
// records a timeout in the watchdog word and returns without writing C.
cudaError_t run_hgemm_stall_selftest(int M, int N, int K, const void *A, const void *B, float *C,
                                     unsigned long long wait_ns, cudaStream_t stream);

// C = beta * C over an M x N window (alpha == 0 or K == 0), with the epilogue
// bias/act applied when given (the FP16 path), in sgemm.cu.
cudaError_t run_scale_c(int M, int N, float beta, float *C, int ldc, const float *bias, int act,
                        cudaStream_t stream, CallInfo *info);
// The same over a strided batch of `batch` M x N matrices (ldc = N, matrices
// stride_c elements apart) of any output type (c_type 0 = FP32, 1 = FP16,
// 2 = BF16; a 16-bit value is computed in FP32 and rounded once to nearest
// even).
cudaError_t run_scale_c_batched(int batch, int M, int N, float beta, void *C, long long stride_c, int c_type,
                                const float *bias, int act, cudaStream_t stream, CallInfo *info);

// The tensor core's dense kind::f16 rate (FLOP per SM clock), measured by
// timing back-to-back 128 x 256 x 16 MMAs on every SM (probe.cu); synchronous
// on `stream`.  cudaErrorLaunchTimeout if no SM finished within the bounded wait.
cudaError_t run_tc_rate_probe(int iters, double *flop_per_clock_per_sm, cudaStream_t stream);
// FP32 FMAs per clock per SM, packed (__ffma2_rn) or scalar, measured.
cudaError_t run_fma_rate_probe(bool packed, int iters, double *fma_per_clock_per_sm, cudaStream_t stream);
// TMA read rate per SM (bytes per SM clock, median over the CTAs) and in
// total (GB/s, CUDA events) for `clusters` clusters of 2 CTAs streaming
// `kblocks` 32 KB stages from a `region_mb` MB region, with or without
// cluster multicast; synchronous on `stream`.
cudaError_t run_tma_read_probe(int clusters, bool multicast, int stages, int kblocks, int region_mb,
                               double *bytes_per_clock_per_sm, double *total_gbs, cudaStream_t stream);

}  // namespace gemm11
