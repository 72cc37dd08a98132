/*
 * gemm11.h -- C ABI of the GB300 (sm_103a) dense GEMM library libgemm11.so.
 *
 * The operation is the dense matrix product
 *
 *     C = alpha * A x B + beta * C
 *
 * on row-major operands, as defined in "SGEMM优化，从naive到warptiling"
 * (section 项目概况 / 问题与估算: A is MxK, B is KxN, C is MxN, all row-major
 * float).  The FP16-input variant accumulates in FP32 and folds bias, scale
 * and an activation into the epilogue, as the DeepGEMM essay
 * "企业官网建设流程全解析" describes (sections 1.3 "定制点" and 3.2, where the
 * epilogue applies bias, scale and activation to the accumulator before the
 * single store).
 *
 * Conventions shared by every entry point:
 *   - Pointers A, B, C, bias are DEVICE pointers (CUDA global memory of the
 *     current device).  The caller owns them; the library keeps no pointer
 *     after the call returns, apart from the work it has enqueued.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous and stream-ordered: they return once the work is enqueued.
 *   - A, B and bias are read only.  C is read (only when beta != 0) and written
 *     in place.  A, B and C must not overlap.
 *   - Degenerate shapes follow BLAS: M == 0 or N == 0 is a no-op; K == 0 or
 *     alpha == 0 gives C = beta * C without reading A or B; beta == 0 makes C
 *     write-only (NaN or Inf already in C do not propagate).
 *   - Argument errors are detected on the host before anything is launched
 *     and return GEMM_ERR_INVALID_ARG or GEMM_ERR_UNSUPPORTED.
 *   - A CUDA error while enqueueing returns GEMM_ERR_CUDA;
 *     gemm_last_cuda_error() gives the cudaError_t.  Faults during execution
 *     show up at the caller's next synchronisation, as for any CUDA kernel.
 *   - Every wait inside a kernel is bounded.  If one runs out (a pipeline that
 *     stopped making progress) the kernel records it in a device-side status
 *     word and returns early; gemm_check() reports it as GEMM_ERR_TIMEOUT.
 *   - Split-K shapes use a library-owned workspace, allocated lazily once per
 *     (device, stream) and reused; calls on one stream are serialised by the
 *     stream, calls on different streams use different workspaces.
 *   - Debug build.  The same sources compiled with GEMM11_DEBUG=1 give
 *     libgemm11_debug.so (the Python binding loads it when the environment
 *     variable GEMM11_DEBUG is 1).  The DeepGEMM essay "企业官网建设流程全解析"
 *     (section 6.1) advises starting fully synchronous and relaxing later;
 *     this build is the synchronous end of that:
 *       - the pipelines keep one operand stage in flight (the FP32 path
 *         waits for every outstanding copy before it reads a stage; the
 *         tensor-core producers wait for the MMA to consume each stage);
 *       - stores to C and accesses to library scratch check their index
 *         against the extent; a failing check records a fault bit in the
 *         device status word and the access is skipped (nothing traps);
 *       - library scratch is allocated with guard bands of 4 KiB on both
 *         sides, filled with 0xA5 and checked after every call;
 *       - every compute call synchronises its stream before it returns and
 *         returns GEMM_ERR_DEBUG_CHECK (index or guard band) or
 *         GEMM_ERR_TIMEOUT when the device reported one.  Calls are therefore
 *         blocking in this build.
 *     Release builds compile all of this away (gemm_debug_build() tells them
 *     apart).
 */
#ifndef GEMM11_H
#define GEMM11_H

#if defined(__GNUC__)
#define GEMM11_API __attribute__((visibility("default")))
#else
#define GEMM11_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1, /* bad dimension, leading dimension, pointer or enum */
    GEMM_ERR_UNSUPPORTED = -2, /* valid arguments this path cannot take (alignment) */
    GEMM_ERR_CUDA = -3,        /* a CUDA runtime call failed; see gemm_last_cuda_error() */
    GEMM_ERR_TIMEOUT = -4,     /* a bounded in-kernel wait ran out (from gemm_check) */
    GEMM_ERR_SCRATCH_LIMIT = -5, /* the no-allocation entry point's fixed scratch is too small */
    GEMM_ERR_DEBUG_CHECK = -6   /* GEMM11_DEBUG builds: a device-side check failed (see below) */
} gemm_status;

typedef enum {
    GEMM_ACT_NONE = 0,      /* identity */
    GEMM_ACT_GELU = 1,      /* exact GELU: x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2))) */
    GEMM_ACT_RELU = 2,      /* max(x, 0) */
    GEMM_ACT_GELU_TANH = 3  /* 0.5 * x * (1 + tanh(sqrt(2/pi) * (x + 0.044715 * x^3))) */
} gemm_act;

/* Element types of the tensor-core entry point gemm_tc_f32acc_epilogue. */
typedef enum {
    GEMM_DTYPE_F32 = 0,  /* IEEE binary32 */
    GEMM_DTYPE_F16 = 1,  /* IEEE binary16 (__half) */
    GEMM_DTYPE_BF16 = 2  /* bfloat16 (__nv_bfloat16): binary32 with the low 16 bits dropped */
} gemm_dtype;

/*
 * gemm_f32 -- true-FP32 SGEMM on the CUDA cores (FFMA, round-to-nearest).
 *   C[i*ldc + j] = alpha * sum_k A[i*lda + k] * B[k*ldb + j] + beta * C[i*ldc + j]
 * for 0 <= i < M, 0 <= j < N.  Definition: "SGEMM优化，从naive到warptiling",
 * section 项目概况 / 问题与估算 (and the naive kernel of section k1, which is
 * the same sum written as one thread per C element).
 *   M, N, K  >= 0.
 *   A        M x K, row-major, leading dimension lda >= max(1, K) (elements).
 *   B        K x N, row-major, ldb >= max(1, N).
 *   C        M x N, row-major, ldc >= max(1, N).
 * Any alignment and any leading dimension are accepted; 16-byte aligned
 * operands with leading dimensions that are multiples of 4 take the
 * vector-load path, others a 4-byte path with the same results.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (negative size, short leading
 * dimension, NULL pointer with a non-empty extent) or GEMM_ERR_CUDA.
 */
GEMM11_API int gemm_f32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
             float beta, float *C, int ldc, void *stream);

/*
 * gemm_f32_3xtf32 -- the operation, arguments and return codes of gemm_f32,
 * computed on the tcgen05 tensor cores instead of the FP32 FMA units (opt in;
 * gemm_f32 is unchanged).  Each FP32 operand x is split into a TF32 high
 * part h = tf32(x) and a TF32 low part l = tf32(x - h), and each product is
 * taken as a_h b_h + a_h b_l + a_l b_h, which drops terms of about
 * 2^-21 |a b|.  The tensor core sums chunks of 128 k (its FP32 accumulation
 * truncates, a bias that would grow with K); the chunk sums are added in
 * FP32 with round-to-nearest on the CUDA cores.  Measured on GB300: at most
 * 1.7e-6 S for same-sign data and 4e-7 S for mixed signs, for K from 256 to
 * 16384 -- inside gemm_f32's bound |C - C_exact| <= 1e-5 S + 1e-6, but not
 * bit-identical to gemm_f32.
 * "SGEMM优化，从naive到warptiling" (Q9, the optimisations not made) lists
 * TF32 / tensor cores; "第 11 章 Tiled GEMM" (section 11.7) puts the FP32
 * CUDA-core peak at about 1/15 of the dense FP16 tensor-core peak.
 *   Extra constraint: C 16-byte aligned and, when M > 1, ldc % 4 == 0 (C is
 *   written by TMA stores), otherwise GEMM_ERR_UNSUPPORTED; A and B may have any
 *   alignment and leading dimension.  Scratch: 16 (M + N) K' bytes of
 *   library-owned device memory per stream, K' = K rounded up to 4.  Inputs
 *   within 2^-11 of the FP32 overflow threshold are outside the method (their
 *   TF32 high part rounds to infinity).
 */
GEMM11_API int gemm_f32_3xtf32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                               float beta, float *C, int ldc, void *stream);

/*
 * gemm_f16_f32acc_epilogue -- FP16 inputs, FP32 accumulation on the tcgen05
 * tensor cores, fused epilogue:
 *   C[i*N + j] = act( alpha * sum_k A[i*K + k] * B[k*N + j] + beta * C[i*N + j] + bias[j] )
 * Definition: the DeepGEMM essay "企业官网建设流程全解析", sections 1.2
 * (FP16 input, FP32 accumulate), 1.3 and 3.2 (bias, scale and activation in
 * the epilogue); alpha is the scale.
 *   A     __half, M x K, row-major, lda = K.
 *   B     __half, K x N, row-major, ldb = N.
 *   C     float,  M x N, row-major, ldc = N.
 *   bias  float, length N, or NULL for no bias.
 *   act   one of gemm_act; any other value returns GEMM_ERR_INVALID_ARG.
 *         The pages name an activation (GELU) in the epilogue without fixing
 *         its form; exact GELU, ReLU and the tanh form of GELU are offered.
 * The tensor-memory-access path needs K % 8 == 0, N % 8 == 0 and A, B, C
 * 16-byte aligned ("第24讲 ... GEMM 分块与 Tensor Core 思维", section 7.2 item 7:
 * pad tensor-core operands to aligned sizes); anything else returns
 * GEMM_ERR_UNSUPPORTED.  M is unrestricted.
 */
GEMM11_API int gemm_f16_f32acc_epilogue(int M, int N, int K, float alpha, const void *A, const void *B,
                             float beta, float *C, const float *bias, int act, void *stream);

/*
 * gemm_bf16_f32acc_epilogue -- gemm_f16_f32acc_epilogue with BF16 inputs:
 * A and B hold __nv_bfloat16 values (8 exponent bits, 8 significand bits),
 * everything else -- the formula, C, bias, act, the alignment rules, the
 * return codes and the kernels -- is the same.  "第24讲 ... GEMM 分块与
 * Tensor Core 思维", section 5.1 (tensor-core half precision is FP16/BF16)
 * and section 7.2 item 7 (large-model tensor-core operands are FP16 or BF16).
 * Products of two BF16 values are exact in FP32, so the accuracy bound is the
 * FP16 path's: rounding of the FP32 accumulation only.
 */
GEMM11_API int gemm_bf16_f32acc_epilogue(int M, int N, int K, float alpha, const void *A, const void *B,
                                         float beta, float *C, const float *bias, int act, void *stream);

/*
 * gemm_tc_f32acc_epilogue -- the general form of the two entry points above:
 * A and B of element type ab_type (GEMM_DTYPE_F16 or GEMM_DTYPE_BF16), FP32
 * accumulation, and C of element type c_type (GEMM_DTYPE_F32, GEMM_DTYPE_F16
 * or GEMM_DTYPE_BF16):
 *   C[i*N + j] = round_c( act( alpha * sum_k A[i*K + k] * B[k*N + j]
 *                              + beta * C[i*N + j] + bias[j] ) )
 * Everything inside round_c is evaluated in FP32 (the beta term reads the
 * 16-bit C and widens it exactly); round_c is the identity for FP32 and one
 * round-to-nearest-even for the 16-bit types (overflow gives +-inf).  The
 * DeepGEMM essay "企业官网建设流程全解析" (section 1.1) argues for folding
 * the work around a GEMM into its epilogue so that no extra pass over HBM
 * is needed; a 16-bit C is one more such step (it halves C's bytes).
 * Layouts, alignment rules (C 16-byte aligned, N % 8 == 0, K % 8 == 0) and
 * return codes are those of gemm_f16_f32acc_epilogue; an ab_type or c_type
 * outside the lists above returns GEMM_ERR_INVALID_ARG.
 */
GEMM11_API int gemm_tc_f32acc_epilogue(int M, int N, int K, float alpha, const void *A, const void *B, int ab_type,
                                       float beta, void *C, int c_type, const float *bias, int act, void *stream);

/*
 * gemm_tc_strided_batched -- `batch` independent tensor-core GEMMs in one
 * launch, each the operation of gemm_tc_f32acc_epilogue:
 *   C_z = round_c( act( alpha * A_z * op(B_z) + beta * C_z + bias ) ),  0 <= z < batch
 *   A_z = A + z * stride_a   M x K, row-major
 *   B_z = B + z * stride_b   K x N row-major (b_trans = 0, op(B) = B) or
 *                            N x K row-major (b_trans = 1, op(B) = B^T)
 *   C_z = C + z * stride_c   M x N, row-major
 * Strides count elements of the operand's type.  stride_a or stride_b may be
 * 0 (one matrix shared by the whole batch); stride_c >= M * N (the outputs
 * must not overlap).  bias (length N) is shared by every matrix.  The pages
 * name attention as the consumer of such products: "第24讲 ... GEMM 分块与
 * Tensor Core 思维" (its opening guide: QK^T and PV are GEMMs) and the DeepGEMM
 * essay "企业官网建设流程全解析" (section 1.1: projections, attention and FFN
 * are GEMMs); QK^T is the b_trans = 1 form (K stored row-major, S x d).
 * Alignment, as for the single GEMM: A, B, C 16-byte aligned, K % 8 == 0,
 * N % 8 == 0, and for batch > 1 every stride % 8 == 0; otherwise
 * GEMM_ERR_UNSUPPORTED.  batch < 0, b_trans not 0/1, a negative stride or
 * stride_c < M * N (batch > 1) return GEMM_ERR_INVALID_ARG; batch == 0 is a
 * no-op.  The tiles of all matrices form one persistent schedule (one launch
 * for the whole batch).
 */
GEMM11_API int gemm_tc_strided_batched(int batch, int M, int N, int K, float alpha, const void *A, long long stride_a,
                                       const void *B, long long stride_b, int ab_type, int b_trans, float beta,
                                       void *C, long long stride_c, int c_type, const float *bias, int act,
                                       void *stream);

/*
 * gemm_f16_f32acc_epilogue_noalloc -- the same operation and arguments as
 * gemm_f16_f32acc_epilogue, restricted to M <= 64, and guaranteed not to
 * allocate: no cudaMalloc, cudaFree or allocating library routine is called.
 * The pages have no counterpart; this entry point exists for callers that
 * cannot let a library allocate device memory on their behalf, for example a
 * serving loop that reserved all of its memory up front and runs under a
 * fixed budget (a cudaMalloc there can fail under memory pressure, and
 * cudaMalloc/cudaFree may synchronise the whole device and stall the
 * caller's other streams).
 *   Scratch: the split-K partial tiles of the small-M plan live in one
 *   file-scope device array of this library (4 MiB of fp32 partials plus
 *   4096 arrival counters, 4 MiB + 16 KiB); every GPU on which the library's
 *   kernels have been loaded holds it until the process exits.  The K split
 *   count is lowered until the partials fit in the array; a shape for which
 *   not even two splits fit (on a 152-SM GPU only 33 <= M <= 64 with
 *   8193 <= N <= 9728 and K >= 256) returns GEMM_ERR_SCRATCH_LIMIT without launching anything.
 *   M > 64 (in every case, also with alpha == 0, K == 0 or N == 0) and the
 *   alignment rules of gemm_f16_f32acc_epilogue return GEMM_ERR_UNSUPPORTED.
 *   When the array reaches the GPU: under CUDA's default lazy module loading
 *   the driver places the library's kernels -- and this array with them --
 *   on a device when they are first used, which may be this entry point's
 *   first call.  A caller that reserves a fixed memory budget should make one
 *   warm-up call (or set CUDA_MODULE_LOADING=EAGER) before reserving it.
 *   The first call on a device also looks up the array's device address
 *   (with that device current; a failed lookup is retried on the next call);
 *   make that first call before any stream capture.  Every call zeroes the
 *   counters it uses (an async memset on `stream`) before its kernel.
 *   All calls share the one array: calls whose execution overlaps on the GPU
 *   (for example on two streams at once) race on it and give wrong results.
 *   Serialise them, e.g. by issuing them on one stream.
 */
GEMM11_API int gemm_f16_f32acc_epilogue_noalloc(int M, int N, int K, float alpha, const void *A, const void *B,
                                                float beta, float *C, const float *bias, int act, void *stream);

/*
 * Tuned plans.  The planners pick a kernel family, tile width and split-K
 * factor from the shape by fixed rules; a tuning table replaces those rules
 * for exact shapes.  The pages tune the same parameters per shape and per GPU
 * ("SGEMM优化，从naive到warptiling", kernel 9 autotuning and Q10; the DeepGEMM
 * essay "企业官网建设流程全解析", section 1.3, searches tile sizes for the
 * fixed shapes of an inference service).  dense_gemm_11_gb300/autotune.py
 * times the candidates on the GPU and writes such a table.
 *   path     GEMM_PATH_F32: gemm_f32 (M > 1 and N > 1; the GEMV shapes are
 *            not tunable); GEMM_PATH_TC: the tensor-core entry points for a
 *            single matrix (any input/output type; batches are not looked up).
 *   M, N, K  the exact shape.
 *   variant  GEMM_PATH_F32: 1 = 128 x 256 persistent tiles with stream-K,
 *              2 = 64 x 64 tiles with `splits` K slices (0: the planner's count).
 *            GEMM_PATH_TC: 1 = CTA pairs, bn in {256, 224, 192};
 *              2 = single-CTA 128-row tiles, bn in {256, 128}, `splits` K slices;
 *              3 = transposed small-M product (needs M <= bn), bn in {32, 64},
 *              `splits` K slices;
 *              4 = single-CTA 128-row tiles whose K is split over the 2..8
 *              CTAs of a thread-block cluster (partials added in distributed
 *              shared memory), bn in {256, 192, 128}, splits = cluster size
 *              in 2..8 or 0; every CTA of the launch must fit on the GPU at
 *              once (one per SM), else the entry is ignored.
 *   bn       tile width (0: the planner's choice within the family).
 *   splits   split-K factor, 0..32 (0: the planner's rule; clipped to half
 *            the number of 64-wide k blocks).
 * An entry whose family cannot run the shape it names (variant 3 with
 * M > bn, variant 4 with too many CTAs) is ignored at call time.  Results are identical in value across
 * plans only up to the accumulation order.
 */
typedef enum { GEMM_PATH_F32 = 0, GEMM_PATH_TC = 1 } gemm_tune_path;
typedef struct {
    int path, M, N, K;
    int variant, bn, splits;
} gemm_tune_entry;

/*
 * gemm_tune_set -- replace the process-wide tuning table with entries[0..n)
 * (n = 0 clears it; later entries for the same path and shape win).  Returns
 * GEMM_ERR_INVALID_ARG, leaving the table unchanged, if n < 0, entries is
 * NULL with n > 0, or an entry has an unknown path or variant, a tile width
 * outside its family's list, a negative size or splits outside 0..32.
 * Thread-safe; takes effect for calls made after it returns.
 */
GEMM11_API int gemm_tune_set(const gemm_tune_entry *entries, int n);

/* gemm_tune_get -- copy up to `capacity` entries of the table to `out`;
 * returns the number of entries in the table. */
GEMM11_API int gemm_tune_get(gemm_tune_entry *out, int capacity);

/* 1 in a GEMM11_DEBUG build of the library, 0 in a release build. */
GEMM11_API int gemm_debug_build(void);

/* Text for a gemm_status value (static storage, never NULL). */
GEMM11_API const char *gemm_status_string(int status);

/* cudaError_t of the last CUDA failure seen by this thread's calls (0 if none). */
GEMM11_API int gemm_last_cuda_error(void);

/*
 * gemm_check -- synchronise `stream`, then read and clear the current
 * device's watchdog word.  Returns GEMM_ERR_TIMEOUT if a bounded wait ran out
 * in any kernel since the previous check (GEMM_ERR_DEBUG_CHECK instead when a
 * debug build's device-side check failed), GEMM_ERR_CUDA if the
 * synchronisation failed, GEMM_OK otherwise.
 */
GEMM11_API int gemm_check(void *stream);

/*
 * gemm_watchdog_selftest -- diagnostic: enqueue on `stream` a one-thread
 * kernel whose bounded wait (the same wait every GEMM pipeline uses) can
 * never be satisfied, with a limit of wait_ms milliseconds (1..2000).  The
 * kernel returns normally after the limit and records the timeout in the
 * device watchdog word, so the next gemm_check(stream) returns
 * GEMM_ERR_TIMEOUT (and clears it).  This exercises the timeout path without
 * faulting, trapping or hanging the GPU; the context stays usable.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG or GEMM_ERR_CUDA.
 */
GEMM11_API int gemm_watchdog_selftest(int wait_ms, void *stream);

/*
 * gemm_pipeline_stall_selftest -- diagnostic: the timeout path of a real GEMM
 * pipeline.  Enqueues on `stream` the single-CTA tensor-core plan of
 * gemm_f16_f32acc_epilogue (128 x 128 tiles, no K split) for C = A x B, with
 * its TMA producer switched off -- it issues no load and makes no arrival --
 * and every bounded wait of the kernel limited to wait_ms milliseconds
 * (1..2000) instead of the usual 2 s.  The MMA thread's wait for the first
 * operand stage and the epilogue warps' wait for the accumulator run out;
 * the kernel records the timeout in the device watchdog word, frees its
 * tensor memory and returns without writing C (nothing is in flight: no copy
 * was issued), so the next gemm_check(stream) returns GEMM_ERR_TIMEOUT and
 * the context stays usable.  The DeepGEMM essay "企业官网建设流程全解析"
 * (section 6.1) describes the asynchronous-pipeline hazards this guards.
 *   A, B, C, M, N, K: as for gemm_f16_f32acc_epilogue (FP16 A and B, FP32 C,
 *   M, N, K >= 1, K % 8 == 0, N % 8 == 0, 16-byte aligned pointers); A and B
 *   are not read.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (wait_ms out of range, a size < 1, a
 * NULL pointer), GEMM_ERR_UNSUPPORTED (alignment) or GEMM_ERR_CUDA.
 */
GEMM11_API int gemm_pipeline_stall_selftest(int M, int N, int K, const void *A, const void *B, float *C, int wait_ms,
                                            void *stream);

/*
 * gemm_tc_rate_probe -- diagnostic: the tensor core's dense FP16/BF16 rate
 * per SM, measured.  One CTA per SM issues `iters` x 4 back-to-back
 * tcgen05.mma instructions of shape 128 x 256 x 16 (BF16 operands resident in
 * shared memory, FP32 accumulator in tensor memory; no global-memory
 * traffic) and times them with the SM cycle counter; *flop_per_clock_per_sm
 * receives the median over the SMs of 2 * 128 * 256 * 16 * 4 * iters /
 * cycles.  #SM x this rate x the SM clock is the nominal dense peak that the
 * FP16 path's throughput is quoted against besides the measured cuBLAS rate.
 * Synchronous on `stream` (it allocates and frees a small device buffer).
 * iters in 1..2^20 (a few thousand take about a millisecond).  Returns
 * GEMM_OK, GEMM_ERR_INVALID_ARG (iters out of range, NULL output),
 * GEMM_ERR_TIMEOUT (no SM completed within the bounded wait) or
 * GEMM_ERR_CUDA.
 */
GEMM11_API int gemm_tc_rate_probe(int iters, double *flop_per_clock_per_sm, void *stream);

/*
 * gemm_fma_rate_probe -- diagnostic: the FP32 FMA units' throughput per SM,
 * measured on an outer product in registers, for the instruction form an
 * FP32 GEMM can use: packed = 1, the two-wide FMA (__ffma2_rn, one FMA on
 * each of two lanes) with the same scalar in both lanes of one operand --
 * gemm_f32's form; packed = 0, scalar FMAs.  One CTA of 8 warps per SM
 * (gemm_f32's residency); each thread multiplies 8 values a_i by 8 values
 * b_j into 64 accumulators per step, a_i reused across consecutive
 * instructions, for `iters` steps (no memory traffic), timed with the SM
 * cycle counter; *fma_per_clock_per_sm receives the median over the SMs of
 * FMAs per clock (the nominal peak is 128 per SM per clock: 4 schedulers x 32
 * lanes).  gemm_f32's FFMA-pipe roofline is quoted against the nominal peak;
 * this measures how much of it each instruction form reaches at all.
 * Synchronous on `stream` (allocates and frees a small device buffer).
 * packed in {0, 1}, iters in 1..2^20 (a few thousand take about a
 * millisecond).  Returns GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_TIMEOUT (no
 * SM reported) or GEMM_ERR_CUDA.
 */
GEMM11_API int gemm_fma_rate_probe(int packed, int iters, double *fma_per_clock_per_sm, void *stream);

/*
 * gemm_tma_read_probe -- diagnostic: the operand feed of the tensor-core
 * plans, measured.  `clusters` clusters of 2 CTAs (one CTA per SM) each need
 * the same 32 KB per stage and stream `kblocks` stages through a
 * `stages`-deep ring of shared memory (TMA loads, mbarrier full/empty
 * handshake, every wait bounded; the consumer releases each stage as soon as
 * it lands).  The data is read as a K-major GEMM operand: a row-major FP16
 * matrix with 4096-element rows, 128-byte swizzle, each stage the 64-wide k
 * block of a 256-row panel as two boxes of 128 rows x 64 k; the stages walk
 * k, then the next panel, each cluster its own run of panels, wrapping
 * around a region of region_mb MB (region_mb / 2 panels) of a buffer the
 * probe allocates (24 MB stays in L2; 1024 MB streams from HBM).  multicast = 0: each CTA loads
 * both boxes itself; multicast = 1: CTA r loads box r once with cluster
 * multicast into both CTAs.  *bytes_per_clock_per_sm receives the median
 * over the CTAs of bytes received per SM clock (cycle counter around the
 * consumer's loop); *total_gbs the bytes all CTAs received over the launch's
 * CUDA-event time.  One warm-up launch precedes the timed one.  Synchronous
 * on `stream`.  clusters in 1..(SMs / 2), multicast in {0, 1}, stages in
 * 1..6, kblocks in 1..65536, region_mb in 2..4096.  Returns GEMM_OK,
 * GEMM_ERR_INVALID_ARG, GEMM_ERR_TIMEOUT (no CTA finished within the bounded
 * waits) or GEMM_ERR_CUDA.
 */
GEMM11_API int gemm_tma_read_probe(int clusters, int multicast, int stages, int kblocks, int region_mb,
                                   double *bytes_per_clock_per_sm, double *total_gbs, void *stream);

/*
 * Introspection for tests and benchmarks: the name of the kernel plan the
 * calling thread's last successful call used (static storage), and how many
 * kernels that call launched.
 */
GEMM11_API const char *gemm_last_plan(void);
GEMM11_API int gemm_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM11_H */
