// api.cu -- the C ABI of libgemm11.so: argument checks, degenerate shapes,
// dispatch to the FP32 / FP16 paths, status codes, the per-(device, stream)
// split-K scratch and the device watchdog word.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/gemm11.h"
#include "internal.h"
#include "ptx.cuh"

namespace gemm11 {

// One watchdog word per device (every device that loads the library holds a
// copy); kernels receive its address and OR kWatchdogTimeout into it.
__device__ unsigned g_watchdog_word;

namespace {

// One thread waits on an mbarrier that nothing ever arrives on, with the
// same bounded wait the GEMM pipelines use; when it gives up it records the
// timeout in the watchdog word exactly as they do.
__global__ void watchdog_probe_kernel(unsigned *err, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(err, kWatchdogTimeout);
}

// GEMM11_DEBUG builds: guard bands of kCanaryBytes before and after every
// library-owned scratch buffer, filled with kCanaryByte; every call checks
// them after its own work (canary_check_kernel) and reports a corrupted band.
constexpr size_t kCanaryBytes = 4096;
constexpr unsigned char kCanaryByte = 0xA5;
constexpr unsigned kCanaryWord = 0xA5A5A5A5u;

__global__ void canary_check_kernel(const unsigned *lo, const unsigned *hi, int words, unsigned *err) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x)
        if (lo[i] != kCanaryWord || hi[i] != kCanaryWord) atomicOr(err, kDebugCanaryFault);
}

// Test hook of debug builds: overwrite the first word of a guard band (memory
// that the library allocated, so the write is in bounds) to show the check
// catches it.
__global__ void canary_poke_kernel(unsigned *word) { *word = 0u; }

thread_local int t_last_cuda_error = 0;
thread_local const char *t_last_plan = "none";
thread_local int t_last_launches = 0;
thread_local char t_plan_buf[96];

// Record a finished call's plan for gemm_last_plan / gemm_last_launch_count.
void record_plan(const gemm11::CallInfo &info) {
    if (info.tuned) {
        std::snprintf(t_plan_buf, sizeof(t_plan_buf), "%s+tuned", info.plan);
        t_last_plan = t_plan_buf;
    } else {
        t_last_plan = info.plan;
    }
    t_last_launches = info.launches;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    int sm_count = 0;
    unsigned *watchdog = nullptr;
    cudaError_t init_error = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

struct ScratchEntry {
    float *partials = nullptr;
    size_t partial_floats = 0;
    unsigned *counters = nullptr;
    size_t ncounters = 0;
    float *operands = nullptr;
    size_t operand_floats = 0;
};
std::mutex g_scratch_mu;
std::map<std::pair<int, uintptr_t>, ScratchEntry> g_scratch;

// Library scratch allocation: plain cudaMalloc in release builds; debug
// builds put a filled guard band of kCanaryBytes on both sides and hand out
// the address past the first band.
cudaError_t scratch_alloc(void **user, size_t bytes) {
    if (!kDebugBuild) return cudaMalloc(user, bytes);
    unsigned char *raw = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&raw), bytes + 2 * kCanaryBytes);
    if (e != cudaSuccess) return e;
    e = cudaMemset(raw, kCanaryByte, kCanaryBytes);
    if (e == cudaSuccess) e = cudaMemset(raw + kCanaryBytes + bytes, kCanaryByte, kCanaryBytes);
    if (e != cudaSuccess) {
        cudaFree(raw);
        return e;
    }
    *user = raw + kCanaryBytes;
    return cudaSuccess;
}
void scratch_free(void *user) {
    if (!user) return;
    cudaFree(kDebugBuild ? static_cast<unsigned char *>(user) - kCanaryBytes : user);
}
// Enqueue the guard-band check of one buffer (debug builds).
cudaError_t check_bands(const void *user, size_t bytes, unsigned *err, cudaStream_t stream) {
    if (!user) return cudaSuccess;
    const unsigned char *u = static_cast<const unsigned char *>(user);
    canary_check_kernel<<<4, 256, 0, stream>>>(reinterpret_cast<const unsigned *>(u - kCanaryBytes),
                                               reinterpret_cast<const unsigned *>(u + bytes),
                                               static_cast<int>(kCanaryBytes / 4), err);
    return cudaPeekAtLastError();
}

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

DeviceState *device_state() {
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return nullptr;
    DeviceState &s = g_dev[d];
    std::call_once(s.once, [&s, d] {
        cudaError_t e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, d);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void **>(&s.watchdog), g_watchdog_word);
        s.init_error = e;
    });
    return &s;
}

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return GEMM_ERR_CUDA;
}

}  // namespace

int current_device_id() { return current_device(); }

int device_sm_count() {
    DeviceState *s = device_state();
    return (s && s->sm_count > 0) ? s->sm_count : 1;
}

unsigned *watchdog_word() {
    DeviceState *s = device_state();
    return s ? s->watchdog : nullptr;
}

cudaError_t acquire_scratch(cudaStream_t stream, size_t partial_floats, size_t ncounters, Scratch *out) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry &e = g_scratch[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (e.partial_floats < partial_floats) {
        // Work already queued on this stream may still use the old buffer.
        cudaError_t r = cudaStreamSynchronize(stream);
        if (r != cudaSuccess) return r;
        scratch_free(e.partials);
        e.partials = nullptr;
        e.partial_floats = 0;
        size_t want = partial_floats + partial_floats / 4;
        r = scratch_alloc(reinterpret_cast<void **>(&e.partials), want * sizeof(float));
        if (r != cudaSuccess) return r;
        e.partial_floats = want;
    }
    if (e.ncounters < ncounters) {
        cudaError_t r = cudaStreamSynchronize(stream);
        if (r != cudaSuccess) return r;
        scratch_free(e.counters);
        e.counters = nullptr;
        e.ncounters = 0;
        size_t want = ncounters < 1024 ? 1024 : ncounters + ncounters / 4;
        r = scratch_alloc(reinterpret_cast<void **>(&e.counters), want * sizeof(unsigned));
        if (r != cudaSuccess) return r;
        r = cudaMemset(e.counters, 0, want * sizeof(unsigned));
        if (r != cudaSuccess) return r;
        e.ncounters = want;
    }
    out->partials = e.partials;
    out->counters = e.counters;
    return cudaSuccess;
}

cudaError_t acquire_operand_scratch(cudaStream_t stream, size_t floats, float **out) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry &e = g_scratch[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (e.operand_floats < floats) {
        cudaError_t r = cudaStreamSynchronize(stream);  // queued work may still read the old buffer
        if (r != cudaSuccess) return r;
        scratch_free(e.operands);
        e.operands = nullptr;
        e.operand_floats = 0;
        r = scratch_alloc(reinterpret_cast<void **>(&e.operands), floats * sizeof(float));
        if (r != cudaSuccess) return r;
        e.operand_floats = floats;
    }
    *out = e.operands;
    return cudaSuccess;
}

size_t debug_shrink_c() {
    if (!kDebugBuild) return 0;
    const char *v = std::getenv("GEMM11_DEBUG_SHRINK_C");
    return v ? static_cast<size_t>(std::strtoull(v, nullptr, 10)) : 0;
}

namespace {

// Read and clear the current device's status word after synchronising
// `stream`; maps its bits to a status.  A non-zero word also resets the
// split-K arrival counters (a CTA that gave up may have left them non-zero).
int read_status_word(DeviceState *ds, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail_cuda(e);
    unsigned word = 0;
    e = cudaMemcpy(&word, ds->watchdog, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e);
    if (word == 0) return GEMM_OK;
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        for (auto &kv : g_scratch)
            if (kv.first.first == dev && kv.second.counters) {
                e = cudaMemset(kv.second.counters, 0, kv.second.ncounters * sizeof(unsigned));
                if (e != cudaSuccess) return fail_cuda(e);
            }
    }
    const unsigned zero = 0;
    e = cudaMemcpy(ds->watchdog, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e);
    return (word & (kDebugBoundsFault | kDebugCanaryFault)) ? GEMM_ERR_DEBUG_CHECK : GEMM_ERR_TIMEOUT;
}

// The end of every call that enqueued work: record its plan; GEMM11_DEBUG
// builds also check the guard bands of this stream's scratch, wait for the
// call's work and report what the device-side checks found ("start fully
// synchronous").
int finish_call(const CallInfo &info, cudaStream_t stream) {
    record_plan(info);
    if (!kDebugBuild) return GEMM_OK;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        auto it = g_scratch.find({dev, reinterpret_cast<uintptr_t>(stream)});
        if (it != g_scratch.end()) {
            ScratchEntry &se = it->second;
            const char *poke = std::getenv("GEMM11_DEBUG_POKE_CANARY");
            if (poke && poke[0] == '1' && se.partials) {
                canary_poke_kernel<<<1, 1, 0, stream>>>(reinterpret_cast<unsigned *>(se.partials + se.partial_floats));
            }
            cudaError_t e = check_bands(se.partials, se.partial_floats * sizeof(float), ds->watchdog, stream);
            if (e == cudaSuccess) e = check_bands(se.counters, se.ncounters * sizeof(unsigned), ds->watchdog, stream);
            if (e == cudaSuccess)
                e = check_bands(se.operands, se.operand_floats * sizeof(float), ds->watchdog, stream);
            if (e != cudaSuccess) return fail_cuda(e);
        }
    }
    return read_status_word(ds, stream);
}

}  // namespace
}  // namespace gemm11

using namespace gemm11;

// ------------------------------------------------------------------ tuning table
namespace {

struct TuneKey {
    int path, M, N, K;
    bool operator<(const TuneKey &o) const {
        if (path != o.path) return path < o.path;
        if (M != o.M) return M < o.M;
        if (N != o.N) return N < o.N;
        return K < o.K;
    }
};
std::mutex g_tune_mutex;
std::map<TuneKey, TunePlan> g_tune_table;
std::atomic<bool> g_tune_any{false};  // lets every call skip the lock while the table is empty

bool valid_tune_entry(const gemm_tune_entry &e) {
    if (e.M < 0 || e.N < 0 || e.K < 0 || e.splits < 0 || e.splits > 32) return false;
    if (e.path == GEMM_PATH_F32) return (e.variant == 1 && e.bn == 0) || (e.variant == 2 && e.bn == 0);
    if (e.path != GEMM_PATH_TC) return false;
    switch (e.variant) {
        case 1: return e.bn == 0 || e.bn == 256 || e.bn == 224 || e.bn == 192;
        case 2: return e.bn == 0 || e.bn == 256 || e.bn == 128;
        case 3: return e.bn == 0 || e.bn == 32 || e.bn == 64;
        case 4: return (e.bn == 0 || e.bn == 256 || e.bn == 192 || e.bn == 128) && (e.splits == 0 || (e.splits >= 2 && e.splits <= 8));
        default: return false;
    }
}

}  // namespace

namespace gemm11 {
bool tune_lookup(int path, int M, int N, int K, TunePlan *out) {
    if (!g_tune_any.load(std::memory_order_acquire)) return false;
    std::lock_guard<std::mutex> lock(g_tune_mutex);
    auto it = g_tune_table.find(TuneKey{path, M, N, K});
    if (it == g_tune_table.end()) return false;
    *out = it->second;
    return true;
}
}  // namespace gemm11

extern "C" {

int gemm_tune_set(const gemm_tune_entry *entries, int n) {
    if (n < 0 || (n > 0 && !entries)) return GEMM_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!valid_tune_entry(entries[i])) return GEMM_ERR_INVALID_ARG;
    std::map<TuneKey, TunePlan> table;
    for (int i = 0; i < n; ++i) {
        const gemm_tune_entry &e = entries[i];
        TunePlan tp;
        tp.variant = e.variant;
        tp.bn = e.bn;
        tp.splits = e.splits;
        table[TuneKey{e.path, e.M, e.N, e.K}] = tp;
    }
    std::lock_guard<std::mutex> lock(g_tune_mutex);
    g_tune_table.swap(table);
    g_tune_any.store(!g_tune_table.empty(), std::memory_order_release);
    return GEMM_OK;
}

int gemm_tune_get(gemm_tune_entry *out, int capacity) {
    std::lock_guard<std::mutex> lock(g_tune_mutex);
    int i = 0;
    for (const auto &kv : g_tune_table) {
        if (out && i < capacity) {
            gemm_tune_entry &e = out[i];
            e.path = kv.first.path;
            e.M = kv.first.M;
            e.N = kv.first.N;
            e.K = kv.first.K;
            e.variant = kv.second.variant;
            e.bn = kv.second.bn;
            e.splits = kv.second.splits;
        }
        ++i;
    }
    return i;
}


int gemm_f32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
             float *C, int ldc, void *stream) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) {
        t_last_plan = "noop_empty";
        t_last_launches = 0;
        return GEMM_OK;
    }
    if (!C) return GEMM_ERR_INVALID_ARG;
    const bool product = (K > 0) && (alpha != 0.f);
    if (product && (!A || !B)) return GEMM_ERR_INVALID_ARG;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CallInfo info;
    cudaError_t e = product ? run_gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s, &info)
                            : run_scale_c(M, N, beta, C, ldc, nullptr, 0, s, &info);
    if (e != cudaSuccess) return fail_cuda(e);
    return finish_call(info, s);
}

int gemm_f32_3xtf32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
                    float *C, int ldc, void *stream) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) {
        t_last_plan = "noop_empty";
        t_last_launches = 0;
        return GEMM_OK;
    }
    if (!C) return GEMM_ERR_INVALID_ARG;
    const bool product = (K > 0) && (alpha != 0.f);
    if (product && (!A || !B)) return GEMM_ERR_INVALID_ARG;
    // C is written by TMA stores: 16-byte aligned base and rows (a single row
    // has no row stride to align).
    if (product && (((reinterpret_cast<uintptr_t>(C) & 15u) != 0) || (M > 1 && (ldc % 4) != 0)))
        return GEMM_ERR_UNSUPPORTED;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CallInfo info;
    cudaError_t e = product ? run_gemm_f32_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s, &info)
                            : run_scale_c(M, N, beta, C, ldc, nullptr, 0, s, &info);
    if (e == cudaErrorNotSupported) return GEMM_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return fail_cuda(e);
    return finish_call(info, s);
}

}  // extern "C"

namespace {

bool valid_act(int act) { return act >= GEMM_ACT_NONE && act <= GEMM_ACT_GELU_TANH; }

// The tensor-core entry points (FP16 or BF16 operands, FP32 accumulate,
// FP32/FP16/BF16 output, fused epilogue, optional strided batch and
// transposed B) share validation and planning.
int gemm_tc_checked(const TcGemm &g, int ab_type, void *stream) {
    if (g.batch < 0 || g.M < 0 || g.N < 0 || g.K < 0) return GEMM_ERR_INVALID_ARG;
    if (!valid_act(g.act)) return GEMM_ERR_INVALID_ARG;
    if (ab_type != GEMM_DTYPE_F16 && ab_type != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
    if (g.c_type != GEMM_DTYPE_F32 && g.c_type != GEMM_DTYPE_F16 && g.c_type != GEMM_DTYPE_BF16)
        return GEMM_ERR_INVALID_ARG;
    if (g.b_trans != 0 && g.b_trans != 1) return GEMM_ERR_INVALID_ARG;
    if (g.batch == 0 || g.M == 0 || g.N == 0) {
        t_last_plan = "noop_empty";
        t_last_launches = 0;
        return GEMM_OK;
    }
    if (!g.C) return GEMM_ERR_INVALID_ARG;
    const long long mn = static_cast<long long>(g.M) * g.N;
    if (g.batch > 1 && (g.stride_a < 0 || g.stride_b < 0 || g.stride_c < mn)) return GEMM_ERR_INVALID_ARG;
    const bool product = (g.K > 0) && (g.alpha != 0.f);
    if (product && (!g.A || !g.B)) return GEMM_ERR_INVALID_ARG;
    // Tensor-map constraints: 16-byte aligned bases, row and matrix strides
    // (the epilogue-only path, alpha == 0 or K == 0, has none).
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (product) {
        const bool ok = (g.K % 8 == 0) && (g.N % 8 == 0) && al16(g.A) && al16(g.B) && al16(g.C) &&
                        (g.batch == 1 || (g.stride_a % 8 == 0 && g.stride_b % 8 == 0 && g.stride_c % 8 == 0));
        if (!ok) return GEMM_ERR_UNSUPPORTED;
    }
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CallInfo info;
    cudaError_t e;
    if (!product) {
        e = run_scale_c_batched(g.batch, g.M, g.N, g.beta, g.C, g.batch > 1 ? g.stride_c : mn, g.c_type, g.bias,
                                g.act, s, &info);
    } else {
        TcGemm gg = g;
        gg.bf16 = ab_type == GEMM_DTYPE_BF16;
        if (gg.batch == 1) gg.stride_a = gg.stride_b = 0, gg.stride_c = mn;
        e = run_gemm_f16(gg, s, &info);
        if (e == cudaErrorNotSupported) return GEMM_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return fail_cuda(e);
    return finish_call(info, s);
}

TcGemm tc_single(int M, int N, int K, float alpha, const void *A, const void *B, float beta, void *C, int c_type,
                 const float *bias, int act) {
    TcGemm g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.alpha = alpha;
    g.A = A;
    g.B = B;
    g.beta = beta;
    g.C = C;
    g.c_type = c_type;
    g.bias = bias;
    g.act = act;
    return g;
}

}  // namespace

extern "C" {

int gemm_f16_f32acc_epilogue(int M, int N, int K, float alpha, const void *A, const void *B, float beta, float *C,
                             const float *bias, int act, void *stream) {
    return gemm_tc_checked(tc_single(M, N, K, alpha, A, B, beta, C, GEMM_DTYPE_F32, bias, act), GEMM_DTYPE_F16,
                           stream);
}

int gemm_bf16_f32acc_epilogue(int M, int N, int K, float alpha, const void *A, const void *B, float beta,
                              float *C, const float *bias, int act, void *stream) {
    return gemm_tc_checked(tc_single(M, N, K, alpha, A, B, beta, C, GEMM_DTYPE_F32, bias, act), GEMM_DTYPE_BF16,
                           stream);
}

int gemm_tc_f32acc_epilogue(int M, int N, int K, float alpha, const void *A, const void *B, int ab_type, float beta,
                            void *C, int c_type, const float *bias, int act, void *stream) {
    return gemm_tc_checked(tc_single(M, N, K, alpha, A, B, beta, C, c_type, bias, act), ab_type, stream);
}

int gemm_tc_strided_batched(int batch, int M, int N, int K, float alpha, const void *A, long long stride_a,
                            const void *B, long long stride_b, int ab_type, int b_trans, float beta, void *C,
                            long long stride_c, int c_type, const float *bias, int act, void *stream) {
    TcGemm g = tc_single(M, N, K, alpha, A, B, beta, C, c_type, bias, act);
    g.batch = batch;
    g.stride_a = stride_a;
    g.stride_b = stride_b;
    g.stride_c = stride_c;
    g.b_trans = b_trans;
    return gemm_tc_checked(g, ab_type, stream);
}

int gemm_f16_f32acc_epilogue_noalloc(int M, int N, int K, float alpha, const void *A, const void *B, float beta,
                                     float *C, const float *bias, int act, void *stream) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (!valid_act(act)) return GEMM_ERR_INVALID_ARG;
    if (M > 64) return GEMM_ERR_UNSUPPORTED;  // whatever alpha, K or N: this entry point is for M <= 64
    if (M == 0 || N == 0) {
        t_last_plan = "noop_empty";
        t_last_launches = 0;
        return GEMM_OK;
    }
    if (!C) return GEMM_ERR_INVALID_ARG;
    const bool product = (K > 0) && (alpha != 0.f);
    if (product && (!A || !B)) return GEMM_ERR_INVALID_ARG;
    if (product) {
        const bool ok = (K % 8 == 0) && (N % 8 == 0) && ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(B) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
        if (!ok) return GEMM_ERR_UNSUPPORTED;
    }
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CallInfo info;
    cudaError_t e;
    if (!product) {
        e = run_scale_c(M, N, beta, C, N, bias, act, s, &info);
    } else {
        int reject = 0;
        e = run_gemm_f16_small_m_noalloc(M, N, K, alpha, A, B, beta, C, bias, act, s, &info, &reject);
        if (e == cudaErrorNotSupported) return GEMM_ERR_UNSUPPORTED;
        if (e == cudaSuccess && reject == 1) return GEMM_ERR_UNSUPPORTED;
        if (e == cudaSuccess && reject == 2) return GEMM_ERR_SCRATCH_LIMIT;
    }
    if (e != cudaSuccess) return fail_cuda(e);
    return finish_call(info, s);
}

const char *gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: arguments outside this path's constraints";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA runtime call failed";
        case GEMM_ERR_DEBUG_CHECK:
            return "GEMM_ERR_DEBUG_CHECK: a device-side check of a GEMM11_DEBUG build failed (index out of range or "
                   "a scratch guard band overwritten)";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a bounded in-kernel wait ran out";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "GEMM_ERR_SCRATCH_LIMIT: the shape needs more split-K scratch than the fixed no-allocation "
                   "buffer holds (4 MiB of partial tiles, 4096 counters)";
        default: return "unknown gemm status";
    }
}

int gemm_last_cuda_error(void) { return t_last_cuda_error; }

int gemm_debug_build(void) { return kDebugBuild ? 1 : 0; }

int gemm_check(void *stream) {
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    return read_status_word(ds, static_cast<cudaStream_t>(stream));
}

int gemm_watchdog_selftest(int wait_ms, void *stream) {
    if (wait_ms < 1 || wait_ms > 2000) return GEMM_ERR_INVALID_ARG;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    watchdog_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        ds->watchdog, static_cast<unsigned long long>(wait_ms) * 1000000ull);
    const cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_plan = "watchdog_probe";
    t_last_launches = 1;
    return GEMM_OK;
}

int gemm_pipeline_stall_selftest(int M, int N, int K, const void *A, const void *B, float *C, int wait_ms,
                                 void *stream) {
    if (wait_ms < 1 || wait_ms > 2000) return GEMM_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || !A || !B || !C) return GEMM_ERR_INVALID_ARG;
    const bool ok = (K % 8 == 0) && (N % 8 == 0) && ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) &&
                    ((reinterpret_cast<uintptr_t>(B) & 15u) == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
    if (!ok) return GEMM_ERR_UNSUPPORTED;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    const cudaError_t e = run_hgemm_stall_selftest(M, N, K, A, B, C, static_cast<unsigned long long>(wait_ms) * 1000000ull,
                                                   static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return GEMM_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_plan = "tc_128x128_stalled_producer";
    t_last_launches = 1;
    return GEMM_OK;
}

int gemm_fma_rate_probe(int packed, int iters, double *fma_per_clock_per_sm, void *stream) {
    if ((packed != 0 && packed != 1) || iters < 1 || iters > (1 << 20) || !fma_per_clock_per_sm)
        return GEMM_ERR_INVALID_ARG;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    const cudaError_t e = run_fma_rate_probe(packed != 0, iters, fma_per_clock_per_sm, static_cast<cudaStream_t>(stream));
    t_last_plan = packed ? "fma2_rate_probe" : "fma_rate_probe";
    t_last_launches = 1;
    if (e == cudaErrorLaunchTimeout) return GEMM_ERR_TIMEOUT;
    if (e != cudaSuccess) return fail_cuda(e);
    return GEMM_OK;
}

int gemm_tc_rate_probe(int iters, double *flop_per_clock_per_sm, void *stream) {
    if (iters < 1 || iters > (1 << 20) || !flop_per_clock_per_sm) return GEMM_ERR_INVALID_ARG;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    const cudaError_t e = run_tc_rate_probe(iters, flop_per_clock_per_sm, static_cast<cudaStream_t>(stream));
    t_last_plan = "tc_rate_probe";
    t_last_launches = 1;
    if (e == cudaErrorLaunchTimeout) return GEMM_ERR_TIMEOUT;
    if (e != cudaSuccess) return fail_cuda(e);
    return GEMM_OK;
}

int gemm_tma_read_probe(int clusters, int multicast, int stages, int kblocks, int region_mb,
                        double *bytes_per_clock_per_sm, double *total_gbs, void *stream) {
    if (clusters < 1 || (multicast != 0 && multicast != 1) || stages < 1 || stages > 6 || kblocks < 1 ||
        kblocks > (1 << 16) || region_mb < 2 || region_mb > 4096 || !bytes_per_clock_per_sm || !total_gbs)
        return GEMM_ERR_INVALID_ARG;
    DeviceState *ds = device_state();
    if (!ds) return fail_cuda(cudaErrorInvalidDevice);
    if (ds->init_error != cudaSuccess) return fail_cuda(ds->init_error);
    if (2 * clusters > device_sm_count()) return GEMM_ERR_INVALID_ARG;
    const cudaError_t e = run_tma_read_probe(clusters, multicast != 0, stages, kblocks, region_mb,
                                             bytes_per_clock_per_sm, total_gbs, static_cast<cudaStream_t>(stream));
    t_last_plan = multicast ? "tma_read_probe_multicast" : "tma_read_probe";
    t_last_launches = 2;
    if (e == cudaErrorLaunchTimeout) return GEMM_ERR_TIMEOUT;
    if (e != cudaSuccess) return fail_cuda(e);
    return GEMM_OK;
}

const char *gemm_last_plan(void) { return t_last_plan; }

int gemm_last_launch_count(void) { return t_last_launches; }

}  // extern "C"
