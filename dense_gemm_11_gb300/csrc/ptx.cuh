// ptx.cuh -- thin inline-PTX wrappers for sm_103a: cp.async, mbarrier, TMA
// (cp.async.bulk.tensor), tcgen05 (tensor memory + 5th-generation MMA), and
// the bounded wait used by every pipeline in this library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gemm11 {

// Bit set in the device watchdog word when a bounded wait gives up.
constexpr unsigned kWatchdogTimeout = 1u;

// GEMM11_DEBUG builds (compiled with -DGEMM11_DEBUG=1): device-side checks of
// the indices of global stores and of library scratch accesses.  A failing
// check sets kDebugBoundsFault in the same device status word and the access
// is skipped (nothing traps); kDebugCanaryFault marks a guard band around
// library scratch found overwritten.  Release builds compile the checks away.
#ifndef GEMM11_DEBUG
#define GEMM11_DEBUG 0
#endif
constexpr bool kDebugBuild = GEMM11_DEBUG != 0;
constexpr unsigned kDebugBoundsFault = 2u;
constexpr unsigned kDebugCanaryFault = 4u;

// True when the access may proceed: always in release builds; in debug
// builds only when `ok`, otherwise the fault is recorded in *err.
__device__ __forceinline__ bool debug_in_bounds(bool ok, unsigned *err) {
    if constexpr (kDebugBuild) {
        if (!ok) {
            if (err) atomicOr(err, kDebugBoundsFault);
            return false;
        }
    }
    return true;
}
// A single wait longer than this (nanoseconds of %globaltimer) is treated as
// a stalled pipeline.  No legitimate wait in these kernels comes close.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- epilogue activations
// 0 identity, 1 exact GELU x * Phi(x), 2 ReLU, 3 tanh-approximate GELU
// 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
//
// Both GELU forms are written with one exponential (__expf) and one
// approximate reciprocal (rcp.approx) instead of the library's erff / tanhf.
// Epilogue arithmetic slows the tensor-core pipeline beside it (the SM clock
// is higher, not lower, when it runs), so fewer instructions per element pay:
// FP16 4096 x 11008 x 4096 with exact GELU measured 295 us against 310 us
// with erff and 313 us with a correctly rounded reciprocal (identity: 268 us;
// same GB300, CUDA-graph replays).
//
// Exact GELU: Phi(x) = 1 - Q(x) for x >= 0 and Q(|x|) for x < 0, with the
// upper tail Q(x) = erfc(x / sqrt 2) / 2 taken from Abramowitz & Stegun,
// Handbook of Mathematical Functions, formula 7.1.26 (Hastings):
//   erfc(z) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) + e(z),
//   t = 1 / (1 + p z),  |e(z)| <= 1.5e-7 for z >= 0,
//   p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741,
//   -1.453152027, 1.061405429.
// So |GELU error| <= 0.75e-7 |x| plus FP32 rounding and the few-ulp errors
// of __expf and rcp.approx.
// 1 / x to about 1 ulp (PTX rcp.approx.ftz.f32; 1 / inf = 0).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float gelu_erf(float x) {
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = rcp_approx(fmaf(0.3275911f, z, 1.f));
    float poly = fmaf(1.061405429f, t, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    const float q = 0.5f * poly * t * __expf(-z * z);  // Q(|x|)
    return x * (x >= 0.f ? 1.f - q : q);
}
// tanh-approximate GELU through the identity 0.5 (1 + tanh u) = 1 / (1 + exp(-2u)):
// x / (1 + exp(-2u)), u = sqrt(2/pi) (x + 0.044715 x^3).  exp overflow
// (x very negative) gives x * 0 = -0, underflow x.
__device__ __forceinline__ float gelu_tanh(float x) {
    const float u = 0.79788456080286536f * fmaf(0.044715f * x, x * x, x);
    return x * rcp_approx(1.f + __expf(-2.f * u));
}
__device__ __forceinline__ float apply_activation(int act, float v) {
    switch (act) {
        case 1: return gelu_erf(v);
        case 2: return fmaxf(v, 0.f);
        case 3: return gelu_tanh(v);
        default: return v;
    }
}

// ---------------------------------------------------------------- output element types
// C of the tensor-core path is FP32, FP16 or BF16 (codes of the C ABI's
// gemm_dtype).  16-bit results are rounded once, to nearest even, from the
// FP32 epilogue value.
constexpr int kOutF32 = 0;
constexpr int kOutF16 = 1;
constexpr int kOutBF16 = 2;

__device__ __forceinline__ float load_out(const void *C, size_t idx, int type) {
    if (type == kOutF16) return __half2float(static_cast<const __half *>(C)[idx]);
    if (type == kOutBF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(C)[idx]);
    return static_cast<const float *>(C)[idx];
}

__device__ __forceinline__ void store_out(void *C, size_t idx, int type, float v) {
    if (type == kOutF16)
        static_cast<__half *>(C)[idx] = __float2half_rn(v);
    else if (type == kOutBF16)
        static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(C)[idx] = v;
}

// Two values rounded to a 16-bit type and packed low-first into 32 bits.
__device__ __forceinline__ uint32_t pack2_out16(float lo, float hi, int type) {
    if (type == kOutF16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// Eight packed 16-bit values -> floats.
__device__ __forceinline__ void unpack8_out16(const uint4 &w, int type, float *out) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (type == kOutF16) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        } else {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u[i]));
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
}

// ---------------------------------------------------------------- cp.async
// 16-byte copy global -> shared; src_bytes < 16 zero-fills the rest (0: all zero).
__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(src_bytes)
                 : "memory");
}
// 4-byte copy global -> shared; src_bytes 0 writes a zero.
__device__ __forceinline__ void cp_async_4(void *smem_dst, const void *gmem_src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait until the phase with the given parity has completed.  Bounded: gives
// up after limit_ns and returns false (the caller records the timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 255u) == 0u && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched with programmatic stream serialization may start while
// the previous kernel in the stream is still running.  pdl_wait blocks until
// that kernel has completed and its memory operations are visible (so it must
// come before this kernel's first global-memory access); pdl_launch_dependents
// lets the next such kernel be scheduled (it still waits in its own pdl_wait).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap *map, uint64_t *bar, void *smem_dst, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
// 3-D tiled load (x innermost, z = matrix index of a strided batch).
__device__ __forceinline__ void tma_load_3d(const CUtensorMap *map, uint64_t *bar, void *smem_dst, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// 3-D tiled store shared -> global (out-of-range parts of the box are clipped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *smem_src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// 2-D tiled store shared -> global (out-of-range parts of the box are clipped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// All but the most recent bulk group have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Make generic-proxy writes to shared memory visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
// Allocate `ncols` (power of two >= 32) tensor-memory columns; the base
// address is written to shared memory.  Warp-wide.
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D(tmem) (+)= A(smem desc) x B(smem desc), FP16 inputs, kind::f16.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 32 lanes x 32 columns of 32-bit: thread t gets lane (base + t), columns
// [col, col + 32) in r[0..31].
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// 16 columns: register r[j] = column base + j of this thread's lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- CTA pairs (clusters of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// All threads of all CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Wait for a phase of this CTA's mbarrier whose arrivals were released by
// other CTAs of the cluster (cluster-scope acquire).  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(a, parity)) return true;
        if ((it & 255u) == 0u && globaltimer_ns() - t0 > limit_ns) return false;
    }
}
// Load a float from the shared memory of a CTA of the cluster (address from mapa).
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_cluster_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}
// 2-D tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap *map, uint32_t mbar_cluster_addr, void *smem_dst,
                                                 int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster_addr), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(const CUtensorMap *map, uint32_t mbar_cluster_addr, void *smem_dst,
                                                 int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
        "%4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster_addr), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Pair MMA (issued by one thread of the even CTA): D rows 0..127 in this CTA's
// tensor memory, rows 128..255 in the peer's; A rows and B columns are split
// between the two CTAs' shared memory at the same offsets.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same pair MMA of kind::tf32: A and B tiles hold FP32 words of which the
// MMA uses the TF32 part (sign, 8 exponent bits, the top 10 mantissa bits);
// K = 8 per instruction (32 bytes of each row, as for kind::f16).
__device__ __forceinline__ void umma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// FP32 -> TF32, round to nearest (ties away from zero); the low 13 mantissa
// bits of the result are zero.
__device__ __forceinline__ float tf32_round(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
// Arrive once on the mbarrier at this offset in every CTA of `cta_mask` when
// all pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ---------------------------------------------------------------- UMMA descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), fixed version bits 46..48 = 0b001, base
// offset 0 (operand tiles are 1024-byte aligned), layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}
// Instruction descriptor for kind::f16: FP16 A and B, FP32 accumulator,
// a_mn/b_mn = operand stored MN-major (1) or K-major (0), shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                                  // D format: F32
           | (0u << 7) | (0u << 10)                   // A, B format: F16
           | (static_cast<uint32_t>(a_mn) << 15)      // A major
           | (static_cast<uint32_t>(b_mn) << 16)      // B major
           | (static_cast<uint32_t>(N >> 3) << 17)    // N >> 3
           | (static_cast<uint32_t>(M >> 4) << 24);   // M >> 4
}
// Operand-format bits for BF16 A and B (the same kind::f16 MMA; only the two
// 3-bit format fields change, F16 = 0, BF16 = 1).
constexpr uint32_t kIdescBf16Operands = (1u << 7) | (1u << 10);
// Operand-format bits for TF32 A and B (kind::tf32: format code 2 in both fields).
constexpr uint32_t kIdescTf32Operands = (2u << 7) | (2u << 10);

}  // namespace gemm11
