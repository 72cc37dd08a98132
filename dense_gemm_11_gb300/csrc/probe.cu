// probe.cu -- measured rates per SM: the tensor core's dense FP16/BF16 rate
// and the FP32 FMA units' rate for the two instruction forms an FP32 GEMM
// can use (packed FFMA2 and scalar FFMA).
//
// The FP16 path's roofline is quoted against two peaks: the measured cuBLAS
// bf16 throughput and a nominal dense peak, #SM x (FLOP per clock per SM) x
// clock.  The per-SM rate comes from this kernel rather than a data sheet:
// one CTA per SM, whose single MMA thread issues back-to-back
// tcgen05.mma.cta_group::1.kind::f16 instructions of shape 128 x 256 x 16
// (BF16 operands resident in shared memory, FP32 accumulator in tensor
// memory) and times them with the SM's cycle counter from the first issue to
// the completion of the last (tcgen05.commit on an mbarrier, a bounded wait).
// Nothing is loaded from global memory, so the figure is the tensor pipe's
// issue-limited throughput.
//
// The third probe measures the bytes a CTA receives per SM clock through the
// TMA unit (tma_read_probe_kernel), with and without cluster multicast: the
// operand feed that bounds the memory-bound tensor-core plans.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gemm11 {
namespace {

constexpr int kProbeM = 128, kProbeN = 256, kProbeK = 16;
constexpr int kProbeABytes = kProbeM * 128;  // 128 rows of 128 bytes (64 k, 128-byte swizzle)
constexpr int kProbeBBytes = kProbeN * 128;  // B stored N x K: 256 rows of 128 bytes
// Requested (not used) shared memory: more than half an SM's, so each SM
// holds one CTA and every CTA measures a whole tensor pipe.
constexpr int kProbeSmem = 128 * 1024;

__global__ void __launch_bounds__(128, 1) tc_rate_probe_kernel(int iters, long long *cycles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + kProbeABytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + kProbeBBytes);
    uint32_t *holder = reinterpret_cast<uint32_t *>(bar + 1);
    const int warp = threadIdx.x >> 5;
    // zero operands: the values do not change the rate, and the sums stay 0
    for (int i = threadIdx.x; i < (kProbeABytes + kProbeBBytes) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the generic-proxy writes, before the tensor core reads them
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbarrier_init();
    }
    if (warp == 0) {
        tmem_alloc(holder, kProbeN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    if (threadIdx.x == 0) {
        const uint64_t ad = umma_desc_sw128(smem_u32(sA), 16, 1024);
        const uint64_t bd = umma_desc_sw128(smem_u32(sB), 16, 1024);
        const uint32_t idesc = umma_idesc_f16_f32(kProbeM, kProbeN, 0, 0) | kIdescBf16Operands;
        const long long t0 = clock64();
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_f16(tmem, ad + 2u * kk, bd + 2u * kk, idesc, (i | kk) ? 1u : 0u);
        }
        umma_commit(bar);
        const bool ok = mbar_wait(bar, 0);
        const long long t1 = clock64();
        cycles[blockIdx.x] = ok ? t1 - t0 : -1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kProbeN);
    }
}

// FP32 FMA throughput of an outer product in registers: 8 warps per SM
// (two per scheduler, the SGEMM's residency; the CTA requests more than half
// an SM's shared memory, so no SM holds two), and per thread 8 values a_i
// times 8 values b_j into 64 accumulators per step, a_i reused across
// consecutive instructions as in the SGEMM's inner loop.  PACKED: 32 packed
// FMAs (__ffma2_rn) per step, (a_i, a_i) * (b_2jj, b_2jj+1), the SGEMM's form;
// otherwise 64 scalar fmaf.  No memory traffic inside the timed loop.  Each
// CTA times its loop with the SM cycle counter between two barriers.
constexpr int kFmaProbeThreads = 256;

template <bool PACKED>
__global__ void __launch_bounds__(kFmaProbeThreads, 1) fma_rate_probe_kernel(const float *in, int iters,
                                                                             long long *cycles, float *sink) {
    float a[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a[j] = in[j];
        b[j] = in[8 + j];
    }
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if constexpr (PACKED) {
                const float2 a2 = make_float2(a[i], a[i]);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float2 c = __ffma2_rn(a2, make_float2(b[2 * jj], b[2 * jj + 1]),
                                                make_float2(acc[i][2 * jj], acc[i][2 * jj + 1]));
                    acc[i][2 * jj] = c.x;
                    acc[i][2 * jj + 1] = c.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) s += acc[i][j];
    sink[blockIdx.x * kFmaProbeThreads + threadIdx.x] = s;  // keeps the chains live
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// Median over the SMs of work / cycles from a device array of per-SM cycle counts.
cudaError_t median_rate(const long long *d_cycles, int sms, double work, cudaStream_t stream, double *rate) {
    long long *h = new long long[sms];
    cudaError_t e = cudaMemcpyAsync(h, d_cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) {
        int n = 0;
        for (int i = 0; i < sms; ++i)
            if (h[i] > 0) h[n++] = h[i];
        if (n == 0) {
            e = cudaErrorLaunchTimeout;
        } else {
            std::nth_element(h, h + n / 2, h + n);
            *rate = work / static_cast<double>(h[n / 2]);
        }
    }
    delete[] h;
    return e;
}

// TMA read rate: clusters of 2 CTAs, one per SM; each CTA needs the same
// 32 KB per stage and streams `kblocks` stages through a `stages`-deep ring
// whose consumer releases each stage as soon as it lands.  The data is a
// K-major operand as the tensor-core plans read it: a row-major FP16 matrix
// with K = 4096 (8 KB rows), 128-byte swizzle; a stage is the k block
// (64 k, 128 bytes of each row) of a 256-row panel, as two boxes of 128 rows
// x 64 k; successive stages walk k, and after 64 k blocks the next panel.
// Each cluster reads its own run of panels (disjoint while the region holds
// them all: a large region streams from HBM); the panels wrap around a
// region of `panels` panels, so a small region stays in L2.  multicast = 0: each CTA loads both
// boxes itself; 1: CTA r loads box r with .multicast::cluster into both CTAs
// (every stage then waits for both CTAs to have released it).  The consumer
// thread times its loop with the SM cycle counter; every wait is bounded (a
// timeout leaves -1 for that CTA).
constexpr int kTmaProbeStageBytes = 32768;
constexpr int kTmaProbeK = 4096;                 // elements per row
constexpr int kTmaProbeRowBytes = kTmaProbeK * 2;
constexpr int kTmaProbeKBlocks = kTmaProbeK / 64;  // k blocks per panel

struct TmaProbeArgs {
    int kblocks, stages, multicast, panels;
    long long *cycles;
};

__device__ __forceinline__ void tma_load_2d_multicast(const CUtensorMap *map, uint64_t *bar, void *smem_dst, int x,
                                                      int y, uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, "
        "{%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "h"(cta_mask)
        : "memory");
}

__global__ void __launch_bounds__(64, 1) tma_read_probe_kernel(const __grid_constant__ CUtensorMap tm, TmaProbeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + 8;
    uint8_t *ring = smem + 1024;
    const uint32_t rank = cluster_ctarank();
    const int cid = static_cast<int>(blockIdx.x >> 1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], a.multicast ? 2 : 1);
        }
        fence_mbarrier_init();
    }
    cluster_sync();
    bool ok = true;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.kblocks && ok; ++i) {
            const int s = i % a.stages;
            if (i >= a.stages) ok = mbar_wait(&empty[s], ((i / a.stages) - 1) & 1);
            if (!ok) break;
            mbar_arrive_expect_tx(&full[s], kTmaProbeStageBytes);
            uint8_t *dst = ring + static_cast<size_t>(s) * kTmaProbeStageBytes;
            const int x = (i % kTmaProbeKBlocks) * 64;
            const int ppc = (a.kblocks + kTmaProbeKBlocks - 1) / kTmaProbeKBlocks;  // panels per cluster
            const int y0 = static_cast<int>((static_cast<long long>(cid) * ppc + i / kTmaProbeKBlocks) % a.panels) * 256;
            if (a.multicast) {
                tma_load_2d_multicast(&tm, &full[s], dst + rank * 16384, x, y0 + static_cast<int>(rank) * 128, 0x3);
            } else {
                tma_load_2d(&tm, &full[s], dst, x, y0);
                tma_load_2d(&tm, &full[s], dst + 16384, x, y0 + 128);
            }
        }
    } else if (threadIdx.x == 32) {
        const long long t0 = clock64();
        for (int i = 0; i < a.kblocks && ok; ++i) {
            const int s = i % a.stages;
            ok = mbar_wait(&full[s], (i / a.stages) & 1);
            if (!ok) break;
            mbar_arrive(&empty[s]);
            if (a.multicast) mbar_arrive_cluster(mapa_shared(smem_u32(&empty[s]), rank ^ 1u));
        }
        a.cycles[blockIdx.x] = ok ? clock64() - t0 : -1;
    }
    __syncthreads();
    cluster_sync();  // neither CTA leaves while its peer may still write or arrive into it
}

PFN_cuTensorMapEncodeTiled_v12000 probe_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

cudaError_t run_tma_read_probe(int clusters, bool multicast, int stages, int kblocks, int region_mb,
                               double *bytes_per_clock_per_sm, double *total_gbs, cudaStream_t stream) {
    auto enc = probe_encoder();
    if (!enc) return cudaErrorNotSupported;
    const int panels = region_mb / 2;  // 256 rows of 8 KB = 2 MB each
    const size_t region = static_cast<size_t>(panels) * 256 * kTmaProbeRowBytes;
    const int rows_region = panels * 256;  // every box [x, x + 64) x [y, y + 128) lies inside
    uint8_t *buf = nullptr;
    long long *d_cycles = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaMalloc(&buf, region);
    if (e == cudaSuccess) e = cudaMalloc(&d_cycles, sizeof(long long) * 2 * clusters);
    if (e == cudaSuccess) e = cudaMemsetAsync(buf, 0, region, stream);
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    CUtensorMap tm;
    if (e == cudaSuccess) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(kTmaProbeK), static_cast<cuuint64_t>(rows_region)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(kTmaProbeRowBytes)};
        cuuint32_t box[2] = {64, 128}, estr[2] = {1, 1};
        if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, buf, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            e = cudaErrorInvalidValue;
    }
    // the opt-in is made once per device, for the deepest ring (6 stages)
    const int smem = std::max(2048 + stages * kTmaProbeStageBytes, kProbeSmem);
    static unsigned long long smem_set = 0;
    if (e == cudaSuccess) e = ensure_dynamic_smem(tma_read_probe_kernel, 2048 + 6 * kTmaProbeStageBytes, smem_set);
    if (e == cudaSuccess) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * clusters, 1, 1);
        cfg.blockDim = dim3(64, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        TmaProbeArgs args{kblocks, stages, multicast ? 1 : 0, panels, d_cycles};
        // one warm-up launch (a small region is then resident in L2), one timed
        e = cudaLaunchKernelEx(&cfg, tma_read_probe_kernel, tm, args);
        if (e == cudaSuccess) e = cudaEventRecord(e0, stream);
        if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, tma_read_probe_kernel, tm, args);
        if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    }
    if (e == cudaSuccess) {
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, e0, e1);
        if (e == cudaSuccess) {
            const double per_cta = static_cast<double>(kblocks) * kTmaProbeStageBytes;
            *total_gbs = 2.0 * clusters * per_cta / (static_cast<double>(ms) * 1e6);
            e = median_rate(d_cycles, 2 * clusters, per_cta, stream, bytes_per_clock_per_sm);
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(d_cycles);
    cudaFree(buf);
    return e;
}

cudaError_t run_fma_rate_probe(bool packed, int iters, double *fma_per_clock_per_sm, cudaStream_t stream) {
    const int sms = device_sm_count();
    long long *d_cycles = nullptr;
    float *d_buf = nullptr;
    cudaError_t e = cudaMalloc(&d_cycles, sizeof(long long) * sms);
    if (e != cudaSuccess) return e;
    e = cudaMalloc(&d_buf, sizeof(float) * (32 + static_cast<size_t>(sms) * kFmaProbeThreads));
    if (e == cudaSuccess) e = cudaMemsetAsync(d_buf, 0, sizeof(float) * 32, stream);
    if (e == cudaSuccess) {
        static unsigned long long smem_set_packed = 0, smem_set_scalar = 0;
        e = packed ? ensure_dynamic_smem(fma_rate_probe_kernel<true>, kProbeSmem, smem_set_packed)
                   : ensure_dynamic_smem(fma_rate_probe_kernel<false>, kProbeSmem, smem_set_scalar);
        if (e == cudaSuccess) {
            if (packed)
                fma_rate_probe_kernel<true><<<sms, kFmaProbeThreads, kProbeSmem, stream>>>(d_buf, iters, d_cycles,
                                                                                          d_buf + 32);
            else
                fma_rate_probe_kernel<false><<<sms, kFmaProbeThreads, kProbeSmem, stream>>>(d_buf, iters, d_cycles,
                                                                                           d_buf + 32);
            e = cudaPeekAtLastError();
        }
    }
    if (e == cudaSuccess) {
        const double fma = 64.0 * kFmaProbeThreads * static_cast<double>(iters);
        e = median_rate(d_cycles, sms, fma, stream, fma_per_clock_per_sm);
    }
    cudaFree(d_buf);
    cudaFree(d_cycles);
    return e;
}

cudaError_t run_tc_rate_probe(int iters, double *flop_per_clock_per_sm, cudaStream_t stream) {
    const int sms = device_sm_count();
    static unsigned long long smem_set = 0;
    cudaError_t e = ensure_dynamic_smem(tc_rate_probe_kernel, kProbeSmem, smem_set);
    if (e != cudaSuccess) return e;
    long long *d_cycles = nullptr;
    e = cudaMalloc(&d_cycles, sizeof(long long) * sms);
    if (e != cudaSuccess) return e;
    tc_rate_probe_kernel<<<sms, 128, kProbeSmem, stream>>>(iters, d_cycles);
    e = cudaPeekAtLastError();
    // the median over the SMs of FLOP per clock
    if (e == cudaSuccess)
        e = median_rate(d_cycles, sms, 2.0 * kProbeM * kProbeN * kProbeK * 4.0 * iters, stream, flop_per_clock_per_sm);
    cudaFree(d_cycles);
    return e;
}

}  // namespace gemm11
