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
#include <algorithm>
#include <cstdint>

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

}  // namespace

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
