// probe.cu -- the tensor core's dense rate per SM, measured.
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

}  // namespace

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
    long long *h = new long long[sms];
    if (e == cudaSuccess) e = cudaMemcpyAsync(h, d_cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    cudaFree(d_cycles);
    if (e == cudaSuccess) {
        // the median over the SMs of FLOP per clock
        const double flop = 2.0 * kProbeM * kProbeN * kProbeK * 4.0 * iters;
        int n = 0;
        for (int i = 0; i < sms; ++i)
            if (h[i] > 0) h[n++] = h[i];
        if (n == 0) {
            e = cudaErrorLaunchTimeout;
        } else {
            std::nth_element(h, h + n / 2, h + n);
            *flop_per_clock_per_sm = flop / static_cast<double>(h[n / 2]);
        }
    }
    delete[] h;
    return e;
}

}  // namespace gemm11
