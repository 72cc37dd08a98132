// sgemm.cu -- true-FP32 GEMM on the CUDA cores (FFMA), sm_103a.
//
//   C = alpha * A x B + beta * C, row-major, any shape, any leading dimension
//   ("SGEMM优化，从naive到warptiling", section 项目概况 / 问题与估算).
//
// Design (GB300-first; the pages' RTX 3090 / A100 kernels are prior art):
//  * block -> warp -> thread tiling: a CTA owns a BM x BN tile of C, each warp
//    a 64 x (4*TN) sub-tile, each thread TM x TN = 8 x 16 accumulators, the
//    three-level hierarchy of the warptiling kernel (section k10) sized so
//    that 6 shared-memory vector loads feed 128 FFMAs per k step;
//  * A stays K-major in shared memory (the layout the global rows already
//    have) and the inner loop reads 4 consecutive k of a row with one 128-bit
//    load ("第 11 章 Tiled GEMM", section 11.6, k unrolled by four); the
//    16-byte chunks of each 128-byte A row are XOR-swizzled by (row mod 8)
//    so that the 8 rows a warp reads at once hit 8 different bank groups
//    (section 11.5.2 derives the same XOR map for its tile);
//  * STAGES-deep cp.async ring, one __syncthreads per 32-wide k slice, so
//    global loads overlap the FFMA work (section 11.4, double buffer + async
//    copy, generalised to more stages);
//  * loads past M, N or K are zero-filled by cp.async's source size, the
//    grid is rounded up and the store is guarded (section 11.3's edge rule),
//    so no shape needs padding; 16-byte copies when A and B rows are 16-byte
//    aligned, 4-byte copies otherwise (lda = 4099 and the like);
//  * the inner product step uses packed FP32 FMAs (__ffma2_rn: two
//    independent fmaf, one rounding each, so results are bit-identical to
//    scalar FFMA) -- half the issue slots for the same FP32 work;
//  * large problems run one persistent CTA per SM: whole tiles round-robin,
//    and the tiles of the last partial wave are shared out by k slices
//    (stream-K) so that all SMs finish together; small problems split K
//    across CTAs.  Either way partial tiles go to a library-owned scratch
//    buffer and the last CTA to finish a tile (atomic arrival count) adds
//    them in k order -- deterministic, and no CTA ever waits for another;
//  * M == 1 and N == 1 are matrix-vector products bound by HBM; they use
//    their own streaming kernels ("第24讲 ... GEMM 分块与 Tensor Core 思维",
//    section 8.3 question 2 discusses these GEMV-like shapes).
#include <algorithm>
#include <cstdint>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace gemm11 {
namespace {

constexpr int kBK = 32;  // k slice per pipeline stage (one 128-byte A row)

struct SgemmArgs {
    int M, N, K;
    float alpha, beta;
    const float *A;
    const float *B;
    float *C;
    int lda, ldb, ldc;
    int tiles_m, tiles_n;
    int splits;      // K splits (grid mode: blockIdx.y)
    int persistent;  // 1: one CTA per SM, stream-K tail + data-parallel tiles
    int dp_tiles;    // persistent: tiles done whole, round-robin
    int sk_tiles;    // persistent: tiles shared out by k slices
    int grid_ctas;   // persistent: CTAs launched
    int c_vec;       // C rows 16-byte aligned
    float *ws;
    unsigned *counters;
#if GEMM11_DEBUG
    // GEMM11_DEBUG builds only (0 = unchecked): elements of C from this
    // argument block's C pointer, floats of ws; err receives the fault bit.
    // Release builds leave the fields out: the persistent kernel sits at its
    // register limit, and a larger argument block alone moved it to spilling.
    size_t c_extent, ws_floats;
    unsigned *err;
#endif
};

// The debug fields, as constants in release builds.
__host__ __device__ __forceinline__ size_t sg_c_extent(const SgemmArgs &p) {
#if GEMM11_DEBUG
    return p.c_extent;
#else
    (void)p;
    return 0;
#endif
}
__host__ __device__ __forceinline__ size_t sg_ws_floats(const SgemmArgs &p) {
#if GEMM11_DEBUG
    return p.ws_floats;
#else
    (void)p;
    return 0;
#endif
}
__host__ __device__ __forceinline__ unsigned *sg_err(const SgemmArgs &p) {
#if GEMM11_DEBUG
    return p.err;
#else
    (void)p;
    return nullptr;
#endif
}
// Host: set the debug fields (no-op in release builds).
inline void sg_set_debug(SgemmArgs &a, size_t c_extent, size_t ws_floats, unsigned *err) {
#if GEMM11_DEBUG
    a.c_extent = c_extent;
    a.ws_floats = ws_floats;
    a.err = err;
#else
    (void)a, (void)c_extent, (void)ws_floats, (void)err;
#endif
}

__device__ __forceinline__ int ctaid_x() {
    int v;
    asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(v));
    return v;
}
__device__ __forceinline__ int ctaid_y() {
    int v;
    asm volatile("mov.u32 %0, %%ctaid.y;" : "=r"(v));
    return v;
}

__device__ __forceinline__ float f4get(const float4 &v, int q) {
    return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// KG > 1: the CTA holds KG groups of WARPS_M x WARPS_N warps that share one
// tile; each pipeline stage carries KG consecutive 32-wide k slices and
// group g takes slice g of every stage, so a tile's K is split among the
// CTA's own warps (a small problem with few tiles still gives each scheduler
// several warps).  The groups' partial tiles are added in shared memory,
// groups in k order, before the epilogue.
template <int BM, int BN, int WARPS_M, int WARPS_N, int TM, int TN, int STAGES, bool VEC, int KG = 1>
struct SgemmTile {
    static constexpr int kGroupThreads = WARPS_M * WARPS_N * 32;  // one k group
    static constexpr int kThreads = kGroupThreads * KG;
    static constexpr int kWM = 8 * TM;  // 8 lanes down M, TM rows each (8 apart)
    static constexpr int kWN = 4 * TN;  // 4 lanes across N, TN/4 float4 each (16 apart)
    static constexpr int kAStage = BM * kBK * KG;
    static constexpr int kBStage = kBK * BN * KG;
    static constexpr int kSmemBytes = STAGES * (kAStage + kBStage) * 4;
    static_assert(BM == WARPS_M * kWM && BN == WARPS_N * kWN, "tile does not match warp layout");
    static_assert(TN % 4 == 0, "TN must be a multiple of 4");
    static_assert((BM * kBK / 4) % kGroupThreads == 0 && (kBK * BN / 4) % kGroupThreads == 0, "load split");
    static_assert(KG == 1 || (KG - 1) * BM * BN * 4 <= kSmemBytes, "the groups' partial tiles fit in the ring");
};

template <int BM, int BN, int WARPS_M, int WARPS_N, int TM, int TN, int STAGES, bool VEC, bool PERSIST, int KG = 1>
__global__ void __launch_bounds__(WARPS_M *WARPS_N * 32 * KG,
                                  (WARPS_M * WARPS_N * 32 * KG <= 128) ? 2
                                  : KG > 1                            ? 512 / (WARPS_M * WARPS_N * 32 * KG)
                                                                      : 1)
    sgemm_tiled_kernel(const SgemmArgs p) {
    using T = SgemmTile<BM, BN, WARPS_M, WARPS_N, TM, TN, STAGES, VEC, KG>;
    static_assert(KG == 1 || !PERSIST, "k groups: grid mode only");
    // Loads and compute below are per k group: kThreads threads of group g
    // copy and multiply the group's own 32-wide slice of each stage.
    constexpr int kThreads = T::kGroupThreads;
    extern __shared__ __align__(128) float smem[];
    __shared__ int s_last;
    const int g = KG > 1 ? static_cast<int>(threadIdx.x) / kThreads : 0;
    float *As = smem + g * (BM * kBK);
    float *Bs = smem + STAGES * T::kAStage + g * (kBK * BN);

    const int tid = KG > 1 ? static_cast<int>(threadIdx.x) % kThreads : static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int wm = warp / WARPS_N, wn = warp % WARPS_N;
    const int lm = lane & 7, ln = lane >> 3;
    const int M = p.M, N = p.N, K = p.K;
    const int KT = (K + kBK * KG - 1) / (kBK * KG);  // pipeline stages of KG k slices

    // Per-thread copy coordinates.  A: 8 threads per 128-byte row, rows
    // kARowStep apart; B: BN/4 threads per row, rows kBRowStep apart.
    constexpr int kARowStep = kThreads / 8;
    constexpr int kBChunks = BN / 4;
    constexpr int kBRowStep = kThreads / kBChunks;
    const int a_row = tid >> 3, a_kc = tid & 7;
    const int b_kr = tid / kBChunks, b_nc = tid % kBChunks;
    const uint32_t a_dst0 = smem_u32(As) + (a_row * kBK + ((a_kc ^ (a_row & 7)) << 2)) * 4;
    const uint32_t b_dst0 = smem_u32(Bs) + (b_kr * BN + b_nc * 4) * 4;

    float acc[TM][TN];

    // Grouped raster: 8 M-tiles share each sweep over N so that concurrently
    // resident CTAs reuse the same A and B panels from L2.
    auto tile_origin = [&](int t, int &m0, int &n0) {
        const int group_tiles = 8 * p.tiles_n;
        const int first_m = (t / group_tiles) * 8;
        const int gsz = min(p.tiles_m - first_m, 8);
        m0 = (first_m + (t % group_tiles) % gsz) * BM;
        n0 = ((t % group_tiles) / gsz) * BN;
    };

    // acc = sum over k slices [kt0, kt1) of the tile at (m0, n0).
    auto mainloop = [&](int m0, int n0, int kt0, int kt1) {
        const int nkt = kt1 - kt0;
        const bool full_mn = (m0 + BM <= M) && (n0 + BN <= N);
        const float *a_src = p.A + static_cast<size_t>(m0 + a_row) * p.lda + a_kc * 4;
        const float *b_src = p.B + static_cast<size_t>(b_kr) * p.ldb + n0 + b_nc * 4;

        auto load_stage = [&](int stage, int kt) {
            const int k0 = (kt * KG + g) * kBK;
            if constexpr (VEC) {
                if (full_mn && k0 + kBK <= K) {
                    // interior slice: every copy is a full, in-bounds 16-byte chunk
#pragma unroll
                    for (int it = 0; it < BM * kBK / 4 / kThreads; ++it)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                                         a_dst0 + (stage * T::kAStage + it * kARowStep * kBK) * 4),
                                     "l"(a_src + static_cast<size_t>(it) * kARowStep * p.lda + k0)
                                     : "memory");
#pragma unroll
                    for (int it = 0; it < kBK * BN / 4 / kThreads; ++it)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                                         b_dst0 + (stage * T::kBStage + it * kBRowStep * BN) * 4),
                                     "l"(b_src + static_cast<size_t>(k0 + it * kBRowStep) * p.ldb)
                                     : "memory");
                    return;
                }
            }
            float *as = As + stage * T::kAStage;
            float *bs = Bs + stage * T::kBStage;
            if constexpr (VEC) {
#pragma unroll
                for (int it = 0; it < BM * kBK / 4 / kThreads; ++it) {
                    const int c = tid + it * kThreads;
                    const int row = c >> 3, kc = c & 7;
                    const int gm = m0 + row, gk = k0 + kc * 4;
                    int bytes = 0;
                    const float *src = p.A;
                    if (gm < M && gk < K) {
                        bytes = min(K - gk, 4) * 4;
                        src = p.A + static_cast<size_t>(gm) * p.lda + gk;
                    }
                    cp_async_16(as + row * kBK + ((kc ^ (row & 7)) << 2), src, bytes);
                }
#pragma unroll
                for (int it = 0; it < kBK * BN / 4 / kThreads; ++it) {
                    const int c = tid + it * kThreads;
                    const int kr = c / (BN / 4), nc = c % (BN / 4);
                    const int gk = k0 + kr, gn = n0 + nc * 4;
                    int bytes = 0;
                    const float *src = p.B;
                    if (gk < K && gn < N) {
                        bytes = min(N - gn, 4) * 4;
                        src = p.B + static_cast<size_t>(gk) * p.ldb + gn;
                    }
                    cp_async_16(bs + kr * BN + nc * 4, src, bytes);
                }
            } else {
                if (full_mn && k0 + kBK <= K) {
                    // interior slice, 4-byte copies: thread tid copies column
                    // (tid & 31) of rows (tid >> 5) + it * kThreads / 32 of A, and
                    // column tid of rows it * kThreads / BN of B (all in bounds)
                    constexpr int kARows = kThreads / 32;
                    const int ak = tid & 31, ar = tid >> 5;
                    const float *asrc = p.A + static_cast<size_t>(m0 + ar) * p.lda + k0 + ak;
#pragma unroll 4
                    for (int it = 0; it < BM * kBK / kThreads; ++it) {
                        const int row = ar + it * kARows;
                        cp_async_4(as + row * kBK + (((ak >> 2) ^ (row & 7)) << 2) + (ak & 3),
                                   asrc + static_cast<size_t>(it) * kARows * p.lda, 4);
                    }
                    constexpr int kBRows = kThreads / BN;
                    const int bn = tid % BN, br = tid / BN;
                    const float *bsrc = p.B + static_cast<size_t>(k0 + br) * p.ldb + n0 + bn;
                    float *bdst = bs + br * BN + bn;
#pragma unroll 4
                    for (int it = 0; it < kBK * BN / kThreads; ++it)
                        cp_async_4(bdst + it * kBRows * BN, bsrc + static_cast<size_t>(it) * kBRows * p.ldb, 4);
                    return;
                }
#pragma unroll 4
                for (int it = 0; it < BM * kBK / kThreads; ++it) {
                    const int e = tid + it * kThreads;
                    const int row = e >> 5, k = e & 31;
                    const int gm = m0 + row, gk = k0 + k;
                    const bool ok = gm < M && gk < K;
                    const float *src = ok ? p.A + static_cast<size_t>(gm) * p.lda + gk : p.A;
                    cp_async_4(as + row * kBK + ((((k >> 2) ^ (row & 7))) << 2) + (k & 3), src, ok ? 4 : 0);
                }
#pragma unroll 4
                for (int it = 0; it < kBK * BN / kThreads; ++it) {
                    const int e = tid + it * kThreads;
                    const int kr = e / BN, n = e % BN;
                    const int gk = k0 + kr, gn = n0 + n;
                    const bool ok = gk < K && gn < N;
                    const float *src = ok ? p.B + static_cast<size_t>(gk) * p.ldb + gn : p.B;
                    cp_async_4(bs + kr * BN + n, src, ok ? 4 : 0);
                }
            }
        };

#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

        __syncthreads();  // the previous work item may still be reading the ring
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s) {
            if (s < nkt) load_stage(s, kt0 + s);
            cp_async_commit();
        }
        for (int it = 0; it < nkt; ++it) {
            // GEMM11_DEBUG builds wait for every copy in flight ("start fully
            // synchronous"): the ring still prefetches, but no stage is read
            // while any copy is outstanding.
            cp_async_wait<kDebugBuild ? 0 : STAGES - 2>();
            __syncthreads();
            const int nxt = it + STAGES - 1;
            if (nxt < nkt) load_stage(nxt % STAGES, kt0 + nxt);
            cp_async_commit();

            const int s = it % STAGES;
            const float *as = As + s * T::kAStage + (wm * T::kWM + lm) * kBK;
            const float *bs = Bs + s * T::kBStage + wn * T::kWN + ln * 4;
#pragma unroll
            for (int kg = 0; kg < kBK / 4; ++kg) {
                float4 a[TM];
                const int sw = (kg ^ lm) << 2;  // row & 7 == lm for every row this thread reads
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = *reinterpret_cast<const float4 *>(as + i * 8 * kBK + sw);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 b[TN / 4];
#pragma unroll
                    for (int jj = 0; jj < TN / 4; ++jj)
                        b[jj] = *reinterpret_cast<const float4 *>(bs + (kg * 4 + q) * BN + jj * 16);
                    // Outer product with packed FP32 FMAs: each __ffma2_rn is two
                    // independent fmaf (one rounding each), acc[i][j] += a_i * b_j.
#pragma unroll
                    for (int i = 0; i < TM; ++i) {
                        const float av = f4get(a[i], q);
                        const float2 a2 = make_float2(av, av);
#pragma unroll
                        for (int jj = 0; jj < TN / 4; ++jj) {
                            float2 c0 = make_float2(acc[i][jj * 4], acc[i][jj * 4 + 1]);
                            float2 c1 = make_float2(acc[i][jj * 4 + 2], acc[i][jj * 4 + 3]);
                            c0 = __ffma2_rn(a2, make_float2(b[jj].x, b[jj].y), c0);
                            c1 = __ffma2_rn(a2, make_float2(b[jj].z, b[jj].w), c1);
                            acc[i][jj * 4] = c0.x;
                            acc[i][jj * 4 + 1] = c0.y;
                            acc[i][jj * 4 + 2] = c1.x;
                            acc[i][jj * 4 + 3] = c1.y;
                        }
                    }
                }
            }
        }
        cp_async_wait<0>();
        if constexpr (KG > 1) {
            // Add the groups' partial tiles, in k order, into group 0's
            // registers; the ring is free once every group has left the loop.
            const int r_base = wm * T::kWM + lm, c_base = wn * T::kWN + ln * 4;
            __syncthreads();
            if (g > 0) {
                float *red = smem + (g - 1) * (BM * BN);
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int jj = 0; jj < TN / 4; ++jj)
                        *reinterpret_cast<float4 *>(red + (r_base + 8 * i) * BN + c_base + 16 * jj) =
                            make_float4(acc[i][jj * 4], acc[i][jj * 4 + 1], acc[i][jj * 4 + 2], acc[i][jj * 4 + 3]);
            }
            __syncthreads();
            if (g == 0) {
#pragma unroll 1
                for (int gg = 1; gg < KG; ++gg) {
                    const float *red = smem + (gg - 1) * (BM * BN);
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int jj = 0; jj < TN / 4; ++jj) {
                            const float4 v =
                                *reinterpret_cast<const float4 *>(red + (r_base + 8 * i) * BN + c_base + 16 * jj);
                            acc[i][jj * 4] += v.x;
                            acc[i][jj * 4 + 1] += v.y;
                            acc[i][jj * 4 + 2] += v.z;
                            acc[i][jj * 4 + 3] += v.w;
                        }
                }
            }
            __syncthreads();  // the next use of the ring overwrites the partials
        }
    };

    const int r_base = wm * T::kWM + lm;  // tile-local row of acc[0][*]
    const int c_base = wn * T::kWN + ln * 4;

    // Epilogue: C = alpha * acc + beta * C (C not read when beta == 0).
    auto epilogue = [&](int m0, int n0) {
        const float alpha = p.alpha, beta = p.beta;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int gr = m0 + r_base + 8 * i;
            if (gr >= M) continue;
            float *crow = p.C + static_cast<size_t>(gr) * p.ldc;
#pragma unroll
            for (int jj = 0; jj < TN / 4; ++jj) {
                const int gc = n0 + c_base + 16 * jj;
                const size_t ci = static_cast<size_t>(gr) * p.ldc + gc;
                if (p.c_vec && gc + 3 < N) {
                    if (!debug_in_bounds(sg_c_extent(p) == 0 || ci + 4 <= sg_c_extent(p), sg_err(p))) continue;
                    float4 v = make_float4(alpha * acc[i][jj * 4], alpha * acc[i][jj * 4 + 1],
                                           alpha * acc[i][jj * 4 + 2], alpha * acc[i][jj * 4 + 3]);
                    if (beta != 0.f) {
                        const float4 o = *reinterpret_cast<const float4 *>(crow + gc);
                        v.x = fmaf(beta, o.x, v.x);
                        v.y = fmaf(beta, o.y, v.y);
                        v.z = fmaf(beta, o.z, v.z);
                        v.w = fmaf(beta, o.w, v.w);
                    }
                    *reinterpret_cast<float4 *>(crow + gc) = v;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (gc + e < N && debug_in_bounds(sg_c_extent(p) == 0 || ci + e < sg_c_extent(p), sg_err(p))) {
                            float v = alpha * acc[i][jj * 4 + e];
                            if (beta != 0.f) v = fmaf(beta, crow[gc + e], v);
                            crow[gc + e] = v;
                        }
                    }
                }
            }
        }
    };

    // A partial tile's scratch slot lies inside the scratch (debug builds check).
    auto slot_ok = [&](const float *slot) {
        return debug_in_bounds(sg_ws_floats(p) == 0 || static_cast<size_t>(slot - p.ws) + BM * BN <= sg_ws_floats(p),
                               sg_err(p));
    };
    // Raw partial tile -> scratch slot (tile-local [BM][BN], row-major).
    auto store_partial = [&](float *slot) {
        if (!slot_ok(slot)) return;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int jj = 0; jj < TN / 4; ++jj)
                *reinterpret_cast<float4 *>(slot + (r_base + 8 * i) * BN + c_base + 16 * jj) =
                    make_float4(acc[i][jj * 4], acc[i][jj * 4 + 1], acc[i][jj * 4 + 2], acc[i][jj * 4 + 3]);
    };
    // acc += slot (L2 reads: the slot was written by another CTA).
    auto add_partial = [&](const float *slot, bool first) {
        if (!slot_ok(slot)) return;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int jj = 0; jj < TN / 4; ++jj) {
                const float4 v =
                    __ldcg(reinterpret_cast<const float4 *>(slot + (r_base + 8 * i) * BN + c_base + 16 * jj));
                if (first) {
                    acc[i][jj * 4] = v.x;
                    acc[i][jj * 4 + 1] = v.y;
                    acc[i][jj * 4 + 2] = v.z;
                    acc[i][jj * 4 + 3] = v.w;
                } else {
                    acc[i][jj * 4] += v.x;
                    acc[i][jj * 4 + 1] += v.y;
                    acc[i][jj * 4 + 2] += v.z;
                    acc[i][jj * 4 + 3] += v.w;
                }
            }
    };
    // Arrival on a tile's counter; true for the CTA that completes the tile.
    auto arrive_last = [&](unsigned *counter, unsigned arrivals) -> bool {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = (atomicAdd(counter, 1u) == arrivals - 1u);
        __syncthreads();
        const bool last = s_last != 0;
        if (last) __threadfence();
        return last;
    };

    if constexpr (!PERSIST) {
        // One tile per CTA (blockIdx.x), K split blockIdx.y ways.
        const int tile = blockIdx.x;
        int m0, n0;
        tile_origin(tile, m0, n0);
        const int split = blockIdx.y;
        const int kt0 = static_cast<int>(static_cast<long long>(KT) * split / p.splits);
        const int kt1 = static_cast<int>(static_cast<long long>(KT) * (split + 1) / p.splits);
        mainloop(m0, n0, kt0, kt1);
        // With k groups, group 0 holds the tile's sum; the other groups only
        // take part in the CTA-wide barriers below.
        if (p.splits > 1) {
            // re-read the CTA coordinates here so they are not held across the main loop
            const int tile2 = ctaid_x(), split2 = ctaid_y();
            float *base = p.ws + static_cast<size_t>(tile2) * p.splits * (BM * BN);
            if (g == 0) store_partial(base + static_cast<size_t>(split2) * (BM * BN));
            if (!arrive_last(&p.counters[tile2], static_cast<unsigned>(p.splits))) return;
            if (g == 0)
                for (int sp = 0; sp < p.splits; ++sp) add_partial(base + static_cast<size_t>(sp) * (BM * BN), sp == 0);
            if (threadIdx.x == 0) p.counters[tile2] = 0u;  // ready for the next call on this stream
        }
        if (g != 0) return;
        tile_origin(ctaid_x(), m0, n0);
        epilogue(m0, n0);
    } else {
        // Persistent CTAs (one per SM).  Stream-K part first: the last
        // sk_tiles tiles of the raster are cut into G contiguous ranges of k
        // slices, one per CTA (each range at most one tile long, so it
        // touches at most two tiles).  A CTA that covers a whole tile
        // finishes it; otherwise it writes its partial tile to its slot
        // (2 * cta + segment) and sgemm_streamk_fixup_kernel, launched next on
        // the same stream, adds the slots of each tile in k order.  The
        // segment list lives in shared memory so that it is not held in
        // registers across the main loop.
        __shared__ int s_seg[2][3];  // sk-local tile, first and end k slice
        __shared__ int s_nseg;
        const int G = gridDim.x;
        const int cta = blockIdx.x;
        if (tid == 0) {
            int n = 0;
            if (p.sk_tiles > 0) {
                const long long I = static_cast<long long>(p.sk_tiles) * KT;
                const long long b = cta * I / G, e = (cta + 1) * I / G;
                for (long long i0 = b; i0 < e && n < 2; ++n) {
                    const int ts = static_cast<int>(i0 / KT);
                    s_seg[n][0] = ts;
                    s_seg[n][1] = static_cast<int>(i0 - static_cast<long long>(ts) * KT);
                    s_seg[n][2] = static_cast<int>(min(static_cast<long long>(KT), e - static_cast<long long>(ts) * KT));
                    i0 = static_cast<long long>(ts + 1) * KT;
                }
            }
            s_nseg = n;
        }
        __syncthreads();
        const volatile int *vseg = &s_seg[0][0];
        const int n_sk = s_nseg;
        const int n_dp = cta < p.dp_tiles ? (p.dp_tiles - cta + G - 1) / G : 0;
        for (int w = 0; w < n_sk + n_dp; ++w) {
            int m0, n0;
            if (w < n_sk) {
                tile_origin(p.dp_tiles + vseg[w * 3], m0, n0);
                mainloop(m0, n0, vseg[w * 3 + 1], vseg[w * 3 + 2]);
                if (!(vseg[w * 3 + 1] == 0 && vseg[w * 3 + 2] == KT)) {
                    store_partial(p.ws + static_cast<size_t>(2 * ctaid_x() + (vseg[w * 3] - vseg[0])) * (BM * BN));
                    continue;
                }
                tile_origin(p.dp_tiles + vseg[w * 3], m0, n0);
            } else {
                tile_origin(cta + (w - n_sk) * G, m0, n0);
                mainloop(m0, n0, 0, KT);
                tile_origin(ctaid_x() + (w - n_sk) * G, m0, n0);
            }
            epilogue(m0, n0);
        }
    }
}

// Stream-K fixup: for stream-K tile blockIdx.x, add the partial tiles of the
// CTAs that covered it in k order (owner(i) = ((i+1)G - 1) / I is the CTA
// whose range holds k slice i) and apply the epilogue.  Tiles covered whole
// by one CTA were finished by the main kernel.  blockIdx.y picks 8 rows.
template <int BM, int BN>
__global__ void __launch_bounds__(256) sgemm_streamk_fixup_kernel(const SgemmArgs p) {
    const int KT = (p.K + kBK - 1) / kBK;
    const int G = p.grid_ctas;
    const int ts = blockIdx.x;
    const long long I = static_cast<long long>(p.sk_tiles) * KT;
    const long long f = static_cast<long long>(ts) * KT;
    const int c0 = static_cast<int>(((f + 1) * G - 1) / I);
    const int c1 = static_cast<int>(((f + KT) * G - 1) / I);
    if (c0 == c1) return;
    const int tile = p.dp_tiles + ts;
    const int group_tiles = 8 * p.tiles_n;
    const int first_m = (tile / group_tiles) * 8;
    const int gsz = min(p.tiles_m - first_m, 8);
    const int m0 = (first_m + (tile % group_tiles) % gsz) * BM;
    const int n0 = ((tile % group_tiles) / gsz) * BN;
    // slot of each contributing CTA, in k order (a tile has few contributors)
    constexpr int kMaxOwners = 64;
    __shared__ int s_slot[kMaxOwners];
    const int n_own = min(c1 - c0 + 1, kMaxOwners);
    for (int i = threadIdx.x; i < n_own; i += blockDim.x) {
        const int cc = c0 + i;
        s_slot[i] = 2 * cc + (ts - static_cast<int>((static_cast<long long>(cc) * I / G) / KT));
    }
    __syncthreads();
    constexpr int kVecPerRow = BN / 4;
    for (int v = threadIdx.x; v < 8 * kVecPerRow; v += blockDim.x) {
        const int r = blockIdx.y * 8 + v / kVecPerRow;
        const int c = (v % kVecPerRow) * 4;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < n_own; ++i) {
            const size_t wi = static_cast<size_t>(s_slot[i]) * (BM * BN) + r * BN + c;
            if (!debug_in_bounds(sg_ws_floats(p) == 0 || wi + 4 <= sg_ws_floats(p), sg_err(p))) continue;
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(p.ws + wi));
            if (i == 0) {
                s = x;
            } else {
                s.x += x.x;
                s.y += x.y;
                s.z += x.z;
                s.w += x.w;
            }
        }
        const int gr = m0 + r, gc = n0 + c;
        if (gr >= p.M) continue;
        float *crow = p.C + static_cast<size_t>(gr) * p.ldc;
        const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (gc + e < p.N &&
                debug_in_bounds(sg_c_extent(p) == 0 || static_cast<size_t>(gr) * p.ldc + gc + e < sg_c_extent(p),
                                sg_err(p))) {
                float val = p.alpha * sv[e];
                if (p.beta != 0.f) val = fmaf(p.beta, crow[gc + e], val);
                crow[gc + e] = val;
            }
        }
    }
}

// ------------------------------------------------------------------ GEMV
// N == 1: y_i = alpha * sum_k A[i, k] * x_k + beta * y_i, one warp per row,
// x_k = B[k * incx], y_i = C[i * incy].  A streams once from HBM.  vec: A's
// rows are 16-byte aligned (lda % 4 == 0) and read as float4; x is read as
// float4 too when contiguous (incx == 1, 16-byte aligned), else element by
// element (a column of a row-major B).
__global__ void __launch_bounds__(256) sgemv_rows_kernel(int M, int K, float alpha, const float *__restrict__ A,
                                                         int lda, const float *__restrict__ x, int incx,
                                                         float beta, float *y, int incy, int vec) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const float *a = A + static_cast<size_t>(row) * lda;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    int kdone = 0;
    if (vec) {
        const int K4 = K >> 2;
        const float4 *a4 = reinterpret_cast<const float4 *>(a);
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
#pragma unroll 16
        for (int c = lane; c < K4; c += 32) {
            const float4 av = __ldcs(a4 + c);
            const float4 xv =
                incx == 1 ? __ldg(x4 + c)
                          : make_float4(__ldg(x + static_cast<size_t>(4 * c) * incx),
                                        __ldg(x + static_cast<size_t>(4 * c + 1) * incx),
                                        __ldg(x + static_cast<size_t>(4 * c + 2) * incx),
                                        __ldg(x + static_cast<size_t>(4 * c + 3) * incx));
            s0 = fmaf(av.x, xv.x, s0);
            s1 = fmaf(av.y, xv.y, s1);
            s2 = fmaf(av.z, xv.z, s2);
            s3 = fmaf(av.w, xv.w, s3);
        }
        kdone = K4 << 2;
    }
#pragma unroll 4
    for (int k = kdone + lane; k < K; k += 32) s0 = fmaf(a[k], x[static_cast<size_t>(k) * incx], s0);
    float s = (s0 + s1) + (s2 + s3);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
        float v = alpha * s;
        float *yp = y + static_cast<size_t>(row) * incy;
        if (beta != 0.f) v = fmaf(beta, *yp, v);
        *yp = v;
    }
}

// N == 1, 16-byte aligned rows and a contiguous x: a CTA of 256 threads
// sweeps 4 consecutive rows together, so each CTA streams one contiguous
// block of A (measured 5.4 TB/s vs 4.1 TB/s for one warp per row at
// 4096 x 4096).  Each thread keeps a partial sum per row over its strided
// float4 columns; the CTA combines them in a fixed order.
constexpr int kRowsPerCta = 4;
__global__ void __launch_bounds__(256) sgemv_rows_block_kernel(int M, int K, float alpha, const float *__restrict__ A,
                                                               int lda, const float *__restrict__ x, float beta,
                                                               float *y, int incy) {
    __shared__ float red[8][kRowsPerCta];
    const int r0 = blockIdx.x * kRowsPerCta;
    const int K4 = K >> 2;
    float acc[kRowsPerCta];
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) acc[r] = 0.f;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
#pragma unroll 4
    for (int c = threadIdx.x; c < K4; c += 256) {
        const float4 xv = __ldg(x4 + c);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) {
            if (r0 + r < M) {
                const float4 av =
                    __ldcs(reinterpret_cast<const float4 *>(A + static_cast<size_t>(r0 + r) * lda) + c);
                acc[r] = fmaf(av.w, xv.w, fmaf(av.z, xv.z, fmaf(av.y, xv.y, fmaf(av.x, xv.x, acc[r]))));
            }
        }
    }
    for (int k = (K4 << 2) + threadIdx.x; k < K; k += 256) {  // K % 4 tail
        const float xv = __ldg(x + k);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r)
            if (r0 + r < M) acc[r] = fmaf(A[static_cast<size_t>(r0 + r) * lda + k], xv, acc[r]);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) {
        float v = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][r] = v;
    }
    __syncthreads();
    if (threadIdx.x < kRowsPerCta && r0 + threadIdx.x < M) {
        float v = red[0][threadIdx.x];
#pragma unroll
        for (int w = 1; w < 8; ++w) v += red[w][threadIdx.x];
        float *yp = y + static_cast<size_t>(r0 + threadIdx.x) * incy;
        float out = alpha * v;
        if (beta != 0.f) out = fmaf(beta, *yp, out);
        *yp = out;
    }
}

// M == 1: y_j = alpha * sum_k x_k * B[k, j] + beta * y_j with x = A's row,
// y = C's row.  A CTA owns 128 columns (4 per lane) and one K chunk (blockIdx.y);
// its 8 warps take interleaved rows of B and are combined in warp order.
// With several K chunks the partial rows go to scratch and the last CTA of a
// column block adds them in chunk order.
__global__ void __launch_bounds__(256) sgemv_cols_kernel(int N, int K, float alpha, const float *__restrict__ x,
                                                         const float *__restrict__ B, int ldb, float beta,
                                                         float *y, int vec, int splits, float *ws,
                                                         unsigned *counters) {
    __shared__ float4 red[8][32];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int col = blockIdx.x * 128 + lane * 4;
    const int chunk = blockIdx.y;
    const int k0 = static_cast<int>(static_cast<long long>(K) * chunk / splits);
    const int k1 = static_cast<int>(static_cast<long long>(K) * (chunk + 1) / splits);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec && col + 3 < N) {
#pragma unroll 16
        for (int k = k0 + warp; k < k1; k += 8) {
            const float xv = __ldg(x + k);
            const float4 bv = __ldcs(reinterpret_cast<const float4 *>(B + static_cast<size_t>(k) * ldb + col));
            s.x = fmaf(xv, bv.x, s.x);
            s.y = fmaf(xv, bv.y, s.y);
            s.z = fmaf(xv, bv.z, s.z);
            s.w = fmaf(xv, bv.w, s.w);
        }
    } else if (col < N) {
        for (int k = k0 + warp; k < k1; k += 8) {
            const float xv = __ldg(x + k);
            const float *br = B + static_cast<size_t>(k) * ldb + col;
            s.x = fmaf(xv, br[0], s.x);
            if (col + 1 < N) s.y = fmaf(xv, br[1], s.y);
            if (col + 2 < N) s.z = fmaf(xv, br[2], s.z);
            if (col + 3 < N) s.w = fmaf(xv, br[3], s.w);
        }
    }
    red[warp][lane] = s;
    __syncthreads();
    float4 t = red[0][lane];  // the CTA's sum over its 8 warps, in warp order
#pragma unroll
    for (int w = 1; w < 8; ++w) {
        const float4 v = red[w][lane];
        t.x += v.x;
        t.y += v.y;
        t.z += v.z;
        t.w += v.w;
    }
    if (splits > 1) {
        float4 *slots = reinterpret_cast<float4 *>(ws + static_cast<size_t>(blockIdx.x) * splits * 128);
        if (warp == 0) slots[chunk * 32 + lane] = t;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = (atomicAdd(&counters[blockIdx.x], 1u) == static_cast<unsigned>(splits - 1));
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        // All 8 warps of the last CTA reduce: warp w adds chunks w, w + 8, ...
        // in order, then warp 0 adds the 8 warp sums in order.
        float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = warp; c < splits; c += 8) {
            const float4 v = __ldcg(slots + c * 32 + lane);
            part.x += v.x;
            part.y += v.y;
            part.z += v.z;
            part.w += v.w;
        }
        __syncthreads();  // everyone has read red[][] above
        red[warp][lane] = part;
        __syncthreads();
        if (warp != 0) return;
        t = red[0][lane];
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            const float4 v = red[w][lane];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        if (lane == 0) counters[blockIdx.x] = 0u;
    } else if (warp != 0) {
        return;
    }
    const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (col + e < N) {
            float v = alpha * tv[e];
            if (beta != 0.f) v = fmaf(beta, y[col + e], v);
            y[col + e] = v;
        }
    }
}

// M == 1 with K split over the S CTAs of a thread-block cluster (2 <= S <= 8):
// CTA r of a cluster owns rows [K r / S, K (r + 1) / S) of the cluster's 128
// columns (4 per lane; its WARPS warps take interleaved rows and are added in
// warp order) and leaves its sum in shared memory; after a cluster barrier,
// CTA 0 adds the S sums in rank order through distributed shared memory and
// writes y.  No global scratch, atomics or memory fences.  (The split-K
// kernel above spends ~1.8 us on its fence and arrival count and ~1.3 us on
// the last CTA's sum of 19 partials at 1 x 4096 x 4096, per-CTA timer
// stamps.)  Launched with programmatic dependent launch: it waits for the
// previous kernel of the stream before its first global access.
template <int S, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) sgemv_cols_cluster_kernel(int N, int K, float alpha,
                                                                        const float *__restrict__ x,
                                                                        const float *__restrict__ B, int ldb,
                                                                        float beta, float *y, int vec) {
    __shared__ float4 red[WARPS][32];
    __shared__ float4 part[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = static_cast<int>(cluster_ctarank());
    const int col = (blockIdx.x / S) * 128 + lane * 4;
    const int k0 = static_cast<int>(static_cast<long long>(K) * rank / S);
    const int k1 = static_cast<int>(static_cast<long long>(K) * (rank + 1) / S);
    pdl_wait();
    pdl_launch_dependents();
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec && col + 3 < N) {
#pragma unroll 16
        for (int k = k0 + warp; k < k1; k += WARPS) {
            const float xv = __ldg(x + k);
            const float4 bv = __ldcs(reinterpret_cast<const float4 *>(B + static_cast<size_t>(k) * ldb + col));
            s.x = fmaf(xv, bv.x, s.x);
            s.y = fmaf(xv, bv.y, s.y);
            s.z = fmaf(xv, bv.z, s.z);
            s.w = fmaf(xv, bv.w, s.w);
        }
    } else if (col < N) {
        for (int k = k0 + warp; k < k1; k += WARPS) {
            const float xv = __ldg(x + k);
            const float *br = B + static_cast<size_t>(k) * ldb + col;
            s.x = fmaf(xv, br[0], s.x);
            if (col + 1 < N) s.y = fmaf(xv, br[1], s.y);
            if (col + 2 < N) s.z = fmaf(xv, br[2], s.z);
            if (col + 3 < N) s.w = fmaf(xv, br[3], s.w);
        }
    }
    red[warp][lane] = s;
    __syncthreads();
    if (warp == 0) {
        float4 t = red[0][lane];
#pragma unroll
        for (int w = 1; w < WARPS; ++w) {
            const float4 v = red[w][lane];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        part[lane] = t;
    }
    cluster_sync();  // every CTA's sum written and visible to the cluster
    if (rank == 0 && warp == 0) {
        float4 t = part[lane];
#pragma unroll
        for (int q = 1; q < S; ++q) {
            const float4 v = ld_shared_cluster_v4(mapa_shared(smem_u32(&part[lane]), static_cast<uint32_t>(q)));
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (col + e < N) {
                float v = alpha * tv[e];
                if (beta != 0.f) v = fmaf(beta, y[col + e], v);
                y[col + e] = v;
            }
        }
    }
    cluster_sync();  // the peers' sums stay in place until CTA 0 has read them
}

// alpha == 0 or K == 0: C = act(beta * C + bias) (beta == 0 writes without reading).
__global__ void scale_c_kernel(int M, int N, float beta, float *C, int ldc, const float *bias, int act) {
    const long long total = static_cast<long long>(M) * N;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(e / N), j = static_cast<int>(e % N);
        float *c = C + static_cast<size_t>(i) * ldc + j;
        float v = beta != 0.f ? beta * *c : 0.f;
        if (bias) v += bias[j];
        v = apply_activation(act, v);
        *c = v;
    }
}

// The same over a strided batch of M x N matrices (ldc = N) of any output
// type (c_type as in load_out / store_out).
__global__ void scale_c_batched_kernel(int M, int N, long long total, float beta, void *C, long long stride_c,
                                       int c_type, const float *bias, int act) {
    const long long mn = static_cast<long long>(M) * N;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long z = e / mn, r = e - z * mn;
        const int j = static_cast<int>(r % N);
        const size_t idx = static_cast<size_t>(z * stride_c + r);
        float v = beta != 0.f ? beta * load_out(C, idx, c_type) : 0.f;
        if (bias) v += bias[j];
        store_out(C, idx, c_type, apply_activation(act, v));
    }
}

// Copy a rows x cols window with leading dimension ld_src into a buffer with
// leading dimension ld_dst (a multiple of 4, 16-byte aligned rows).  Each CTA
// copies whole rows (blockIdx.y strides over rows); threads walk the columns.
__global__ void __launch_bounds__(256) repack_rows_kernel(const float *__restrict__ src, int rows, int cols,
                                                          int ld_src, float *__restrict__ dst, int ld_dst) {
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *s = src + static_cast<size_t>(r) * ld_src;
        float *d = dst + static_cast<size_t>(r) * ld_dst;
#pragma unroll 4
        for (int c = threadIdx.x; c < cols; c += 256) d[c] = __ldcs(s + c);
    }
}

template <int BM, int BN, int WARPS_M, int WARPS_N, int TM, int TN, int STAGES, bool VEC, bool PERSIST, int KG = 1>
cudaError_t launch_tiled(const SgemmArgs &a, cudaStream_t stream) {
    using T = SgemmTile<BM, BN, WARPS_M, WARPS_N, TM, TN, STAGES, VEC, KG>;
    auto kern = sgemm_tiled_kernel<BM, BN, WARPS_M, WARPS_N, TM, TN, STAGES, VEC, PERSIST, KG>;
    static unsigned long long smem_set = 0;
    cudaError_t e = ensure_dynamic_smem(kern, T::kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    dim3 grid = PERSIST ? dim3(a.grid_ctas, 1) : dim3(a.tiles_m * a.tiles_n, a.splits);
    return launch_kernel(kern, grid, dim3(T::kThreads), T::kSmemBytes, stream, a);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int S, int WARPS>
cudaError_t launch_gemv_cluster(int col_blocks, int N, int K, float alpha, const float *x, const float *B, int ldb,
                                float beta, float *y, int vec, cudaStream_t stream) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(col_blocks * S, 1, 1);
    cfg.blockDim = dim3(WARPS * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sgemv_cols_cluster_kernel<S, WARPS>, N, K, alpha, x, B, ldb, beta, y, vec);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

// 16 warps per CTA when the clusters give fewer than ~3 CTAs per SM, so that
// as many loads stay in flight as with more, smaller CTAs.
template <int S>
cudaError_t launch_gemv_cluster_w(int col_blocks, int N, int K, float alpha, const float *x, const float *B, int ldb,
                                  float beta, float *y, int vec, cudaStream_t stream) {
    if (col_blocks * S < 3 * device_sm_count())
        return launch_gemv_cluster<S, 16>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
    return launch_gemv_cluster<S, 8>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
}

cudaError_t launch_gemv_cluster_any(int s, int col_blocks, int N, int K, float alpha, const float *x, const float *B,
                                    int ldb, float beta, float *y, int vec, cudaStream_t stream) {
    switch (s) {
        case 2: return launch_gemv_cluster_w<2>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
        case 3: return launch_gemv_cluster_w<3>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
        case 4: return launch_gemv_cluster_w<4>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
        case 5: return launch_gemv_cluster_w<5>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
        case 6: return launch_gemv_cluster_w<6>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
        case 7: return launch_gemv_cluster_w<7>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
        default: return launch_gemv_cluster_w<8>(col_blocks, N, K, alpha, x, B, ldb, beta, y, vec, stream);
    }
}

}  // namespace

cudaError_t run_scale_c(int M, int N, float beta, float *C, int ldc, const float *bias, int act,
                        cudaStream_t stream, CallInfo *info) {
    if (beta == 1.f && !bias && act == 0) {
        info->plan = "noop_beta1";
        info->launches = 0;
        return cudaSuccess;
    }
    const long long total = static_cast<long long>(M) * N;
    const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 4LL * device_sm_count()));
    info->plan = "scale_c";
    info->launches = 1;
    return launch_kernel(scale_c_kernel, dim3(blocks), dim3(256), 0, stream, M, N, beta, C, ldc, bias, act);
}

cudaError_t run_scale_c_batched(int batch, int M, int N, float beta, void *C, long long stride_c, int c_type,
                                const float *bias, int act, cudaStream_t stream, CallInfo *info) {
    if (beta == 1.f && !bias && act == 0) {
        info->plan = "noop_beta1";
        info->launches = 0;
        return cudaSuccess;
    }
    const long long total = static_cast<long long>(batch) * M * N;
    const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 4LL * device_sm_count()));
    info->plan = "scale_c_batched";
    info->launches = 1;
    return launch_kernel(scale_c_batched_kernel, dim3(blocks), dim3(256), 0, stream, M, N, total, beta, C, stride_c,
                      c_type, bias, act);
}

cudaError_t run_gemm_f32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                         float beta, float *C, int ldc, cudaStream_t stream, CallInfo *info) {
    const int sms = device_sm_count();
    if (N == 1) {
        const int vec = aligned16(A) && (lda % 4 == 0) && ldb == 1 && aligned16(B);
        info->launches = 1;
        if (vec) {
            info->plan = "sgemv_rows_block";
            return launch_kernel(sgemv_rows_block_kernel, dim3((M + kRowsPerCta - 1) / kRowsPerCta), dim3(256), 0, stream,
                              M, K, alpha, A, lda, B, beta, C, ldc);
        }
        info->plan = "sgemv_rows";
        return launch_kernel(sgemv_rows_kernel, dim3((M + 7) / 8), dim3(256), 0, stream, M, K, alpha, A, lda, B, ldb, beta,
                          C, ldc, 0);
    }
    if (M == 1) {
        const int vec = aligned16(B) && (ldb % 4 == 0);
        const int col_blocks = (N + 127) / 128;
        // enough CTAs for every SM to stream B: about 4 per SM, each K chunk >= 64 rows
        int splits = std::max(1, std::min((4 * sms + col_blocks - 1) / col_blocks, K / 64));
        splits = std::min(splits, 64);
        // Up to 8 splits, while that still gives every SM a CTA: the splits of a
        // column block are the CTAs of one cluster, summed through distributed
        // shared memory.
        if (splits > 1 && col_blocks * 8 >= sms) {
            const int cs = std::min(splits, 8);
            info->plan = "sgemv_cols_clusterk";
            info->launches = 1;
            return launch_gemv_cluster_any(cs, col_blocks, N, K, alpha, A, B, ldb, beta, C, vec, stream);
        }
        Scratch sc;
        if (splits > 1) {
            cudaError_t e = acquire_scratch(stream, static_cast<size_t>(col_blocks) * splits * 128, col_blocks, &sc);
            if (e != cudaSuccess) return e;
        }
        info->plan = splits > 1 ? "sgemv_cols_splitk" : "sgemv_cols";
        info->launches = 1;
        return launch_kernel(sgemv_cols_kernel, dim3(col_blocks, splits), dim3(256), 0, stream, N, K, alpha, A, B, ldb, beta,
                          C, vec, splits, sc.partials, sc.counters);
    }

    SgemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.alpha = alpha;
    a.beta = beta;
    a.A = A;
    a.B = B;
    a.C = C;
    a.lda = lda;
    a.ldb = ldb;
    a.ldc = ldc;
    a.c_vec = aligned16(C) && (ldc % 4 == 0);
    // checked extent of C (debug builds; a test hook may shrink it)
    size_t c_extent = static_cast<size_t>(M - 1) * ldc + N;
    if (kDebugBuild) c_extent -= std::min<size_t>(c_extent, debug_shrink_c());
    sg_set_debug(a, c_extent, 0, watchdog_word());
    bool vec = aligned16(A) && aligned16(B) && (lda % 4 == 0) && (ldb % 4 == 0);
    const int KT = (K + kBK - 1) / kBK;
    int repacked = 0;
    // Rows that are not 16-byte aligned (lda = 4099 and the like) force 4-byte
    // copies in the main loop (measured 46 vs 62 TFLOP/s at ~4096^3).  For
    // large problems, copy A and B once into 16-byte aligned scratch rows
    // (about 1.5 % of the GEMM time at 4096^3) and run the 16-byte path.
    if (!vec && static_cast<double>(M) * N * K >= 2.0e9) {
        const bool a_ok = aligned16(A) && (lda % 4 == 0), b_ok = aligned16(B) && (ldb % 4 == 0);
        const int lda2 = (K + 3) & ~3, ldb2 = (N + 3) & ~3;
        const size_t a_floats = a_ok ? 0 : ((static_cast<size_t>(M) * lda2 + 63) & ~size_t(63));
        const size_t b_floats = b_ok ? 0 : static_cast<size_t>(K) * ldb2;
        float *ops = nullptr;
        cudaError_t e = acquire_operand_scratch(stream, a_floats + b_floats + 64, &ops);
        if (e != cudaSuccess) return e;
        const int blocks = 8 * sms;
        if (!a_ok) {
            e = launch_kernel(repack_rows_kernel, dim3(blocks), dim3(256), 0, stream, A, M, K, lda, ops, lda2);
            if (e != cudaSuccess) return e;
            a.A = ops;
            a.lda = lda2;
            ++repacked;
        }
        if (!b_ok) {
            float *B2 = ops + a_floats;  // 256-byte aligned
            e = launch_kernel(repack_rows_kernel, dim3(blocks), dim3(256), 0, stream, B, K, N, ldb, B2, ldb2);
            if (e != cudaSuccess) return e;
            a.B = B2;
            a.ldb = ldb2;
            ++repacked;
        }
        e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
        vec = true;
    }

    // Tile table.  128x256 CTAs (8 warps, one per SM) run persistently when
    // there are big tiles for at least ~80 % of the SMs: whole tiles
    // round-robin, and the tiles of the last partial wave shared out by k
    // slices (stream-K), so every SM gets the same number of k slices.
    // Fewer big tiles run faster as 64x64 tiles (autotuner on GB300:
    // 1024^3 51.2 vs 53.6 us, 1000 x 3000 x 777 102.8 vs 110.2 us;
    // 2048^3 with 128 big tiles stays big: 295 vs 320 us).
    const int tiles_big = ((M + 127) / 128) * ((N + 255) / 256);
    bool big = 5 * tiles_big >= 4 * sms;
    TunePlan tp;
    if (tune_lookup(0, M, N, K, &tp)) {  // a tuned plan for this exact shape
        big = tp.variant == 1;
        info->tuned = true;
    }
    cudaError_t e;
    // Edge strip (the pages' main tiles plus separate edge kernels): when the
    // last 256-wide tile column would hold at most 64 real columns, the big
    // tiles cover the first N0 = N - r columns and the r-column strip runs
    // after them -- as a matrix-vector product when r = 1, else as 64x64
    // tiles -- instead of a column of mostly empty 128 x 256 tiles
    // (4095 x 4097 x 4099: 544 -> 512 big tiles).
    const int strip = (big && N > 256 && N % 256 != 0 && N % 256 <= 64) ? N % 256 : 0;
    const int N0 = N - strip;
    if (big) {
        a.N = N0;
        a.tiles_m = (M + 127) / 128;
        a.tiles_n = (N0 + 255) / 256;
        a.splits = 1;
        a.persistent = 1;
        const int tiles_main = a.tiles_m * a.tiles_n;
        const int rem = tiles_main % sms;
        a.dp_tiles = tiles_main - rem;
        a.sk_tiles = rem;
        const long long share = static_cast<long long>(rem) * KT / sms;  // k slices per CTA
        // too few k slices to share out (or too many CTAs per tile for the
        // fixup's owner list): whole tiles only
        if (rem != 0 && (share < 2 || KT / share + 2 > 64)) {
            a.dp_tiles = tiles_main;
            a.sk_tiles = 0;
        }
        a.grid_ctas = a.sk_tiles > 0 ? sms : std::min(sms, tiles_main);
        // A strip of r > 1 columns runs as 64x64 tiles with split K; its
        // partials follow the big tiles' stream-K partials in one scratch
        // request made before anything is launched (a request that grows the
        // buffer synchronises the stream).
        SgemmArgs s2 = a;
        if (strip > 1) {
            s2.N = strip;
            s2.B = a.B + N0;
            s2.C = C + N0;
            sg_set_debug(s2, c_extent > static_cast<size_t>(N0) ? c_extent - N0 : 1, 0, watchdog_word());
            s2.c_vec = aligned16(s2.C) && (ldc % 4 == 0);
            s2.tiles_m = (M + 63) / 64;
            s2.tiles_n = 1;
            s2.persistent = 0;
            s2.dp_tiles = s2.sk_tiles = s2.grid_ctas = 0;
            int splits = 1;
            if (s2.tiles_m < sms && KT > 4) splits = std::max(1, std::min((sms + s2.tiles_m / 2) / s2.tiles_m, KT / 2));
            s2.splits = std::min(splits, 16);
        }
        const size_t main_floats = a.sk_tiles > 0 ? static_cast<size_t>(2) * a.grid_ctas * 128 * 256 : 0;
        const size_t strip_floats = (strip > 1 && s2.splits > 1) ? static_cast<size_t>(s2.tiles_m) * s2.splits * 64 * 64 : 0;
        if (main_floats + strip_floats > 0) {
            Scratch sc;
            e = acquire_scratch(stream, main_floats + strip_floats, strip_floats > 0 ? s2.tiles_m : 0, &sc);
            if (e != cudaSuccess) return e;
            a.ws = sc.partials;
            a.counters = sc.counters;
            sg_set_debug(a, c_extent, main_floats, watchdog_word());
            s2.ws = sc.partials + main_floats;
            s2.counters = sc.counters;
            sg_set_debug(s2, c_extent > static_cast<size_t>(N0) ? c_extent - N0 : 1, strip_floats, watchdog_word());
        }
        e = vec ? launch_tiled<128, 256, 2, 4, 8, 16, 3, true, true>(a, stream)
                : launch_tiled<128, 256, 2, 4, 8, 16, 3, false, true>(a, stream);
        if (e != cudaSuccess) return e;
        if (a.sk_tiles > 0) {
            e = launch_kernel(sgemm_streamk_fixup_kernel<128, 256>, dim3(a.sk_tiles, 128 / 8), dim3(256), 0, stream, a);
        }
        if (e != cudaSuccess) return e;
        info->launches = (a.sk_tiles > 0 ? 2 : 1) + repacked;
        if (a.sk_tiles > 0)
            info->plan = repacked ? "sgemm_repack_128x256_vec16_streamk"
                                  : (vec ? "sgemm_128x256_vec16_streamk" : "sgemm_128x256_vec4b_streamk");
        else
            info->plan = repacked ? "sgemm_repack_128x256_vec16" : (vec ? "sgemm_128x256_vec16" : "sgemm_128x256_vec4b");
        if (strip == 1) {
            // y = C[:, N0] over the rows of A, x = B[:, N0] (stride ldb, read element-wise)
            const int vrow = aligned16(a.A) && (a.lda % 4 == 0);
            e = launch_kernel(sgemv_rows_kernel, dim3((M + 7) / 8), dim3(256), 0, stream, M, K, alpha, a.A, a.lda,
                              a.B + N0, a.ldb, beta, C + N0, ldc, vrow);
            ++info->launches;
        } else if (strip > 1) {
            e = vec ? launch_tiled<64, 64, 2, 2, 4, 8, 3, true, false>(s2, stream)
                    : launch_tiled<64, 64, 2, 2, 4, 8, 3, false, false>(s2, stream);
            ++info->launches;
        }
        if (strip) {
            // the plan of this thread's last call (valid until its next call)
            static thread_local char plan_buf[96];
            std::snprintf(plan_buf, sizeof(plan_buf), "%s+colstrip%s", info->plan, strip == 1 ? "1" : "");
            info->plan = plan_buf;
        }
    } else if (!info->tuned && (M + 63) / 64 * ((N + 63) / 64) * 2 <= sms &&
               (M + 31) / 32 * ((N + 63) / 64) <= sms && K >= 256 && K <= 2048) {
        // Few tiles and a short K (512^3, 256^3): 32x64 tiles, each shared by
        // four k groups of 2 warps (4x8 per thread; group g takes the g-th 32-wide
        // k slice of every stage), so that one wave of CTAs still gives each
        // scheduler two warps; the groups' partials are added in shared memory.
        // Measured on GB300 in CUDA-graph replays: 512^3 11.0 us (12.3 us for
        // 64x64 tiles with 2 K splits), 256^3 7.6 us (8.5 us).
        a.tiles_m = (M + 31) / 32;
        a.tiles_n = (N + 63) / 64;
        a.splits = 1;
        e = vec ? launch_tiled<32, 64, 1, 2, 4, 8, 3, true, false, 4>(a, stream)
                : launch_tiled<32, 64, 1, 2, 4, 8, 3, false, false, 4>(a, stream);
        info->plan = repacked ? "sgemm_repack_32x64_kg4_vec16" : (vec ? "sgemm_32x64_kg4_vec16" : "sgemm_32x64_kg4_vec4b");
        info->launches = 1 + repacked;
    } else {
        // Small problems: 64x64 CTAs (4 warps of 32x32, 4x8 per thread), with
        // K split so that there are about as many CTAs as SMs, each split at
        // least two 32-wide k slices, and no split at all for K <= 128 (the
        // partial-tile round trip costs more than it gains there).  Measured
        // on GB300: 512^3 13.0 us at 2 splits (20.3 us at 8), 256^3 8.8 us at
        // 4, 128^3 6.1 us unsplit (7.4 us at 2).
        a.tiles_m = (M + 63) / 64;
        a.tiles_n = (N + 63) / 64;
        const int tiles = a.tiles_m * a.tiles_n;
        int splits = 1;
        if (tiles < sms && KT > 4) splits = std::max(1, std::min((sms + tiles / 2) / tiles, KT / 2));
        splits = std::min(splits, 16);
        if (info->tuned && tp.splits > 0) splits = std::max(1, std::min(tp.splits, std::max(1, KT / 2)));
        a.splits = splits;
        if (splits > 1) {
            Scratch sc;
            e = acquire_scratch(stream, static_cast<size_t>(tiles) * splits * 64 * 64, tiles, &sc);
            if (e != cudaSuccess) return e;
            a.ws = sc.partials;
            a.counters = sc.counters;
            sg_set_debug(a, c_extent, static_cast<size_t>(tiles) * splits * 64 * 64, watchdog_word());
        }
        e = vec ? launch_tiled<64, 64, 2, 2, 4, 8, 3, true, false>(a, stream)
                : launch_tiled<64, 64, 2, 2, 4, 8, 3, false, false>(a, stream);
        if (splits > 1)
            info->plan = repacked ? "sgemm_repack_64x64_vec16_splitk"
                                  : (vec ? "sgemm_64x64_vec16_splitk" : "sgemm_64x64_vec4b_splitk");
        else
            info->plan = repacked ? "sgemm_repack_64x64_vec16" : (vec ? "sgemm_64x64_vec16" : "sgemm_64x64_vec4b");
        info->launches = 1 + repacked;
    }
    return e;
}

}  // namespace gemm11
