// hgemm.cu -- FP16/BF16-input / FP32-accumulate GEMM on the 5th-generation
// tensor cores (tcgen05) of sm_103a, with the bias / scale / activation
// epilogue fused; also strided batches (B optionally stored N x K) and the
// FP32-accuracy product through three TF32 products.
//
//   C = act(alpha * A x B + beta * C + bias),  A: M x K row-major,
//   B: K x N (or N x K) row-major, C: M x N fp32/fp16/bf16, bias: N fp32.
//
// The DeepGEMM essay "企业官网建设流程全解析" describes the Hopper version of
// this pipeline: TMA tiles into a 4-stage shared-memory ring guarded by
// mbarriers (sections 3.2, 3.3), accumulators that never leave the register
// file until the epilogue (section 4.3), the fused bias/scale/activation
// epilogue with a single store (sections 1.3, 3.2), an L2-aware tile raster
// (section 3.4), main tiles plus edge handling and split-K for awkward
// shapes (sections 5.3, 6.3).  On sm_103a the same ideas map to:
//   * one persistent CTA per SM, three warp roles: a TMA producer warp, an
//     MMA warp whose single thread issues tcgen05.mma, and four epilogue
//     warps;
//   * the accumulator lives in tensor memory (TMEM), double-buffered, so the
//     epilogue of tile i overlaps the main loop of tile i+1;
//   * operand tiles are staged by TMA with the 128-byte swizzle, which is the
//     canonical layout the MMA reads (A K-major, B MN-major: B is row-major
//     K x N, so N is its contiguous dimension);
//   * the epilogue reads TMEM with tcgen05.ld, applies alpha, beta*C, bias
//     and GELU in registers, stages the 32x32 fp32 block in swizzled shared
//     memory and writes it with a TMA store (edges clipped by the tensor map);
//   * M > 128: CTA pairs (tcgen05.mma.cta_group::2) compute 256-row tiles,
//     each CTA staging its 128 rows of A and half of B;
//   * small M (<= 64): the product is computed transposed, C^T = B^T A^T, so
//     that N fills the 128-row side of the MMA and M becomes its N side;
//   * too few tiles for the SMs: K is split over the CTAs of a thread-block
//     cluster and the partial tiles are added in split order through
//     distributed shared memory (no global scratch); the no-allocation entry
//     and tuned plans can also split K through a scratch buffer, where the
//     last epilogue warp to finish a 32-row slice of a tile (atomic arrival
//     count) adds the slices in split order -- deterministic either way.
// Every mbarrier wait is bounded; a timeout sets the watchdog word and the
// CTA unwinds (waits for its TMA copies and MMAs, frees TMEM, returns).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace gemm11 {
namespace {

constexpr int kBM = 128;          // MMA M (rows of the accumulator = TMEM lanes)
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row of fp16
constexpr int kUmmaK = 16;        // k per tcgen05.mma (kind::f16)
constexpr int kThreads = 192;     // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpiWarps = 4;
constexpr int kX3ChunkKB = 4;     // FP32-accuracy mode: k blocks (of 32) per tensor-core accumulation

struct HgemmArgs {
    int M, N, K;
    float alpha, beta;
    const float *bias;
    int act;
    void *C;     // row-major M x N, rows ldc elements apart (beta reads, transposed stores)
    int ldc;
    int c_type;  // kOutF32, kOutF16 or kOutBF16
    int tiles_m, tiles_n, kb_total, splits, units;
    float *ws;
    unsigned *counters;
    unsigned *err;
    uint32_t idesc_fmt;  // operand-format bits of the MMA instruction descriptor (BF16: A and B)
    uint32_t idesc;      // the whole instruction descriptor (set by the launcher for its tile shape)
    // Strided batch: matrix z of A/B/C starts z * stride elements after the
    // first (the tensor maps carry the strides).  za / zb are 0 for an operand
    // shared by every matrix of the batch (stride 0), else 1.
    int batch, za, zb;
    long long stride_c;
    int b_kmajor;  // 1: B is stored N x K (the product uses its transpose), 0: K x N
    int c64;       // 16-bit C stored in 32 x 64 boxes (128-byte rows; pair kernel, tile width % 64 == 0)
    // Single-CTA kernel only: the limit of each of its bounded waits, and a
    // diagnostic switch under which the TMA producer issues nothing at all (no
    // load, no arrival), so that the MMA and epilogue waits must run out.
    unsigned long long wait_ns = kWaitLimitNs;
    int stall_producer = 0;
    // Checked only by GEMM11_DEBUG builds (0 = unchecked): elements of C over
    // the whole batch, and floats of ws.
    size_t c_extent = 0, ws_floats = 0;
};

// Host: the C extent a debug build checks stores against.
inline size_t c_extent_of(const HgemmArgs &a) {
    return static_cast<size_t>(a.batch - 1) * static_cast<size_t>(a.stride_c) + static_cast<size_t>(a.M - 1) * a.ldc +
           static_cast<size_t>(a.N);
}

__host__ __device__ constexpr int tmem_cols_for(int bn) {
    return (2 * bn <= 32) ? 32 : (2 * bn <= 64) ? 64 : (2 * bn <= 128) ? 128 : (2 * bn <= 256) ? 256 : 512;
}

// CSPLIT: the K splits of a tile are the CTAs of one thread-block cluster,
// and the partial tiles are added through distributed shared memory: each
// CTA puts its 128 x BN fp32 partial in its own shared memory, and CTA r of
// the cluster sums rows [r * 128 / s, (r + 1) * 128 / s) of all s partials
// (in split order) and writes them to C.  Two cluster-wide mbarriers per CTA
// hand the partial buffer over: "ready" (every CTA's partial is written) and
// "consumed" (every CTA has read this CTA's partial).  No global scratch,
// atomics or memory fences.
// Not transposed (SWAP false), every CTA computes exactly one unit and its
// partial overwrites the operand ring, which is idle once the unit's MMAs
// have completed; the host launches one CTA per unit.
// EPI: epilogue warps (4, or 8 for the whole-tile non-transposed plan whose
// tiles fit one per CTA, so that the epilogue is not hidden behind another
// tile's main loop: two warps per TMEM lane quarter take alternate 32-column
// chunks, one 4 KB staging buffer each).
template <int BN, int STAGES, bool SWAP, bool CSPLIT = false, int EPI = 4>
struct HgemmCfg {
    static constexpr int kThreads = 64 + 32 * EPI;
    static constexpr int kNBuf = EPI == 4 ? 2 : 1;  // 4 KB staging buffers per epilogue warp
    static constexpr int kABytes = kBM * kBK * 2;  // 16 KB: 128 rows of 128 B
    // B: BN rows of 128 B (K-major), or whole 64-column boxes of 64 k-rows
    // (MN-major; with BN = 96 the second box reaches 32 columns past the tile)
    static constexpr int kBBytes = SWAP ? BN * kBK * 2 : (BN + 63) / 64 * 64 * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr bool kPartInRing = CSPLIT && !SWAP;
    static constexpr int kCStageBytes =
        kPartInRing ? BN * 4  // the tile's bias slice
                    : (CSPLIT ? kBM * BN * 4 : (SWAP ? 0 : EPI * kNBuf * 32 * 32 * 4));  // partial tile, or staging
    static constexpr int kBarBytes = (2 * STAGES + 7) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kCStageBytes + kBarBytes;
    static constexpr int kTmemCols = tmem_cols_for(BN);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "MMA N (and 32-column TMEM reads)");
    static_assert(STAGES <= 8, "stage bookkeeping uses 8-bit masks");
    static_assert(!kPartInRing || STAGES * kStageBytes >= kBM * BN * 4, "the partial tile fits in the operand ring");
    static_assert(!kPartInRing || BN % 64 == 0, "partial rows are 32-column groups of 8 swizzled 16-byte chunks");
    static_assert(EPI == 4 || (EPI == 8 && !SWAP && !CSPLIT), "8 epilogue warps: whole non-transposed tiles only");
};


struct UnitCoord {
    int tile, split, m0, n0, kb0, kb1, batch;
};

// An element store to C, skipped (and recorded) by debug builds when the
// index lies outside C.
__device__ __forceinline__ void store_c(const HgemmArgs &p, size_t ci, float v) {
    if (debug_in_bounds(p.c_extent == 0 || ci < p.c_extent, p.err)) store_out(p.C, ci, p.c_type, v);
}

// Tile number (over the whole batch) -> matrix index and tile origin.
__device__ __forceinline__ void tile_origin(const HgemmArgs &p, int tile, int bn_tile, bool swap, UnitCoord &c) {
    const int per = p.tiles_m * p.tiles_n;
    c.batch = tile / per;
    const int t = tile - c.batch * per;
    if (swap) {
        c.m0 = 0;
        c.n0 = t * kBM;
    } else {
        // Grouped raster: 8 M-tiles per sweep over N (L2 reuse of B panels).
        const int group_tiles = 8 * p.tiles_n;
        const int first_m = (t / group_tiles) * 8;
        const int gsz = min(p.tiles_m - first_m, 8);
        c.m0 = (first_m + (t % group_tiles) % gsz) * kBM;
        c.n0 = ((t % group_tiles) / gsz) * bn_tile;
    }
}

__device__ __forceinline__ UnitCoord decode_unit(const HgemmArgs &p, int u, int bn_tile, bool swap) {
    UnitCoord c;
    c.tile = u / p.splits;
    c.split = u % p.splits;
    tile_origin(p, c.tile, bn_tile, swap, c);
    c.kb0 = static_cast<int>(static_cast<long long>(p.kb_total) * c.split / p.splits);
    c.kb1 = static_cast<int>(static_cast<long long>(p.kb_total) * (c.split + 1) / p.splits);
    return c;
}

// The idx-th unit of this CTA (units u = blockIdx.x + idx * gridDim.x);
// false past the last one.  All three warp roles walk the same sequence.
__device__ __forceinline__ bool next_unit(const HgemmArgs &p, int idx, int bn_tile, bool swap, UnitCoord &c) {
    const int u = blockIdx.x + idx * gridDim.x;
    if (u >= p.units) return false;
    c = decode_unit(p, u, bn_tile, swap);
    return true;
}

__device__ __forceinline__ void flag_timeout(volatile int *abort_flag, unsigned *err) {
    *abort_flag = 1;
    atomicOr(err, kWatchdogTimeout);
}

// Bias of the 32-column chunks a warp will process, in its order: lane l
// holds the bias of column n0 + 32 chunk(i) + l in b[i] (0 past N or without
// bias).  Loaded before the epilogue waits for the accumulator, so the
// loads' latency (an L2 round trip per chunk otherwise) hides behind the
// main loop; the epilogue broadcasts b[0] by shuffles, then rotates b.
template <int NCH, typename ChunkOf>
__device__ __forceinline__ void load_bias_lanes(const HgemmArgs &p, int n0, int lane, ChunkOf chunk_of,
                                                float (&b)[NCH]) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int n = n0 + chunk_of(i) * 32 + lane;
        b[i] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f;
    }
}
template <int NCH>
__device__ __forceinline__ void rotate_bias_lanes(float (&b)[NCH]) {
#pragma unroll
    for (int i = 0; i + 1 < NCH; ++i) b[i] = b[i + 1];
}

// Epilogue of one row chunk: v[j] holds the accumulator of C[grow][col0 + j],
// j < 32.  Each optional term is one uniform pass over the chunk (the flags
// are kernel arguments), so the common alpha-only case is 32 multiplies:
// v = act(alpha * acc + beta * C + bias).  N % 8 == 0 and 16-byte aligned
// C rows let in-range groups of 4 columns use 128-bit loads.  The bias of
// column col0 + lane arrives in this lane's `blane` (the whole warp calls
// this together).
__device__ __forceinline__ void epilogue_row_chunk(float (&v)[32], const HgemmArgs &p, int grow, int col0,
                                                   size_t cbase, float blane) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= p.alpha;
    if (p.beta != 0.f && grow < p.M) {
        if (p.c_type == kOutF32) {
            const float *crow = static_cast<const float *>(p.C) + cbase + static_cast<size_t>(grow) * p.ldc;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int gc = col0 + 4 * q;
                if (gc + 4 <= p.N) {  // 16-byte aligned: ldc % 4 == 0 and C 16-byte aligned
                    const float4 c4 = *reinterpret_cast<const float4 *>(crow + gc);
                    v[4 * q] = fmaf(p.beta, c4.x, v[4 * q]);
                    v[4 * q + 1] = fmaf(p.beta, c4.y, v[4 * q + 1]);
                    v[4 * q + 2] = fmaf(p.beta, c4.z, v[4 * q + 2]);
                    v[4 * q + 3] = fmaf(p.beta, c4.w, v[4 * q + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (gc + i < p.N) v[4 * q + i] = fmaf(p.beta, crow[gc + i], v[4 * q + i]);
                }
            }
        } else {
            // 16-bit C: groups of 8 columns are 16-byte aligned (N % 8 == 0)
            const uint16_t *crow = static_cast<const uint16_t *>(p.C) + cbase + static_cast<size_t>(grow) * p.ldc;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int gc = col0 + 8 * q;
                if (gc < p.N) {
                    float c8[8];
                    unpack8_out16(*reinterpret_cast<const uint4 *>(crow + gc), p.c_type, c8);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[8 * q + i] = fmaf(p.beta, c8[i], v[8 * q + i]);
                }
            }
        }
    }
    if (p.bias) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, blane, j);
    }
    // One uniform pass per activation (the branch is taken once per chunk).
    // The GELU forms run as a rolled loop over four groups of 8 that rotates
    // the register array by 8 each trip (register moves): 8 inlined copies of
    // the function per call site instead of 32, which measured 3-4 % faster
    // on the CTA-pair kernel (smaller code beside the MMA issuer's loop).
    if (p.act == 2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.f);
    } else if (p.act == 1 || p.act == 3) {
        const int act = p.act;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = act == 1 ? gelu_erf(v[i]) : gelu_tanh(v[i]);
#pragma unroll
            for (int i = 0; i < 24; ++i) v[i] = v[i + 8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[24 + i] = t[i];
        }
    }
}

// Stage one finished 32 x 32 block (this lane's row: v) in one of the warp's
// two 4 KB buffers and TMA-store it at (row0, col0).  FP32: 128-byte rows,
// 128-byte swizzle (16-byte chunk c of row r at c ^ (r & 7)).  16-bit types:
// 64-byte rows, 64-byte swizzle (chunk c of row r at c ^ ((r >> 1) & 3)).
// Both patterns put the 32 lanes' 16-byte writes on distinct banks per
// quarter warp.  One bulk group is committed per chunk (possibly empty), so
// with two buffers waiting for all but the newest group frees the buffer
// about to be reused (with one buffer: waiting for all groups).
template <int NBUF = 2>
__device__ __forceinline__ void store_row_chunk(const float (&v)[32], const HgemmArgs &p, const CUtensorMap *tm_c,
                                                uint8_t *stage_base, uint32_t &n_staged, int lane, int row0,
                                                int col0, int batch) {
    static_assert(NBUF == 1 || NBUF == 2, "one or two staging buffers per warp");
    uint8_t *stage = stage_base + (NBUF == 2 ? (n_staged & 1u) * 4096 : 0u);
    ++n_staged;
    if (lane == 0) {
        if (NBUF == 2)
            bulk_wait_read_all_but_one();
        else
            bulk_wait_read_all();
    }
    __syncwarp();
    if (p.c_type == kOutF32) {
        float *st = reinterpret_cast<float *>(stage) + lane * 32;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4 *>(st + ((c4 ^ (lane & 7)) << 2)) =
                make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
    } else {
        uint4 *st = reinterpret_cast<uint4 *>(stage + lane * 64);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            uint4 w;
            w.x = pack2_out16(v[8 * c8], v[8 * c8 + 1], p.c_type);
            w.y = pack2_out16(v[8 * c8 + 2], v[8 * c8 + 3], p.c_type);
            w.z = pack2_out16(v[8 * c8 + 4], v[8 * c8 + 5], p.c_type);
            w.w = pack2_out16(v[8 * c8 + 6], v[8 * c8 + 7], p.c_type);
            st[c8 ^ ((lane >> 1) & 3)] = w;
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (row0 < p.M && col0 < p.N) tma_store_3d(tm_c, stage, col0, row0, batch);
        bulk_commit();
    }
}

// 16-bit C, 64 columns per store: `w` holds this lane's row (8 x 16 bytes);
// staged as 32 rows of 128 bytes with the 128-byte swizzle (chunk c of row r
// at c ^ (r & 7)) and written by one TMA store of a 32 x 64 box.  Halving the
// stores of the 32-column path measured ~1.6x on store-bound tiles.
template <int NBUF>
__device__ __forceinline__ void store_row_unit64(const uint4 (&w)[8], const CUtensorMap *tm_c, uint8_t *stage_base,
                                                 uint32_t &n_staged, int lane, int row0, int col0, int batch, int M,
                                                 int N) {
    uint8_t *stage = stage_base + (NBUF == 2 ? (n_staged & 1u) * 4096 : 0u);
    ++n_staged;
    if (lane == 0) {
        if (NBUF == 2)
            bulk_wait_read_all_but_one();
        else
            bulk_wait_read_all();
    }
    __syncwarp();
    uint4 *st = reinterpret_cast<uint4 *>(stage + lane * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) st[c ^ (lane & 7)] = w[c];
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (row0 < M && col0 < N) tma_store_3d(tm_c, stage, col0, row0, batch);
        bulk_commit();
    }
}

// act(alpha * v + beta * cold + b) for four values, the activation's branch
// taken once for all four so that their chains interleave (a branch per value
// makes the four run one after another).
__device__ __forceinline__ void epi_values4(float (&v)[4], const HgemmArgs &p, const float (&cold)[4],
                                            const float (&b)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = p.alpha * v[i];
        if (p.beta != 0.f) v[i] = fmaf(p.beta, cold[i], v[i]);
        v[i] += b[i];
    }
    if (p.act == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = gelu_erf(v[i]);
    } else if (p.act == 3) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = gelu_tanh(v[i]);
    } else if (p.act == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = fmaxf(v[i], 0.f);
    }
}

// Transposed tile, this thread owning column gn of C: rows ch * 32 + j of C
// (j < 32, below M) get act(alpha * v[j] + beta * C + bias), four rows at a
// time through epi_values4.
__device__ __forceinline__ void store_col_rows32(const float (&v)[32], const HgemmArgs &p, int ch, int gn,
                                                 size_t cbase, float b_n) {
    const float b4[4] = {b_n, b_n, b_n, b_n};
#pragma unroll
    for (int j4 = 0; j4 < 32; j4 += 4) {
        if (ch * 32 + j4 >= p.M) break;  // rows m grow with j
        float w[4], cold[4];
        size_t ci[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gm = ch * 32 + j4 + i;
            ci[i] = cbase + static_cast<size_t>(gm) * p.ldc + gn;
            cold[i] = (p.beta != 0.f && gm < p.M) ? load_out(p.C, ci[i], p.c_type) : 0.f;
            w[i] = v[j4 + i];
        }
        epi_values4(w, p, cold, b4);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (ch * 32 + j4 + i < p.M) store_c(p, ci[i], w[i]);
    }
}

// Cluster split-K of the transposed small-M product: CTA `c.split` sums tile
// row rr = split * R + et % R (R = 128 / NSP; column n of C) of the NSP
// partials ([accumulator column][row] in each CTA's shared memory), in split
// order, over the accumulator columns g + NSP * jj (rows m of C; g = et / R,
// jj < NCOL = BN / NSP) that are below M: the columns are dealt round-robin
// so that every warp has the same share of the real rows of C when M is
// below the MMA's padded N.  Then it releases the partials (every CTA's
// "consumed" barrier) and writes act(alpha * sum + beta * C + bias), four
// columns per trip of a rolled loop: four independent epilogue chains per
// trip hide each other's latency (a trip per column measured 1.3 us for 8
// columns at 16 x 4096 x 4096), while the rolled loop keeps the code that
// each CTA fetches once short.
template <int BN, int NSP>
__device__ __forceinline__ void swap_csplit_reduce(const HgemmArgs &p, const UnitCoord &c, uint32_t part_addr,
                                                   uint32_t consumed_addr, size_t cbase, int et, float b_n) {
    constexpr int R = kBM / NSP, NCOL = BN / NSP;
    static_assert(kBM % NSP == 0 && BN % NSP == 0 && NCOL % 4 == 0, "power-of-two cluster sizes");
    static_assert(kEpiWarps * 32 / R == NSP, "one column group per split");
    const int rr = c.split * R + et % R;
    const int g = et / R;
    // every source's loads in flight before the first add (one remote latency)
    float t[NSP][NCOL];
#pragma unroll
    for (int src = 0; src < NSP; ++src) {
        const uint32_t base = mapa_shared(part_addr, src) + static_cast<uint32_t>(g * kBM + rr) * 4u;
#pragma unroll
        for (int jj = 0; jj < NCOL; ++jj)
            t[src][jj] = g + NSP * jj < p.M ? ld_shared_cluster_f32(base + jj * NSP * kBM * 4) : 0.f;
    }
    float acc[NCOL];
#pragma unroll
    for (int jj = 0; jj < NCOL; ++jj) {
        acc[jj] = t[0][jj];
#pragma unroll
        for (int src = 1; src < NSP; ++src) acc[jj] += t[src][jj];
    }
    // one arrival per warp on each CTA's barrier (lane r -> CTA r), after
    // the warp's loads (the warp barrier orders them before the release)
    __syncwarp();
    if ((threadIdx.x & 31) < NSP) mbar_arrive_cluster(mapa_shared(consumed_addr, threadIdx.x & 31));
    const int gn = c.n0 + rr;
    if (gn >= p.N) return;
    // the values rotate through acc[0..3], four register moves per column
#pragma unroll 1
    for (int j4 = 0; j4 < NCOL && g + NSP * j4 < p.M; j4 += 4) {
        float v[4], cold[4];
        size_t ci[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = acc[i];
            ci[i] = cbase + static_cast<size_t>(g + NSP * (j4 + i)) * p.ldc + gn;
            cold[i] = (p.beta != 0.f && g + NSP * (j4 + i) < p.M) ? load_out(p.C, ci[i], p.c_type) : 0.f;
        }
#pragma unroll
        for (int i = 0; i + 4 < NCOL; ++i) acc[i] = acc[i + 4];
        const float b4[4] = {b_n, b_n, b_n, b_n};
        epi_values4(v, p, cold, b4);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (g + NSP * (j4 + i) < p.M) store_c(p, ci[i], v[i]);
    }
}

// Cluster split-K, not transposed: CTA `c.split` of the cluster sums rows
// [r0, r1) = [split * 128 / NSP, (split + 1) * 128 / NSP) of the NSP partial
// tiles (row-major, chunk-swizzled as written by the epilogue) in split order
// and writes act(alpha * sum + beta * C + bias).  The 128 epilogue threads
// take consecutive 4-column groups (coalesced C accesses) in a rolled loop
// that keeps the next group's remote loads in flight while it finishes the
// current one: this runs once per CTA, and unrolled straight-line code spent
// more time in instruction fetch than in the work.  `sbias` holds the
// tile's bias slice (shared memory).
template <int BN, int NSP>
__device__ __forceinline__ void csplit_reduce_rows(const HgemmArgs &p, const UnitCoord &c, uint32_t part_addr,
                                                   size_t cbase, int et, const float *sbias) {
    constexpr int kGroups = BN / 4;
    constexpr int kStep = kEpiWarps * 32;
    const int r0 = c.split * kBM / NSP, r1 = (c.split + 1) * kBM / NSP;
    const int total = (r1 - r0) * kGroups;
    // the own partial through ordinary shared loads (the cluster path carries
    // only ~16 B per clock per SM), the peers' through distributed shared memory
    uint32_t base[NSP];
#pragma unroll
    for (int sidx = 0; sidx < NSP; ++sidx) base[sidx] = mapa_shared(part_addr, sidx);
    const int own = c.split;
    auto load_part = [&](int sidx, uint32_t off) -> float4 {
        if (sidx == own) {
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                         : "r"(part_addr + off)
                         : "memory");
            return v;
        }
        return ld_shared_cluster_v4(base[sidx] + off);
    };
    auto offset = [&](int e) {
        const int row = r0 + e / kGroups, g = e % kGroups;
        return static_cast<uint32_t>(row * BN + (g >> 3) * 32 + (((g & 7) ^ (row & 7)) << 2)) * 4u;
    };
    float4 nxt[NSP];
    if (et < total) {
        const uint32_t off = offset(et);
#pragma unroll
        for (int sidx = 0; sidx < NSP; ++sidx) nxt[sidx] = load_part(sidx, off);
    }
#pragma unroll 1
    for (int e = et; e < total; e += kStep) {
        float4 cur[NSP];
#pragma unroll
        for (int sidx = 0; sidx < NSP; ++sidx) cur[sidx] = nxt[sidx];
        if (e + kStep < total) {
            const uint32_t off = offset(e + kStep);
#pragma unroll
            for (int sidx = 0; sidx < NSP; ++sidx) nxt[sidx] = load_part(sidx, off);
        }
        float v[4] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w};
#pragma unroll
        for (int sidx = 1; sidx < NSP; ++sidx) {
            v[0] += cur[sidx].x;
            v[1] += cur[sidx].y;
            v[2] += cur[sidx].z;
            v[3] += cur[sidx].w;
        }
        const int row = r0 + e / kGroups, g = e % kGroups;
        const int gm = c.m0 + row, gn = c.n0 + 4 * g;
        if (gm >= p.M || gn >= p.N) continue;  // N % 8 == 0: the whole group is inside
        const size_t ci = cbase + static_cast<size_t>(gm) * p.ldc + gn;
        float cold[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.beta != 0.f) {
            if (p.c_type == kOutF32) {
                const float4 c4 = *reinterpret_cast<const float4 *>(static_cast<const float *>(p.C) + ci);
                cold[0] = c4.x, cold[1] = c4.y, cold[2] = c4.z, cold[3] = c4.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) cold[i] = load_out(p.C, ci + i, p.c_type);
            }
        }
        float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.bias) b4 = *reinterpret_cast<const float4 *>(sbias + 4 * g);
        const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
        epi_values4(v, p, cold, bv);
        if (!debug_in_bounds(p.c_extent == 0 || ci + 4 <= p.c_extent, p.err)) continue;
        if (p.c_type == kOutF32) {
            *reinterpret_cast<float4 *>(static_cast<float *>(p.C) + ci) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            uint2 w;
            w.x = pack2_out16(v[0], v[1], p.c_type);
            w.y = pack2_out16(v[2], v[3], p.c_type);
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.C) + ci) = w;
        }
    }
}

template <int BN, int STAGES, bool SWAP, bool CSPLIT, int EPI = 4>
__global__ void __launch_bounds__(64 + 32 * EPI, 1)
    hgemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_c, const HgemmArgs p) {
    using Cfg = HgemmCfg<BN, STAGES, SWAP, CSPLIT, EPI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                                 // STAGES x 16 KB (MMA operand A)
    uint8_t *sB = smem + STAGES * Cfg::kABytes;         // STAGES x kBBytes (MMA operand B)
    uint8_t *sC = sB + STAGES * Cfg::kBBytes;           // 4 x 4 KB epilogue staging
    uint64_t *bars = reinterpret_cast<uint64_t *>(sC + Cfg::kCStageBytes);
    uint64_t *full = bars;                              // TMA -> MMA, per stage
    uint64_t *empty = bars + STAGES;                    // MMA -> TMA, per stage
    uint64_t *tfull = bars + 2 * STAGES;                // MMA -> epilogue, per accumulator
    uint64_t *tempty = bars + 2 * STAGES + 2;           // epilogue -> MMA, per accumulator
    uint64_t *mma_done = bars + 2 * STAGES + 4;
    uint64_t *part_ready = bars + 2 * STAGES + 5;     // CSPLIT: every CTA's partial written
    uint64_t *part_consumed = bars + 2 * STAGES + 6;  // CSPLIT: every CTA has read this partial
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 7);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kBnTile = SWAP ? kBM : BN;  // columns of C per tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], EPI);
        }
        mbar_init(mma_done, 1);
        if (CSPLIT) {
            mbar_init(part_ready, p.splits * kEpiWarps);  // one arrival per epilogue warp of each CTA
            mbar_init(part_consumed, p.splits * kEpiWarps);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        if (!SWAP && !CSPLIT) tma_prefetch_desc(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    if (CSPLIT)
        cluster_sync();  // every CTA's hand-over barriers exist before any remote arrive
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Everything above (barriers, tensor memory, descriptor prefetch) may
    // overlap the previous kernel of the stream, and so may each role's work
    // up to its first global-memory access: the producer waits for the
    // previous kernel (pdl_wait) just before its first TMA load, the epilogue
    // warps before their first load; the MMA warp touches no global memory.
    pdl_launch_dependents();

    uint32_t armed = 0, armed_parity = 0;  // producer bookkeeping for the final drain

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        // bytes per stage: a K-major B tile is BN rows, an MN-major one whole boxes
        const uint32_t stage_tx = (!SWAP && p.b_kmajor) ? Cfg::kABytes + BN * kBK * 2 : Cfg::kStageBytes;
        int stage = 0;
        uint32_t phase = 0;
        for (int idx = 0; !*abort_flag && !p.stall_producer; ++idx) {
            UnitCoord c;
            if ((Cfg::kPartInRing && idx > 0) || !next_unit(p, idx, kBnTile, SWAP, c)) break;
            for (int kb = c.kb0; kb < c.kb1; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], stage_tx);
                if (idx == 0 && kb == c.kb0) pdl_wait();  // the operands may come from the previous kernel
                const int k0 = kb * kBK;
                uint8_t *a_dst = sA + stage * Cfg::kABytes;
                uint8_t *b_dst = sB + stage * Cfg::kBBytes;
                const int za = c.batch * p.za, zb = c.batch * p.zb;
                if constexpr (!SWAP) {
                    tma_load_3d(&tm_a, &full[stage], a_dst, k0, c.m0, za);
                    if (p.b_kmajor) {
                        tma_load_3d(&tm_b, &full[stage], b_dst, k0, c.n0, zb);  // BN rows of 64 k
                    } else {
#pragma unroll
                        for (int j = 0; j < (BN + 63) / 64; ++j)
                            tma_load_3d(&tm_b, &full[stage], b_dst + j * 8192, c.n0 + 64 * j, k0, zb);
                    }
                } else {
                    // MMA operand A = B^T (N rows; MN-major, or K-major when B
                    // is stored N x K), operand B = A (M rows, K-major).
                    if (p.b_kmajor) {
                        tma_load_3d(&tm_b, &full[stage], a_dst, k0, c.n0, zb);
                    } else {
                        tma_load_3d(&tm_b, &full[stage], a_dst, c.n0, k0, zb);
                        tma_load_3d(&tm_b, &full[stage], a_dst + 8192, c.n0 + 64, k0, zb);
                    }
                    tma_load_3d(&tm_a, &full[stage], b_dst, k0, 0, za);
                }
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                // GEMM11_DEBUG builds keep one stage in flight: the next load
                // waits until the MMA has consumed this one.  (Not in cluster
                // split-K, whose peers read each other's shared memory: its
                // pipeline keeps its depth.)
                if (kDebugBuild && !CSPLIT && !mbar_wait(&empty[stage], phase, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    break;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        // Shared-memory descriptors of stage 0; later stages and k steps only
        // move the 14-bit start-address field (address / 16, below 2^14 for
        // any shared-memory address), so the loop adds small constants.
        const uint64_t k_desc0 = umma_desc_sw128(smem_u32(SWAP ? sB : sA), 16, 1024);  // K-major operand
        const uint64_t o_desc0 = p.b_kmajor ? umma_desc_sw128(smem_u32(SWAP ? sA : sB), 16, 1024)
                                            : umma_desc_sw128(smem_u32(SWAP ? sA : sB), 8192, 1024);
        constexpr uint32_t k_stage = (SWAP ? Cfg::kBBytes : Cfg::kABytes) >> 4;
        constexpr uint32_t o_stage = (SWAP ? Cfg::kABytes : Cfg::kBBytes) >> 4;
        const uint32_t o_kstep = p.b_kmajor ? 2u : 128u;  // 32 B (K-major) or 2048 B (MN-major) per k16
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        for (int idx = 0; !*abort_flag; ++idx, ++local) {
            UnitCoord c;
            if ((Cfg::kPartInRing && idx > 0) || !next_unit(p, idx, kBnTile, SWAP, c)) break;
            const int buf = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(&tempty[buf], acc_phase ^ 1u, p.wait_ns)) {
                flag_timeout(abort_flag, p.err);
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
            bool ok = true;
            for (int kb = c.kb0; kb < c.kb1; ++kb) {
                if (!mbar_wait(&full[stage], phase, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t kd = k_desc0 + stage * k_stage;
                const uint64_t od = o_desc0 + stage * o_stage;
#pragma unroll
                for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                    const uint64_t kdesc = kd + 2u * kk;  // K-major: +32 B per k16
                    const uint64_t odesc = od + o_kstep * kk;
                    const uint64_t adesc = SWAP ? odesc : kdesc;
                    const uint64_t bdesc = SWAP ? kdesc : odesc;
                    umma_f16(d_tmem, adesc, bdesc, p.idesc, (kb > c.kb0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(&tfull[buf]);  // accumulator complete
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue warps
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row_in_tile = q * 32 + lane;
        // Four warps: two 4 KB staging buffers per warp used alternately
        // (running chunk count), so a chunk's shared-memory writes only wait
        // for the TMA store issued two chunks earlier.  Eight warps: one
        // buffer each, and warp half h takes the chunks ch = h (mod 2).
        const int ch_first = (warp - 2) >> 2, ch_step = EPI / 4;
        uint8_t *const stage_base = sC + (warp - 2) * (Cfg::kNBuf * 4096);
        uint32_t n_staged = 0;
        int local = 0;
        pdl_wait();  // before the first bias, C or scratch access
        for (int idx = 0; !*abort_flag; ++idx, ++local) {
            UnitCoord c;
            if ((Cfg::kPartInRing && idx > 0) || !next_unit(p, idx, kBnTile, SWAP, c)) break;
            const int buf = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            // The unit's bias, loaded while its main loop runs: per lane and
            // chunk (not transposed), this thread's column n (transposed), or
            // the tile's slice in shared memory (cluster split, not transposed).
            float blane[(BN / 32 + EPI / 4 - 1) / (EPI / 4)];
            float b_n = 0.f;
            float *const sbias = reinterpret_cast<float *>(sC);
            const int et = threadIdx.x - 64;  // epilogue thread 0..127
            if constexpr (Cfg::kPartInRing) {
                if (p.bias)
                    for (int j = et; j < BN; j += kEpiWarps * 32)
                        sbias[j] = c.n0 + j < p.N ? __ldg(p.bias + c.n0 + j) : 0.f;
            } else if constexpr (CSPLIT) {
                const int gn = c.n0 + c.split * (kBM / p.splits) + et % (kBM / p.splits);
                b_n = (p.bias && gn < p.N) ? __ldg(p.bias + gn) : 0.f;
            } else if constexpr (SWAP) {
                const int gn = c.n0 + row_in_tile;
                b_n = (p.bias && gn < p.N) ? __ldg(p.bias + gn) : 0.f;
            } else {
                load_bias_lanes(p, c.n0, lane, [&](int i) { return ch_first + i * ch_step; }, blane);
            }
            if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns)) {
                flag_timeout(abort_flag, p.err);
                break;
            }
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
            // Pass 1: TMEM -> registers.  Either the finished epilogue (no split)
            // or the raw partial to scratch (K split over CTAs, splits > 1).
            const size_t cbase = static_cast<size_t>(c.batch) * static_cast<size_t>(p.stride_c);
            if constexpr (Cfg::kPartInRing) {
                // 1. this CTA's partial -> the idle operand ring, [row][column]
                //    with the 16-byte chunks of each 32-column group swizzled by
                //    the row (chunk c of row r at c ^ (r & 7)): conflict-free
                //    writes per quarter warp, and each reader walks one row.
                //    The next chunk's tensor-memory load is in flight while
                //    this one is written.
                float *part = reinterpret_cast<float *>(sA);
                fence_proxy_async_smem();  // after the async-proxy (TMA, MMA) use of the ring
                auto put = [&](const uint32_t (&r)[32], int ch) {
                    float4 *dst = reinterpret_cast<float4 *>(part + row_in_tile * BN + ch * 32);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4)
                        dst[c4 ^ (row_in_tile & 7)] =
                            make_float4(__uint_as_float(r[4 * c4]), __uint_as_float(r[4 * c4 + 1]),
                                        __uint_as_float(r[4 * c4 + 2]), __uint_as_float(r[4 * c4 + 3]));
                };
                {
                    uint32_t ra[32], rb[32];
                    tmem_ld_32x32b_x32(t_row, ra);
                    tmem_wait_ld();
#pragma unroll
                    for (int ch = 0; ch < BN / 32; ch += 2) {
                        tmem_ld_32x32b_x32(t_row + (ch + 1) * 32, rb);
                        put(ra, ch);
                        tmem_wait_ld();
                        if (ch + 2 < BN / 32) tmem_ld_32x32b_x32(t_row + (ch + 2) * 32, ra);
                        put(rb, ch + 1);
                        tmem_wait_ld();
                    }
                }
                tc_fence_before();
                __syncwarp();  // also orders the warp's partial (and bias) writes before the arrivals
                if (lane == 0) mbar_arrive(&tempty[buf]);
                const int nsp = p.splits;
                if (lane < nsp) mbar_arrive_cluster(mapa_shared(smem_u32(part_ready), lane));
                if (!mbar_wait_cluster(part_ready, 0, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    break;
                }
                // 2. rows [r0, r1) of the tile, summed over the partials in split order
                switch (nsp) {
                    case 2: csplit_reduce_rows<BN, 2>(p, c, smem_u32(part), cbase, et, sbias); break;
                    case 3: csplit_reduce_rows<BN, 3>(p, c, smem_u32(part), cbase, et, sbias); break;
                    case 4: csplit_reduce_rows<BN, 4>(p, c, smem_u32(part), cbase, et, sbias); break;
                    case 5: csplit_reduce_rows<BN, 5>(p, c, smem_u32(part), cbase, et, sbias); break;
                    case 6: csplit_reduce_rows<BN, 6>(p, c, smem_u32(part), cbase, et, sbias); break;
                    case 7: csplit_reduce_rows<BN, 7>(p, c, smem_u32(part), cbase, et, sbias); break;
                    default: csplit_reduce_rows<BN, 8>(p, c, smem_u32(part), cbase, et, sbias); break;
                }
                __syncwarp();
                if (lane < nsp) mbar_arrive_cluster(mapa_shared(smem_u32(part_consumed), lane));
                continue;
            }
            if constexpr (CSPLIT) {
                // 1. this CTA's partial -> own shared memory, [column][row]
                float *part = reinterpret_cast<float *>(sC);
                if (local > 0 && !mbar_wait_cluster(part_consumed, (local - 1) & 1, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    break;
                }
#pragma unroll 1
                for (int ch = 0; ch < BN / 32 && ch * 32 < p.M; ++ch) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + ch * 32, r);
                    tmem_wait_ld();
                    // columns at or past M (the MMA's padding) are never read
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (ch * 32 + j < p.M) part[(ch * 32 + j) * kBM + row_in_tile] = __uint_as_float(r[j]);
                }
                tc_fence_before();
                __syncwarp();  // also orders the warp's partial writes before the arrivals
                if (lane == 0) mbar_arrive(&tempty[buf]);
                const int nsp = p.splits;
                if (lane < nsp) mbar_arrive_cluster(mapa_shared(smem_u32(part_ready), lane));
                // 2. rows [rank * R, rank * R + R) of the sum of all partials, in split order
                if (!mbar_wait_cluster(part_ready, local & 1, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    break;
                }
                // sizes 2, 4 or 8 (the planner's powers of two)
                if (nsp == 2)
                    swap_csplit_reduce<BN, 2>(p, c, smem_u32(part), smem_u32(part_consumed), cbase, et, b_n);
                else if (nsp == 4)
                    swap_csplit_reduce<BN, 4>(p, c, smem_u32(part), smem_u32(part_consumed), cbase, et, b_n);
                else
                    swap_csplit_reduce<BN, 8>(p, c, smem_u32(part), smem_u32(part_consumed), cbase, et, b_n);
                continue;
            }
            bool partial = EPI == 4 && p.splits > 1;  // the planner splits only with 4 warps
            float *part = nullptr;
            if (partial) part = p.ws + (static_cast<size_t>(c.tile) * p.splits + c.split) * (kBM * BN);
            // debug builds: a slot outside the scratch is neither written nor counted
            const bool part_ok =
                !partial || debug_in_bounds(p.ws_floats == 0 ||
                                                (static_cast<size_t>(c.tile) * p.splits + c.split + 1) * (kBM * BN) <=
                                                    p.ws_floats,
                                            p.err);
#pragma unroll 1
            for (int ch = ch_first; ch < BN / 32; ch += ch_step) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + ch * 32, r);
                tmem_wait_ld();
                if (partial) {
                    if (!part_ok) continue;
                    // scratch layout per unit: [chunk][column j][row 0..127] -> coalesced
                    float *dst = part + ch * 32 * kBM + row_in_tile;
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[j * kBM] = __uint_as_float(r[j]);
                    continue;
                }
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                if constexpr (!SWAP) {
                    const int grow = c.m0 + row_in_tile;
                    const int col0 = c.n0 + ch * 32;
                    epilogue_row_chunk(v, p, grow, col0, cbase, blane[0]);
                    rotate_bias_lanes(blane);
                    store_row_chunk<Cfg::kNBuf>(v, p, &tm_c, stage_base, n_staged, lane, c.m0 + q * 32, col0, c.batch);
                } else {
                    // transposed: this thread owns column n of C, registers walk rows m
                    const int gn = c.n0 + row_in_tile;
                    if (gn < p.N) store_col_rows32(v, p, ch, gn, cbase, b_n);
                }
            }
            // Accumulator buffer free for the MMA warp.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);

            if (partial && part_ok) {
                // The last contributor to arrive on this 32-row slice of the
                // tile adds all contributions in k order (split index).
                const int n_contrib = p.splits;
                const int cnt_idx = c.tile * 4 + q;
                __threadfence();
                __syncwarp();
                unsigned last = 0;
                if (lane == 0) last = atomicAdd(&p.counters[cnt_idx], 1u) == static_cast<unsigned>(n_contrib - 1);
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    auto contrib = [&](int i) -> const float * {
                        return p.ws + (static_cast<size_t>(c.tile) * p.splits + i) * (kBM * BN);
                    };
#pragma unroll 1
                    for (int ch = 0; ch < BN / 32; ++ch) {
                        // Two contributions (64 loads) in flight per round, added in
                        // k order: a reduction over n partials costs ~n/2 round trips.
                        float v[32];
                        {
                            const float *s0 = contrib(0) + ch * 32 * kBM + row_in_tile;
                            if (n_contrib > 1) {
                                const float *s1 = contrib(1) + ch * 32 * kBM + row_in_tile;
                                float t[32];
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    v[j] = __ldcg(s0 + j * kBM);
                                    t[j] = __ldcg(s1 + j * kBM);
                                }
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] += t[j];
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = __ldcg(s0 + j * kBM);
                            }
                        }
                        for (int s = 2; s < n_contrib; s += 2) {
                            const float *sa = contrib(s) + ch * 32 * kBM + row_in_tile;
                            float t0[32], t1[32];
                            const bool two = s + 1 < n_contrib;
                            const float *sb = two ? contrib(s + 1) + ch * 32 * kBM + row_in_tile : sa;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                t0[j] = __ldcg(sa + j * kBM);
                                t1[j] = two ? __ldcg(sb + j * kBM) : 0.f;
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] += t0[j];
                            if (two)
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] += t1[j];
                        }
                        if constexpr (!SWAP) {
                            const int grow = c.m0 + row_in_tile;
                            const int col0 = c.n0 + ch * 32;
                            epilogue_row_chunk(v, p, grow, col0, cbase, blane[0]);
                            rotate_bias_lanes(blane);
                            store_row_chunk<Cfg::kNBuf>(v, p, &tm_c, stage_base, n_staged, lane, c.m0 + q * 32, col0, c.batch);
                        } else {
                            const int gn = c.n0 + row_in_tile;
                            if (gn < p.N) store_col_rows32(v, p, ch, gn, cbase, b_n);
                        }
                    }
                    if (lane == 0) p.counters[cnt_idx] = 0u;
                }
            }
        }
        if (CSPLIT && local > 0 && !*abort_flag) {
            // the peers must have read this CTA's last partial before it exits
            if (!mbar_wait_cluster(part_consumed, (local - 1) & 1, p.wait_ns)) flag_timeout(abort_flag, p.err);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------- drain and unwind
    if (warp == 0 && lane == 0) {
        // every TMA copy this CTA issued must have landed before it exits
        for (int s = 0; s < STAGES; ++s)
            if (armed & (1u << s))
                if (!mbar_wait(&full[s], (armed_parity >> s) & 1u, p.wait_ns)) flag_timeout(abort_flag, p.err);
    }
    if (warp == 1 && lane == 0) {
        umma_commit(mma_done);  // completes when all MMAs issued above have finished
        if (!mbar_wait(mma_done, 0, p.wait_ns)) flag_timeout(abort_flag, p.err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
// Same roles as hgemm_tc_kernel, on a cluster of two CTAs on neighbouring
// SMs that compute one 256 x BN tile together with tcgen05.mma.cta_group::2:
// CTA r stages A rows [m0 + 128r, +128) and B columns [n0 + r*BN/2, +BN/2)
// in its own shared memory; the even CTA's MMA thread multiplies the pair
// (each SM's tensor core reads its own A rows and both halves of B) and the
// accumulator rows land in each CTA's own tensor memory.  Per SM this moves
// half the B bytes of the single-CTA 128 x BN tile for the same MMA work.
// Barriers: each CTA's TMA loads count on the even CTA's "full" barrier;
// the MMA thread's commits arrive on both CTAs' "empty" and "accumulator
// full" barriers (multicast); both CTAs' epilogue warps arrive on the even
// CTA's "accumulator empty" barrier.
// X3: FP32-accuracy mode.  A and B arrive split into TF32 high and low parts
// (A_hi + A_lo, B_hi + B_lo, B stored N x K); each stage holds both parts of
// both operands, 32 k per 128-byte row, and the MMA thread issues
// A_lo B_hi + A_hi B_lo + A_hi B_hi (kind::tf32) per k step.
template <int BN, int STAGES, int EPI, bool X3 = false>
struct HgemmPairCfg {
    static constexpr int kNBuf = EPI == 4 ? 2 : 1;    // 4 KB staging buffers per epilogue warp
    static constexpr int kThreadsPair = 64 + 32 * EPI;
    static constexpr int kKB = X3 ? 32 : kBK;      // k per stage: one 128-byte swizzle row
    static constexpr int kABytes = kBM * 128;      // this CTA's 128 rows (one part)
    static constexpr int kBHalf = BN / 2;          // this CTA's columns of B
    static constexpr int kBBoxes = (kBHalf + 63) / 64;
    static constexpr int kBBytes = X3 ? kBHalf * 128 : kBBoxes * 64 * kBK * 2;  // one part
    static constexpr int kParts = X3 ? 2 : 1;
    static constexpr int kAStage = kParts * kABytes;
    static constexpr int kBStage = kParts * kBBytes;
    static constexpr int kStageBytes = kAStage + kBStage;
    static constexpr int kCStageBytes = EPI * kNBuf * 32 * 32 * 4;
    static constexpr int kBarBytes = (2 * STAGES + 5) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kCStageBytes + kBarBytes;
    static constexpr int kTmemCols = tmem_cols_for(BN);
    static_assert(BN % 32 == 0 && BN <= 256 && kBHalf % 16 == 0, "pair MMA N");
    static_assert(EPI == 4 || EPI == 8, "epilogue warps");
    static_assert(STAGES <= 8, "stage bookkeeping uses 8-bit masks");
    static_assert(kBBytes % 1024 == 0, "operand tiles stay 1024-byte aligned");
};

// Pair tile t (over the whole batch) -> (matrix index, first row of the
// pair, first column), grouped raster of 4 pair rows per sweep over N.
__device__ __forceinline__ void pair_tile_origin(const HgemmArgs &p, int t, int bn, int &m0, int &n0, int &batch) {
    const int per = p.tiles_m * p.tiles_n;
    batch = t / per;
    t -= batch * per;
    const int group_tiles = 4 * p.tiles_n;
    const int first_m = (t / group_tiles) * 4;
    const int gsz = min(p.tiles_m - first_m, 4);
    m0 = (first_m + (t % group_tiles) % gsz) * (2 * kBM);
    n0 = ((t % group_tiles) / gsz) * bn;
}

template <int BN, int STAGES, int EPI, bool X3>
__global__ void __launch_bounds__(64 + 32 * EPI, 1)
    hgemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_a2,
                         const __grid_constant__ CUtensorMap tm_b2, const HgemmArgs p) {
    using Cfg = HgemmPairCfg<BN, STAGES, EPI, X3>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                               // STAGES x kAStage (A, or A_hi | A_lo)
    uint8_t *sB = smem + STAGES * Cfg::kAStage;       // STAGES x kBStage (B, or B_hi | B_lo)
    uint8_t *sC = sB + STAGES * Cfg::kBStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sC + Cfg::kCStageBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = bars + 2 * STAGES + 2;
    uint64_t *mma_done = bars + 2 * STAGES + 4;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cid = blockIdx.x >> 1;
    const int ncl = gridDim.x >> 1;
    // Bytes each CTA stages per k block: its A rows and its half of B (64-column
    // boxes when B is K x N; exactly BN/2 rows of 64 k when B is N x K); both
    // parts of each in the FP32-accuracy mode.
    const uint32_t stage_tx =
        X3 ? Cfg::kStageBytes : Cfg::kABytes + (p.b_kmajor ? Cfg::kBHalf * kBK * 2 : Cfg::kBBytes);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * EPI);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_c);
        if (X3) {
            tma_prefetch_desc(&tm_a2);
            tma_prefetch_desc(&tm_b2);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Everything above (barriers, tensor memory, descriptor prefetch) may
    // overlap the previous kernel of the stream; global memory only below.
    pdl_wait();
    pdl_launch_dependents();

    uint32_t armed = 0, armed_parity = 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        int stage = 0;
        uint32_t phase = 0;
        for (int t = cid; t < p.units && !*abort_flag; t += ncl) {
            int m0, n0, bz;
            pair_tile_origin(p, t, BN, m0, n0, bz);
            const int my_m = m0 + static_cast<int>(rank) * kBM;
            const int my_n = n0 + static_cast<int>(rank) * Cfg::kBHalf;
            const int za = bz * p.za, zb = bz * p.zb;
            bool ok = true;
            for (int kb = 0; kb < p.kb_total; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                    flag_timeout(abort_flag, p.err);
                    ok = false;
                    break;
                }
                if (leader) mbar_arrive_expect_tx(&full[stage], 2 * stage_tx);
                const uint32_t full_even = mapa_shared(smem_u32(&full[stage]), 0);
                const int k0 = kb * Cfg::kKB;
                uint8_t *a_dst = sA + stage * Cfg::kAStage;
                uint8_t *b_dst = sB + stage * Cfg::kBStage;
                tma_load_3d_pair(&tm_a, full_even, a_dst, k0, my_m, za);
                if constexpr (X3) {
                    tma_load_3d_pair(&tm_a2, full_even, a_dst + Cfg::kABytes, k0, my_m, za);
                    tma_load_3d_pair(&tm_b, full_even, b_dst, k0, my_n, zb);
                    tma_load_3d_pair(&tm_b2, full_even, b_dst + Cfg::kBBytes, k0, my_n, zb);
                } else if (p.b_kmajor) {
                    tma_load_3d_pair(&tm_b, full_even, b_dst, k0, my_n, zb);
                } else {
#pragma unroll
                    for (int j = 0; j < Cfg::kBBoxes; ++j)
                        tma_load_3d_pair(&tm_b, full_even, b_dst + j * 8192, my_n + 64 * j, k0, zb);
                }
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                // GEMM11_DEBUG builds: one stage in flight (the MMA's commit
                // arrives on both CTAs' empty barriers)
                if (kDebugBuild && !mbar_wait(&empty[stage], phase, p.wait_ns)) {
                    flag_timeout(abort_flag, p.err);
                    ok = false;
                    break;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------ MMA issuer (even CTA)
        // Descriptors of stage 0, moved by address / 16 per stage and k step.
        const uint64_t a_desc0 = umma_desc_sw128(smem_u32(sA), 16, 1024);
        const bool b_kmajor = X3 || p.b_kmajor;
        const uint64_t b_desc0 = b_kmajor ? umma_desc_sw128(smem_u32(sB), 16, 1024)
                                          : umma_desc_sw128(smem_u32(sB), 8192, 1024);
        const uint32_t b_kstep = b_kmajor ? 2u : 128u;
        // The accumulator is handed to the epilogue once per tile, or in the
        // FP32-accuracy mode once per chunk of kX3ChunkKB k blocks (the epilogue
        // adds the chunks in FP32 registers).
        const int kb_chunk = X3 ? kX3ChunkKB : p.kb_total;
        const int nch = (p.kb_total + kb_chunk - 1) / kb_chunk;
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int t = cid; ok && t < p.units && !*abort_flag; t += ncl) {
            for (int c = 0; c < nch; ++c, ++local) {
                const int buf = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(&tempty[buf], acc_phase ^ 1u)) {
                    flag_timeout(abort_flag, p.err);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                const int kb0 = c * kb_chunk, kb1 = min(p.kb_total, kb0 + kb_chunk);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase)) {
                        flag_timeout(abort_flag, p.err);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + stage * (Cfg::kAStage >> 4);
                    const uint64_t bd = b_desc0 + stage * (Cfg::kBStage >> 4);
                    if constexpr (X3) {
                        // small products first: A_lo B_hi, A_hi B_lo, then A_hi B_hi (K = 8 each)
                        const uint64_t al = ad + (Cfg::kABytes >> 4), bl = bd + (Cfg::kBBytes >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            umma_tf32_pair(d_tmem, al + 2u * kk, bd + 2u * kk, p.idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                            umma_tf32_pair(d_tmem, ad + 2u * kk, bl + 2u * kk, p.idesc, 1u);
                            umma_tf32_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, p.idesc, 1u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk)
                            umma_f16_pair(d_tmem, ad + 2u * kk, bd + b_kstep * kk, p.idesc,
                                          (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit_pair_mc(&empty[stage], 0x3);  // frees the stage in both CTAs
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(&tfull[buf], 0x3);  // both halves of the accumulator complete
            }
        }
    } else if (X3 && warp >= 2) {
        // ------------------------------------------------ epilogue, FP32-accuracy mode
        // Eight warps: warp w reads TMEM lane quarter w % 4 and owns 4 of the
        // 8 column groups of its rows ((w - 2) / 4 selects which), keeping
        // their running sums in registers.  Each chunk accumulator (kX3ChunkKB
        // k blocks, summed by the tensor core) is added in FP32 with
        // round-to-nearest; the tensor core's own accumulation is truncated,
        // so keeping its sums short keeps the total within FP32's error level
        // for any K.
        static_assert(!X3 || (EPI == 8 && BN / 32 <= 8), "FP32-accuracy mode: 8 epilogue warps, <= 256 columns");
        constexpr int kGroups = BN / 32;  // 32-column groups of a tile; warp half h owns [4h, 4h + 4)
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        const int g0 = ((warp - 2) >> 2) * 4;  // first of this warp's 4 column groups
        uint8_t *const stage_base = sC + (warp - 2) * (Cfg::kNBuf * 4096);
        uint32_t n_staged = 0;
        const int nch = (p.kb_total + kX3ChunkKB - 1) / kX3ChunkKB;
        int local = 0;
        bool ok = true;
        for (int t = cid; ok && t < p.units && !*abort_flag; t += ncl) {
            int m0, n0, bz;
            pair_tile_origin(p, t, BN, m0, n0, bz);
            const int my_m = m0 + static_cast<int>(rank) * kBM;
            const size_t cbase = static_cast<size_t>(bz) * static_cast<size_t>(p.stride_c);
            float tot[4][32];
            for (int c = 0; c < nch; ++c, ++local) {
                const int buf = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(&tfull[buf], acc_phase)) {
                    flag_timeout(abort_flag, p.err);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_row =
                    tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
#pragma unroll
                for (int gh = 0; gh < 8; ++gh) {  // half groups of 16 columns (fewer live registers)
                    const int gi = gh >> 1, j0 = (gh & 1) * 16;
                    if (g0 + gi >= kGroups) continue;
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(t_row + (g0 + gi) * 32 + j0, r);
                    tmem_wait_ld();
                    if (c == 0) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) tot[gi][j0 + j] = __uint_as_float(r[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) tot[gi][j0 + j] += __uint_as_float(r[j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        mbar_arrive(&tempty[buf]);
                    else
                        mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
                }
            }
            if (!ok) break;
            const int grow = my_m + row_in_tile;
            float blane[4];  // loaded here: the running sums hold most registers during the loop above
            load_bias_lanes(p, n0, lane, [&](int i) { return g0 + i; }, blane);
#pragma unroll
            for (int gi = 0; gi < 4; ++gi) {
                if (g0 + gi >= kGroups) continue;
                const int col0 = n0 + (g0 + gi) * 32;
                epilogue_row_chunk(tot[gi], p, grow, col0, cbase, blane[gi]);
                store_row_chunk<Cfg::kNBuf>(tot[gi], p, &tm_c, stage_base, n_staged, lane, my_m + q * 32, col0, bz);
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue warps (both CTAs)
        // Warp w reads TMEM lane quarter w % 4.  With 8 epilogue warps two
        // warps share a quarter and take alternate 32-column chunks.  Four
        // warps use two 4 KB staging buffers each, alternately (a chunk's
        // shared-memory writes only wait for the TMA store issued two chunks
        // earlier); eight warps one each.
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        const int ch_first = (warp - 2) >> 2, ch_step = EPI / 4;
        uint8_t *const stage_base = sC + (warp - 2) * (Cfg::kNBuf * 4096);
        uint32_t n_staged = 0;
        int local = 0;
        for (int t = cid; t < p.units && !*abort_flag; t += ncl, ++local) {
            int m0, n0, bz;
            pair_tile_origin(p, t, BN, m0, n0, bz);
            const int my_m = m0 + static_cast<int>(rank) * kBM;
            const size_t cbase = static_cast<size_t>(bz) * static_cast<size_t>(p.stride_c);
            const int buf = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            // bias of this warp's chunks, loaded while the tile's main loop runs
            constexpr int kStep = EPI / 4;  // ch_step
            constexpr int kNchPlain = (BN / 32 + kStep - 1) / kStep;
            constexpr int kNchUnits = 2 * ((BN / 64 + kStep - 1) / kStep);  // 64-column units, two chunks each
            constexpr int kNch = kNchPlain > kNchUnits ? kNchPlain : kNchUnits;
            float blane[kNch];
            if (p.c64)
                load_bias_lanes(p, n0, lane, [&](int i) { return 2 * (ch_first + (i >> 1) * ch_step) + (i & 1); },
                                blane);
            else
                load_bias_lanes(p, n0, lane, [&](int i) { return ch_first + i * ch_step; }, blane);
            if (!mbar_wait(&tfull[buf], acc_phase)) {
                flag_timeout(abort_flag, p.err);
                break;
            }
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
            const int grow = my_m + row_in_tile;
            if (p.c64) {
                // 16-bit C in 64-column units: two TMEM chunks per store
#pragma unroll 1
                for (int u = ch_first; u < BN / 64; u += ch_step) {
                    uint4 w[8];
                    // both chunks' tensor-memory loads in flight before one wait
                    uint32_t r2[2][32];
                    tmem_ld_32x32b_x32(t_row + (2 * u) * 32, r2[0]);
                    tmem_ld_32x32b_x32(t_row + (2 * u + 1) * 32, r2[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r2[h][j]);
                        epilogue_row_chunk(v, p, grow, n0 + (2 * u + h) * 32, cbase, blane[0]);
                        rotate_bias_lanes(blane);
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            w[h * 4 + c8].x = pack2_out16(v[8 * c8], v[8 * c8 + 1], p.c_type);
                            w[h * 4 + c8].y = pack2_out16(v[8 * c8 + 2], v[8 * c8 + 3], p.c_type);
                            w[h * 4 + c8].z = pack2_out16(v[8 * c8 + 4], v[8 * c8 + 5], p.c_type);
                            w[h * 4 + c8].w = pack2_out16(v[8 * c8 + 6], v[8 * c8 + 7], p.c_type);
                        }
                    }
                    store_row_unit64<Cfg::kNBuf>(w, &tm_c, stage_base, n_staged, lane, my_m + q * 32, n0 + u * 64, bz,
                                                 p.M, p.N);
                }
            } else {
#pragma unroll 1
                for (int ch = ch_first; ch < BN / 32; ch += ch_step) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + ch * 32, r);
                    tmem_wait_ld();
                    const int col0 = n0 + ch * 32;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    epilogue_row_chunk(v, p, grow, col0, cbase, blane[0]);
                    rotate_bias_lanes(blane);
                    store_row_chunk<Cfg::kNBuf>(v, p, &tm_c, stage_base, n_staged, lane, my_m + q * 32, col0, bz);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&tempty[buf]);
                else
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------- drain and unwind
    if (warp == 0 && lane == 0 && leader) {
        // the even CTA's full barriers count the copies of both CTAs
        for (int s = 0; s < STAGES; ++s)
            if (armed & (1u << s))
                if (!mbar_wait(&full[s], (armed_parity >> s) & 1u)) flag_timeout(abort_flag, p.err);
    }
    if (warp == 1 && lane == 0 && leader) {
        umma_commit_pair_mc(mma_done, 0x1);
        if (!mbar_wait(mma_done, 0)) flag_timeout(abort_flag, p.err);
    }
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while the pair's MMAs or copies may touch it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

// A strided batch of `depth` row-major matrices (outer rows of inner
// elements, rows row_stride apart, matrices mat_stride apart; elements).
// With depth 1 the matrix stride is unused and set to one matrix.
bool encode_3d(CUtensorMap *map, CUtensorMapDataType dt, int elem_bytes, const void *base, uint64_t inner,
               uint64_t outer, uint64_t depth, uint64_t row_stride, uint64_t mat_stride, uint32_t box_inner,
               uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto enc = get_encoder();
    if (!enc) return false;
    const uint64_t eb = static_cast<uint64_t>(elem_bytes);
    cuuint64_t dims[3] = {inner, outer, depth};
    cuuint64_t strides[2] = {row_stride * eb, (depth > 1 ? mat_stride : row_stride * outer) * eb};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Store map of C: 32 x 32 boxes; FP32 rows of the box are 128 bytes (128-byte
// swizzle), 16-bit rows 64 bytes (64-byte swizzle), matching store_row_chunk.
bool encode_c(CUtensorMap *map, const TcGemm &g, int ldc, bool c64 = false) {
    if (g.c_type == kOutF32)
        return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.C, g.N, g.M, g.batch, ldc, g.stride_c, 32, 32);
    const CUtensorMapDataType dt =
        g.c_type == kOutF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (c64)  // 32 x 64 boxes of 128-byte rows (store_row_unit64)
        return encode_3d(map, dt, 2, g.C, g.N, g.M, g.batch, ldc, g.stride_c, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    return encode_3d(map, dt, 2, g.C, g.N, g.M, g.batch, ldc, g.stride_c, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Operand maps.  A: K x M per matrix, boxes of 64 k x `rows` rows.  B stored
// K x N: boxes of 64 columns x 64 k; stored N x K: boxes of 64 k x `rows` rows.
bool encode_a(CUtensorMap *map, const TcGemm &g, CUtensorMapDataType dt, uint32_t rows) {
    return encode_3d(map, dt, 2, g.A, g.K, g.M, g.stride_a ? g.batch : 1, g.K, g.stride_a, kBK, rows);
}
bool encode_b(CUtensorMap *map, const TcGemm &g, CUtensorMapDataType dt, uint32_t rows) {
    if (g.b_trans) return encode_3d(map, dt, 2, g.B, g.K, g.N, g.stride_b ? g.batch : 1, g.K, g.stride_b, kBK, rows);
    return encode_3d(map, dt, 2, g.B, g.N, g.K, g.stride_b ? g.batch : 1, g.N, g.stride_b, 64, kBK);
}

template <int BN, int STAGES, bool SWAP, bool CSPLIT = false, int EPI = 4>
cudaError_t launch_hgemm(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const HgemmArgs &a,
                         int grid, cudaStream_t stream) {
    using Cfg = HgemmCfg<BN, STAGES, SWAP, CSPLIT, EPI>;
    auto kern = hgemm_tc_kernel<BN, STAGES, SWAP, CSPLIT, EPI>;
    static unsigned long long smem_set = 0;
    cudaError_t e = ensure_dynamic_smem(kern, Cfg::kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    // The tile's MMA shape and operand majors: A is K-major; B is MN-major
    // when stored K x N, K-major when stored N x K.  The transposed variant
    // swaps the operands (B^T first).
    HgemmArgs args = a;
    const int b_mn = a.b_kmajor ? 0 : 1;
    args.idesc = (SWAP ? umma_idesc_f16_f32(kBM, BN, b_mn, 0) : umma_idesc_f16_f32(kBM, BN, 0, b_mn)) | a.idesc_fmt;
    // Programmatic dependent launch: the prologue may overlap the previous
    // kernel (the kernel waits in pdl_wait before touching global memory);
    // with CSPLIT, clusters of `splits` CTAs, one K split each (the grid is a
    // multiple of it).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CSPLIT ? static_cast<unsigned>(a.splits) : 1u;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = CSPLIT ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, args);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

// Clusters of `cs` CTAs of hgemm_tc_kernel<BN, STAGES, false, true> that the
// GPU holds at once (cached per cluster size; one device type per process).
template <int BN, int STAGES>
int cluster_split_capacity(int cs) {
    static int cap[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};  // atomic accesses: planners may run concurrently
    if (cs < 1 || cs > 8) return 0;
    const int known = __atomic_load_n(&cap[cs], __ATOMIC_ACQUIRE);
    if (known >= 0) return known;
    using Cfg = HgemmCfg<BN, STAGES, false, true>;
    auto kern = hgemm_tc_kernel<BN, STAGES, false, true>;
    static unsigned long long smem_set = 0;
    if (ensure_dynamic_smem(kern, Cfg::kSmemBytes, smem_set) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs * device_sm_count(), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    __atomic_store_n(&cap[cs], n, __ATOMIC_RELEASE);
    return n;
}

int cluster_split_capacity_for(int bn, int cs) {
    if (bn == 256) return cluster_split_capacity<256, 4>(cs);
    if (bn == 192) return cluster_split_capacity<192, 5>(cs);
    return cluster_split_capacity<128, 6>(cs);
}

template <int BN, int STAGES, int EPI, bool X3 = false>
cudaError_t launch_hgemm_pair(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const HgemmArgs &a,
                              cudaStream_t stream, int *clusters_used, const CUtensorMap *ta2 = nullptr,
                              const CUtensorMap *tb2 = nullptr) {
    using Cfg = HgemmPairCfg<BN, STAGES, EPI, X3>;
    auto kern = hgemm_tc_pair_kernel<BN, STAGES, EPI, X3>;
    static int max_clusters = -1;  // per instantiation; one device type per process; atomic accesses
    static unsigned long long smem_set = 0;
    cudaError_t e = ensure_dynamic_smem(kern, Cfg::kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // prologue may overlap the previous kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(Cfg::kThreadsPair, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters_max = __atomic_load_n(&max_clusters, __ATOMIC_ACQUIRE);
    if (clusters_max < 0) {
        cfg.gridDim = dim3(2 * device_sm_count(), 1, 1);
        e = cudaOccupancyMaxActiveClusters(&clusters_max, kern, &cfg);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&max_clusters, clusters_max, __ATOMIC_RELEASE);
    }
    if (clusters_max < 1) return cudaErrorNotSupported;
    const int clusters = std::min(a.units, clusters_max);
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    *clusters_used = clusters;
    HgemmArgs args = a;
    args.idesc = X3 ? umma_idesc_f16_f32(2 * kBM, BN, 0, 0) | kIdescTf32Operands
                    : umma_idesc_f16_f32(2 * kBM, BN, 0, a.b_kmajor ? 0 : 1) | a.idesc_fmt;
    cfg.numAttrs = 2;  // the occupancy query above used the cluster shape alone
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, ta2 ? *ta2 : ta, tb2 ? *tb2 : tb, args);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

// Cluster split-K for few 128-row tiles (not transposed).  A time model
// fitted to GB300 measurements: a CTA streams its operand bytes at ~100 GB/s
// (the bytes each SM keeps in flight bound it, not HBM, while the SMs are
// few); a split adds ~5 us of hand-over and reduction (peers' skew, the
// barriers, the reduction loop with its epilogue) plus the partial's remote
// reads at ~30 GB/s (distributed shared memory, ~16 B per clock per SM).
// Without a tuned entry: only when whole 128 x 128 tiles leave at least half
// the SMs idle, and only when the best split beats the whole tiles by 10 %
// (128 x 4096 x 4096: 4 x 128-wide, 19.6 -> 13.6 us; 96 x 8192 x 2048 and
// 100 x 8192 x 1024 stay whole: 12.9 and 8.4 us, split 15.4 and 12.7 us).  With a tuned
// entry, its width and size (0: any) are taken if they can run.  Returns
// false when no split qualifies.
bool pick_cluster_split(int tiles_m, int N, int batch, int kb_total, int sms, const TunePlan *tp, int *bn_out,
                        int *cs_out) {
    constexpr double kStreamBps = 100e9, kRemoteBps = 30e9, kHandover = 5e-6;
    auto stream_s = [&](int kb, int w) { return static_cast<double>(kb) * (kBM + w) * 128 / kStreamBps; };
    const long long tiles128 = static_cast<long long>(tiles_m) * ((N + 127) / 128) * batch;
    if (!tp && tiles128 * 2 > sms) return false;
    const double whole = stream_s(kb_total, 128);
    double best = -1.0;
    int best_bn = 0, best_cs = 0;
    for (int w : {256, 192, 128}) {
        if (tp && tp->bn && tp->bn != w) continue;
        const long long t = static_cast<long long>(tiles_m) * ((N + w - 1) / w) * batch;
        for (int cs = 2; cs <= 8 && cs <= kb_total / 2; ++cs) {
            if (tp && tp->splits && tp->splits != cs) continue;
            if (t * cs > sms) break;
            if (t > cluster_split_capacity_for(w, cs)) continue;
            const double c = stream_s((kb_total + cs - 1) / cs, w) + kHandover +
                             (cs - 1.0) / cs * kBM * w * 4 / kRemoteBps;
            if (best < 0 || c < best) {
                best = c;
                best_bn = w;
                best_cs = cs;
            }
        }
    }
    if (!tp && best >= 0.9 * whole) return false;
    *bn_out = best_bn;
    *cs_out = best_cs;
    return best_cs > 0;
}

}  // namespace

cudaError_t run_gemm_f16(const TcGemm &g, cudaStream_t stream, CallInfo *info) {
    const int sms = device_sm_count();
    const int M = g.M, N = g.N, K = g.K;
    // FP16 and BF16 inputs share every kernel: the tensor maps carry the
    // element type and the MMA instruction descriptor the operand format.
    const CUtensorMapDataType in_dt = g.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    HgemmArgs a{};
    a.idesc_fmt = g.bf16 ? kIdescBf16Operands : 0u;
    a.M = M;
    a.N = N;
    a.K = K;
    a.alpha = g.alpha;
    a.beta = g.beta;
    a.bias = g.bias;
    a.act = g.act;
    a.C = g.C;
    a.ldc = g.N;
    a.c_type = g.c_type;
    a.kb_total = (K + kBK - 1) / kBK;
    a.err = watchdog_word();
    a.batch = g.batch;
    a.za = g.stride_a ? 1 : 0;
    a.zb = g.stride_b ? 1 : 0;
    a.stride_c = g.stride_c;
    a.b_kmajor = g.b_trans ? 1 : 0;
    a.c_extent = c_extent_of(a);

    // Tile table.  M <= 64: transposed product with MMA N = M rounded up to
    // 32 or 64 (K split over a cluster when its tiles fill at most half the
    // SMs).  M > 128 with enough pair tiles: CTA pairs.  Otherwise 128-row
    // tiles, 128 x 256 (128 x 128, or 128 x 96 with at most one tile per SM,
    // when that puts more SMs to work), K split
    // over a cluster when a time model says it pays (pick_cluster_split).
    // Every CTA is persistent and takes whole tiles round-robin (tiles of all
    // matrices of a batch in one sequence).  A tuned plan for this exact
    // shape (single matrices only) replaces the rules below; a plan that
    // cannot run the shape is ignored.
    TunePlan tp;
    bool tuned = g.batch == 1 && tune_lookup(1, M, N, K, &tp);
    if (tuned && tp.variant == 3 && M > (tp.bn ? tp.bn : 64)) tuned = false;
    int csplit_bn = 0, csplit_cs = 0;
    if (tuned && tp.variant == 4 &&
        !pick_cluster_split((M + kBM - 1) / kBM, N, g.batch, a.kb_total, sms, &tp, &csplit_bn, &csplit_cs))
        tuned = false;
    info->tuned = tuned;
    const bool swap = tuned ? tp.variant == 3 : M <= 64;
    int bn;
    if (swap) {
        bn = (tuned && tp.bn) ? tp.bn : (M <= 32 ? 32 : 64);
    } else {
        // Few tiles of 128 x 256: 128 x 128 tiles put twice as many SMs to work
        // streaming B (measured at 128 x 11008 x 4096: 36.5 us vs 48.8 us).
        const long long t256 = static_cast<long long>((M + kBM - 1) / kBM) * ((N + 255) / 256) * g.batch;
        bn = (N > 128 && t256 >= sms / 2) ? 256 : 128;
        // Fewer 128-wide tiles than SMs and K of 16 k blocks or more: 96-wide
        // tiles, still at most one per SM, put more SMs to work streaming B
        // (128 x 11008 x 4096: 115 tiles instead of 86, 24.2 -> 23.5 us;
        // 120 x 9000 x 520, 9 k blocks: 9.8 -> 10.1 us, so not there).
        const long long rows_t = static_cast<long long>((M + kBM - 1) / kBM) * g.batch;
        if (!tuned && bn == 128 && a.kb_total >= 16 && rows_t * ((N + 127) / 128) < sms &&
            rows_t * ((N + 95) / 96) <= sms)
            bn = 96;
        if (tuned && tp.variant == 2 && tp.bn) bn = tp.bn;
    }
    const int bn_tile = swap ? kBM : bn;
    a.tiles_m = swap ? 1 : (M + kBM - 1) / kBM;
    a.tiles_n = (N + bn_tile - 1) / bn_tile;
    const long long tiles_ll = static_cast<long long>(a.tiles_m) * a.tiles_n * g.batch;
    if (tiles_ll > (1LL << 26)) return cudaErrorNotSupported;  // keeps every unit index and counter in int
    const int tiles = static_cast<int>(tiles_ll);
    // Transposed plan: K is split into at most one unit per SM while the
    // tiles fill at most half the SMs, the splits added through distributed
    // shared memory (measured: 16 x 4096 x 4096 is best at 4 splits of 32
    // tiles; 32 x 8192 x 8192 at 2 splits of 64 tiles, 30.4 us against 41.7 us
    // unsplit).  Not transposed, K is split only over a cluster, when
    // pick_cluster_split expects it to pay (below), or by a tuned entry.
    int splits = 1;
    if (swap && tiles * 2 <= sms) splits = std::max(1, std::min(sms / tiles, a.kb_total / 2));
    splits = std::min(splits, 32);
    if (tuned && (tp.variant == 2 || tp.variant == 3) && tp.splits > 0) splits = std::max(1, std::min(tp.splits, std::max(1, a.kb_total / 2)));
    a.splits = splits;
    a.units = tiles * splits;
    // (Stream-K for the partial last wave measured slower on GB300 at
    // 4096^3, 126 us vs 110 us for whole tiles: the last arriver's reduction
    // of ~2.7 partial tiles is latency-bound inside one CTA.  CTA pairs with
    // the tile width chosen by waves replaced it.)
    // CTA pairs: M > 128 with enough 256-row pair tiles for the SMs.  The
    // tile width is picked from {256, 224, 192} by the number of waves of
    // pair tiles, then the narrowest: a tile takes nearly the same time at all
    // three widths (each CTA loads the same 64-column B boxes per k block;
    // measured ~24 us per wave at K = 4096), so 4096 x 11008 x 4096 runs
    // 43 x 256 in 10 waves (238 us) rather than 50 x 224 in 11 (266 us),
    // while 4096^3 runs 19 x 224 in 4 full waves (87 us; 256-wide tiles also
    // take 4 waves, the last one 37 % full: 91 us).
    const bool try_pair = tuned ? tp.variant == 1 : (!swap && M > kBM);
    if (try_pair && sms >= 2) {
        const int pairs = sms / 2;
        const int rows2 = (M + 2 * kBM - 1) / (2 * kBM);
        int best_bn = 0;
        double best_cost = 0.0;
        for (int cand : {256, 224, 192}) {
            const long long tn = (N + cand - 1) / cand;
            const long long t2 = static_cast<long long>(rows2) * tn * g.batch;
            // waves first; among equal waves, the narrower tile
            const double cost = static_cast<double>((t2 + pairs - 1) / pairs) * 1e9 + static_cast<double>(cand);
            if (best_bn == 0 || cost < best_cost - 1e-9) {
                best_bn = cand;
                best_cost = cost;
            }
        }
        if (tuned && tp.bn) best_bn = tp.bn;
        const int t2 = rows2 * ((N + best_bn - 1) / best_bn) * g.batch;
        if (tuned || t2 * 2 >= pairs) {
            a.tiles_m = rows2;
            a.tiles_n = (N + best_bn - 1) / best_bn;
            a.splits = 1;
            a.units = t2;
            a.c64 = (g.c_type != kOutF32 && best_bn % 64 == 0) ? 1 : 0;
            CUtensorMap ta, tb, tc;
            if (!encode_a(&ta, g, in_dt, kBM) || !encode_b(&tb, g, in_dt, best_bn / 2) ||
                !encode_c(&tc, g, g.N, a.c64 != 0))
                return cudaErrorNotSupported;
            int used = 0;
            cudaError_t e;
            // Short K (at most 8 k blocks per tile): the tile's MMA takes less
            // time than its epilogue, so 8 epilogue warps (two per TMEM lane
            // quarter, alternate 32-column chunks, one staging buffer each)
            // drain the accumulators; with long K the epilogue is hidden behind
            // the next tile's MMA and 4 warps measured as fast.
            const bool epi8 = a.kb_total <= 8;
            if (best_bn == 256) {
                e = epi8 ? launch_hgemm_pair<256, 6, 8, false>(ta, tb, tc, a, stream, &used)
                         : launch_hgemm_pair<256, 6, 4, false>(ta, tb, tc, a, stream, &used);
                info->plan = epi8 ? "tc_pair_256x256_epi8" : "tc_pair_256x256";
            } else if (best_bn == 224) {
                e = epi8 ? launch_hgemm_pair<224, 6, 8, false>(ta, tb, tc, a, stream, &used)
                         : launch_hgemm_pair<224, 6, 4, false>(ta, tb, tc, a, stream, &used);
                info->plan = epi8 ? "tc_pair_256x224_epi8" : "tc_pair_256x224";
            } else {
                e = epi8 ? launch_hgemm_pair<192, 6, 8, false>(ta, tb, tc, a, stream, &used)
                         : launch_hgemm_pair<192, 6, 4, false>(ta, tb, tc, a, stream, &used);
                info->plan = epi8 ? "tc_pair_256x192_epi8" : "tc_pair_256x192";
            }
            info->launches = 1;
            return e;
        }
    }
    // (Stream-K over all SMs for these memory-bound M <= 128 shapes measured
    // slower: 45.8 us vs 35.6 us at 128 x 11008 x 4096, the partial-tile
    // round trip costs more than the extra SMs gain.)
    // Fewer 128 x 128 tiles than SMs, not transposed: split K over the CTAs of
    // a cluster and add the partials through distributed shared memory
    // (128 x 11008 x 4096: 43 tiles of 128 x 256 in clusters of 3, 129 CTAs
    // of ~1 MB each, instead of 86 CTAs of 2 MB).
    const bool use_csplit = tuned ? tp.variant == 4
                                  : (!swap && pick_cluster_split(a.tiles_m, N, g.batch, a.kb_total, sms, nullptr,
                                                                 &csplit_bn, &csplit_cs));
    if (use_csplit) {
        a.tiles_n = (N + csplit_bn - 1) / csplit_bn;
        const int t = a.tiles_m * a.tiles_n * g.batch;
        a.splits = csplit_cs;
        a.units = t * csplit_cs;  // one CTA per unit; all of them fit at once
        CUtensorMap ta, tb;
        if (!encode_a(&ta, g, in_dt, kBM) || !encode_b(&tb, g, in_dt, csplit_bn)) return cudaErrorNotSupported;
        cudaError_t e;
        if (csplit_bn == 256) {
            e = launch_hgemm<256, 4, false, true>(ta, tb, tb, a, a.units, stream);
            info->plan = "tc_128x256_clusterk";
        } else if (csplit_bn == 192) {
            e = launch_hgemm<192, 5, false, true>(ta, tb, tb, a, a.units, stream);
            info->plan = "tc_128x192_clusterk";
        } else {
            e = launch_hgemm<128, 6, false, true>(ta, tb, tb, a, a.units, stream);
            info->plan = "tc_128x128_clusterk";
        }
        info->launches = 1;
        return e;
    }
    // The transposed small-M plan splits K over the CTAs of a cluster and adds
    // the partials through distributed shared memory (2, 4 or 8 splits).
    if (swap && splits > 1) {
        int cs = 1;
        while (cs * 2 <= std::min(splits, 8)) cs *= 2;
        a.splits = cs;
        a.units = tiles * cs;
        const int grid = std::min(a.units, (sms / cs) * cs);
        CUtensorMap ta, tb;
        if (!encode_a(&ta, g, in_dt, bn) || !encode_b(&tb, g, in_dt, kBM)) return cudaErrorNotSupported;
        cudaError_t e;
        if (bn == 32) {
            e = launch_hgemm<32, 8, true, true>(ta, tb, tb, a, grid, stream);
            info->plan = "tc_swap_n32_clusterk";
        } else {
            e = launch_hgemm<64, 8, true, true>(ta, tb, tb, a, grid, stream);
            info->plan = "tc_swap_n64_clusterk";
        }
        info->launches = 1;
        return e;
    }
    if (splits > 1) {
        Scratch sc;
        cudaError_t e =
            acquire_scratch(stream, static_cast<size_t>(tiles) * splits * kBM * bn, static_cast<size_t>(tiles) * 4, &sc);
        if (e != cudaSuccess) return e;
        a.ws = sc.partials;
        a.counters = sc.counters;
        a.ws_floats = static_cast<size_t>(tiles) * splits * kBM * bn;
    }
    const int grid = std::min(a.units, sms);

    CUtensorMap ta, tb, tc;
    std::memset(&tc, 0, sizeof(tc));
    bool ok = true;
    if (!swap) {
        ok = ok && encode_a(&ta, g, in_dt, kBM);
        ok = ok && encode_b(&tb, g, in_dt, bn);
        ok = ok && encode_c(&tc, g, g.N);
    } else {
        ok = ok && encode_a(&ta, g, in_dt, bn);
        ok = ok && encode_b(&tb, g, in_dt, kBM);
        tc = tb;  // unused by the transposed variant
    }
    if (!ok) return cudaErrorNotSupported;

    cudaError_t e;
    if (!swap) {
        // Whole tiles, one per CTA: nothing hides a tile's epilogue, so 8
        // epilogue warps share it.
        const bool epi8 = splits == 1 && a.units <= sms;
        if (bn == 256) {
            e = epi8 ? launch_hgemm<256, 4, false, false, 8>(ta, tb, tc, a, grid, stream)
                     : launch_hgemm<256, 4, false>(ta, tb, tc, a, grid, stream);
            info->plan = splits > 1 ? "tc_128x256_splitk" : (epi8 ? "tc_128x256_epi8" : "tc_128x256");
        } else if (bn == 96) {
            e = epi8 ? launch_hgemm<96, 6, false, false, 8>(ta, tb, tc, a, grid, stream)
                     : launch_hgemm<96, 6, false>(ta, tb, tc, a, grid, stream);
            info->plan = splits > 1 ? "tc_128x96_splitk" : (epi8 ? "tc_128x96_epi8" : "tc_128x96");
        } else {
            e = epi8 ? launch_hgemm<128, 6, false, false, 8>(ta, tb, tc, a, grid, stream)
                     : launch_hgemm<128, 6, false>(ta, tb, tc, a, grid, stream);
            info->plan = splits > 1 ? "tc_128x128_splitk" : (epi8 ? "tc_128x128_epi8" : "tc_128x128");
        }
    } else {
        if (bn == 32) {
            e = launch_hgemm<32, 8, true>(ta, tb, tc, a, grid, stream);
            info->plan = splits > 1 ? "tc_swap_n32_splitk" : "tc_swap_n32";
        } else {
            e = launch_hgemm<64, 8, true>(ta, tb, tc, a, grid, stream);
            info->plan = splits > 1 ? "tc_swap_n64_splitk" : "tc_swap_n64";
        }
    }
    info->launches = 1;
    return e;
}

// ------------------------------------------------------------------ FP32 through 3 x TF32
// The FP32 product on the tensor cores: every FP32 operand x is split into a
// TF32 high part h = tf32(x) and a TF32 low part l = tf32(x - h) (x - h is
// exact in FP32), so x = h + l + e with |e| <= 2^-22 |x|, and
//   a b ~= a_h b_h + a_h b_l + a_l b_h        (a_l b_l ~ 2^-22 |a b| dropped).
// A pre-pass writes A_h, A_l (M x Kp) and B_h^T, B_l^T (N x Kp, so that both
// MMA operands are K-major), Kp = K rounded up to 4 (16-byte rows), zero-filled
// past K; the CTA-pair kernel then runs three kind::tf32 MMAs per k step.
namespace {

__global__ void __launch_bounds__(256) split_rows_tf32_kernel(const float *__restrict__ A, int lda, int M, int K,
                                                              int Kp, float *__restrict__ hi, float *__restrict__ lo) {
    for (int r = blockIdx.x; r < M; r += gridDim.x) {
        const float *src = A + static_cast<size_t>(r) * lda;
        float *h = hi + static_cast<size_t>(r) * Kp;
        float *l = lo + static_cast<size_t>(r) * Kp;
        for (int c = threadIdx.x; c < Kp; c += 256) {
            const float x = c < K ? __ldcs(src + c) : 0.f;
            const float xh = tf32_round(x);
            h[c] = xh;
            l[c] = tf32_round(x - xh);
        }
    }
}

// B (K x N, ldb) -> B_h^T, B_l^T (N x Kp) through 32 x 32 shared-memory tiles:
// reads along n and writes along k are both coalesced.
__global__ void __launch_bounds__(256) split_cols_tf32_kernel(const float *__restrict__ B, int ldb, int K, int N,
                                                              int Kp, float *__restrict__ hi, float *__restrict__ lo) {
    __shared__ float tile[32][33];
    const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const int k = k0 + ty + j, n = n0 + tx;
        tile[ty + j][tx] = (k < K && n < N) ? __ldcs(B + static_cast<size_t>(k) * ldb + n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const int n = n0 + ty + j, k = k0 + tx;
        if (n < N && k < Kp) {
            const float x = tile[tx][ty + j];
            const float xh = tf32_round(x);
            hi[static_cast<size_t>(n) * Kp + k] = xh;
            lo[static_cast<size_t>(n) * Kp + k] = tf32_round(x - xh);
        }
    }
}

}  // namespace

cudaError_t run_gemm_f32_3xtf32(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                                float beta, float *C, int ldc, cudaStream_t stream, CallInfo *info) {
    const int sms = device_sm_count();
    const int Kp = (K + 3) & ~3;
    const size_t a_elems = static_cast<size_t>(M) * Kp, b_elems = static_cast<size_t>(N) * Kp;
    float *ws = nullptr;
    cudaError_t e = acquire_operand_scratch(stream, 2 * a_elems + 2 * b_elems, &ws);
    if (e != cudaSuccess) return e;
    float *a_hi = ws, *a_lo = ws + a_elems, *bt_hi = a_lo + a_elems, *bt_lo = bt_hi + b_elems;
    e = launch_kernel(split_rows_tf32_kernel, dim3(std::min(M, 8 * sms)), dim3(256), 0, stream, A, lda, M, K, Kp, a_hi,
                   a_lo);
    if (e != cudaSuccess) return e;
    const dim3 tgrid((N + 31) / 32, (Kp + 31) / 32);
    if (tgrid.y > 65535u) return cudaErrorNotSupported;
    e = launch_kernel(split_cols_tf32_kernel, tgrid, dim3(256), 0, stream, B, ldb, K, N, Kp, bt_hi, bt_lo);
    if (e != cudaSuccess) return e;

    // Pair tile width by the planner's rule for CTA pairs: fewest waves, then
    // the narrowest of {256, 224, 192}.
    const int pairs = std::max(1, sms / 2);
    const int rows2 = (M + 2 * kBM - 1) / (2 * kBM);
    int BN = 0;
    long long best_waves = 0;
    for (int cand : {256, 224, 192}) {
        const long long t2c = static_cast<long long>(rows2) * ((N + cand - 1) / cand);
        const long long waves = (t2c + pairs - 1) / pairs;
        if (BN == 0 || waves <= best_waves) {
            BN = cand;
            best_waves = waves;
        }
    }
    HgemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.alpha = alpha;
    a.beta = beta;
    a.C = C;
    a.ldc = ldc;
    a.c_type = kOutF32;
    a.kb_total = (K + 31) / 32;
    a.err = watchdog_word();
    a.batch = 1;
    a.za = a.zb = 0;
    a.stride_c = static_cast<long long>(M) * ldc;
    a.b_kmajor = 1;
    a.c_extent = c_extent_of(a);
    a.tiles_m = (M + 2 * kBM - 1) / (2 * kBM);
    a.tiles_n = (N + BN - 1) / BN;
    const long long t2 = static_cast<long long>(a.tiles_m) * a.tiles_n;
    if (t2 > (1LL << 26)) return cudaErrorNotSupported;
    a.splits = 1;
    a.units = static_cast<int>(t2);
    TcGemm g;
    g.M = M;
    g.N = N;
    g.C = C;
    CUtensorMap ta, ta2, tb, tb2, tc;
    const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (!encode_3d(&ta, f32, 4, a_hi, K, M, 1, Kp, 0, 32, kBM) || !encode_3d(&ta2, f32, 4, a_lo, K, M, 1, Kp, 0, 32, kBM) ||
        !encode_3d(&tb, f32, 4, bt_hi, K, N, 1, Kp, 0, 32, BN / 2) ||
        !encode_3d(&tb2, f32, 4, bt_lo, K, N, 1, Kp, 0, 32, BN / 2) ||
        !encode_c(&tc, g, M == 1 ? (N + 3) & ~3 : ldc))  // one row: any 16-byte row stride describes it
        return cudaErrorNotSupported;
    int used = 0;
    if (BN == 256) {
        e = launch_hgemm_pair<256, 3, 8, true>(ta, tb, tc, a, stream, &used, &ta2, &tb2);
        info->plan = "tf32x3_pair_256x256";
    } else if (BN == 224) {
        e = launch_hgemm_pair<224, 3, 8, true>(ta, tb, tc, a, stream, &used, &ta2, &tb2);
        info->plan = "tf32x3_pair_256x224";
    } else {
        e = launch_hgemm_pair<192, 3, 8, true>(ta, tb, tc, a, stream, &used, &ta2, &tb2);
        info->plan = "tf32x3_pair_256x192";
    }
    info->launches = 3;
    return e;
}

// ------------------------------------------------------------------ no-allocation variant
// The small-M (M <= 64) transposed split-K plan of run_gemm_f16, with its
// split-K scratch taken from a fixed array in device memory instead of the
// library's lazily allocated per-stream buffer, for callers that cannot let
// the library call cudaMalloc.  The array below is part of the module image:
// every GPU that loads the library holds it until the process exits.
namespace {

constexpr size_t kNoAllocCounters = 4096;                   // arrival counters (4 per tile)
constexpr size_t kNoAllocPartialFloats = size_t(1) << 20;   // fp32 partial tiles: 4 MiB
constexpr size_t kNoAllocBytes = kNoAllocCounters * sizeof(unsigned) + kNoAllocPartialFloats * sizeof(float);

// Counters first (16 KiB), partial tiles after them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocSlot {
    std::mutex mu;
    unsigned char *base = nullptr;  // device address of g_noalloc_scratch; set only once a lookup succeeded
};
NoAllocSlot g_noalloc_slot[64];

}  // namespace

cudaError_t run_gemm_f16_small_m_noalloc(int M, int N, int K, float alpha, const void *A, const void *B, float beta,
                                         float *C, const float *bias, int act, cudaStream_t stream, CallInfo *info,
                                         int *reject) {
    *reject = 0;
    if (M > 64) {
        *reject = 1;
        return cudaSuccess;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // Set-up, once per device, with that device current: host code cannot use
    // the array's name as a device address, so look the address up.  A failed
    // lookup is not remembered; the next call on the device tries again.
    NoAllocSlot &slot = g_noalloc_slot[dev];
    unsigned char *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(slot.mu);
        if (!slot.base) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            slot.base = static_cast<unsigned char *>(p);
        }
        base = slot.base;
    }
    unsigned *counters = reinterpret_cast<unsigned *>(base);
    float *partials = reinterpret_cast<float *>(base + kNoAllocCounters * sizeof(unsigned));

    const int sms = device_sm_count();
    HgemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.alpha = alpha;
    a.beta = beta;
    a.bias = bias;
    a.act = act;
    a.C = C;
    a.ldc = N;
    a.kb_total = (K + kBK - 1) / kBK;
    a.err = watchdog_word();
    a.batch = 1;
    a.za = a.zb = 0;
    a.stride_c = static_cast<long long>(M) * N;
    a.c_extent = c_extent_of(a);
    const int bn = M <= 32 ? 32 : 64;
    a.tiles_m = 1;
    a.tiles_n = (N + kBM - 1) / kBM;
    const int tiles = a.tiles_n;
    int splits = 1;
    if (tiles < sms) splits = std::max(1, std::min(sms / tiles, a.kb_total / 2));
    splits = std::min(splits, 32);
    if (splits > 1) {
        // As many K splits as the fixed array holds, up to the planner's count;
        // a plan that cannot keep even two splits' partials there is rejected.
        const size_t per_split = static_cast<size_t>(tiles) * kBM * bn;
        splits = static_cast<int>(std::min<size_t>(splits, kNoAllocPartialFloats / per_split));
        if (splits < 2 || static_cast<size_t>(tiles) * 4 > kNoAllocCounters) {
            *reject = 2;
            return cudaSuccess;
        }
    }
    a.splits = splits;
    a.units = tiles * splits;
    if (splits > 1) {
        const size_t need_counters = static_cast<size_t>(tiles) * 4;
        // The array keeps the previous call's contents: the counters must start at zero.
        e = cudaMemsetAsync(counters, 0, need_counters * sizeof(unsigned), stream);
        if (e != cudaSuccess) return e;
        a.ws = partials;
        a.ws_floats = static_cast<size_t>(tiles) * splits * kBM * bn;
        a.counters = counters;
    }
    TcGemm g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.A = A;
    g.B = B;
    CUtensorMap ta, tb;
    if (!encode_a(&ta, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bn) || !encode_b(&tb, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kBM))
        return cudaErrorNotSupported;
    const int grid = std::min(a.units, sms);
    if (bn == 32) {
        e = launch_hgemm<32, 8, true>(ta, tb, tb, a, grid, stream);
        info->plan = splits > 1 ? "tc_swap_n32_splitk_static" : "tc_swap_n32_static";
    } else {
        e = launch_hgemm<64, 8, true>(ta, tb, tb, a, grid, stream);
        info->plan = splits > 1 ? "tc_swap_n64_splitk_static" : "tc_swap_n64_static";
    }
    info->launches = splits > 1 ? 2 : 1;  // counter clear + GEMM
    return e;
}

// ------------------------------------------------------------------ stalled-pipeline self-test
// The single-CTA plan (128 x 128 tiles, no K split, FP16 operands, FP32 C)
// with its producer switched off: no TMA load is issued and no arrival made,
// so nothing is in flight when the MMA thread's wait for the first stage and
// the epilogue's wait for the accumulator give up after wait_ns.  They record
// the timeout in the watchdog word and leave their loops; the CTA frees its
// tensor memory and returns.  C is not written.
cudaError_t run_hgemm_stall_selftest(int M, int N, int K, const void *A, const void *B, float *C,
                                     unsigned long long wait_ns, cudaStream_t stream) {
    HgemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.alpha = 1.f;
    a.C = C;
    a.ldc = N;
    a.c_type = kOutF32;
    a.kb_total = (K + kBK - 1) / kBK;
    a.err = watchdog_word();
    a.batch = 1;
    a.stride_c = static_cast<long long>(M) * N;
    a.c_extent = c_extent_of(a);
    a.tiles_m = (M + kBM - 1) / kBM;
    a.tiles_n = (N + 127) / 128;
    if (static_cast<long long>(a.tiles_m) * a.tiles_n > (1LL << 26)) return cudaErrorNotSupported;
    a.splits = 1;
    a.units = a.tiles_m * a.tiles_n;
    a.wait_ns = wait_ns;
    a.stall_producer = 1;
    TcGemm g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.A = A;
    g.B = B;
    g.C = C;
    g.stride_c = a.stride_c;
    g.c_type = kOutF32;
    CUtensorMap ta, tb, tc;
    if (!encode_a(&ta, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kBM) || !encode_b(&tb, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 128) ||
        !encode_c(&tc, g, N))
        return cudaErrorNotSupported;
    return launch_hgemm<128, 6, false>(ta, tb, tc, a, std::min(a.units, device_sm_count()), stream);
}

}  // namespace gemm11
