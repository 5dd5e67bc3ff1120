// tcgen05 / TMA kernels for the reweighted clipped sum, whose operands are
// both "row = contraction index" (MN-major) arrays:
//
// The reweighted clipped sum of a layer,
//        S = E^T diag(c) A = sum_i c_i E_i^T A_i     (K = B*T rows),
// and the noise epilogue G = (S + sigma C z) / L computed from TMEM
// ("Privacy-Preserving Machine Learning", section "Differentially private
// stochastic gradient descent", phases 3-5; "Sensitivity Inflation from
// Cross-Record Precision Routing in Private Quantized Fine-Tuning", Eq. 3):
//
//  * k_clipped_sum_fold_pair_tc: T a multiple of 64 and B > 1, the clip
//    factor folded per record in fp32 by the epilogue warps, on CTA pairs.
//  * otherwise c_i A_i or c_i E_i (the operand with fewer columns) is first
//    written into scratch -- by the clip kernel as soon as c_i is known
//    (k_prescale_rows beyond four such layers) -- and the sum runs as a
//    single "record" of K rows with factor 1: k_sum_layers_pair_tc for the
//    layers whose copy the clip kernel wrote (several layers per launch, CTA
//    pairs), k_clipped_sum_tc for the others (one CTA per tile).
//
// Warp roles (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM owner and MMA issuer (one lane; rank 0 of a pair)
//   warps 2-17  the epilogue: fold S += c_i P_i, noise, G
#include <cuda_bf16.h>

#include <atomic>
#include <climits>

#include "common.cuh"
#include "launch.cuh"
#include "tc_common.cuh"

using namespace dpk;

namespace {

// ============================================================ clipped sum
constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kAStage = kBM * kBK * 2;  // E tile: 2 boxes of 64 columns x 64 rows
constexpr int kBStage = kBN * kBK * 2;  // A tile: 4 boxes
constexpr int kStageBytes = kAStage + kBStage;
constexpr int kAccCols = kBN;           // fp32 accumulator columns per buffer
// TMEM allocation (a power of two) holding both accumulator buffers
constexpr uint32_t kTmemCols = 2 * kAccCols <= 256 ? 256 : 512;
constexpr uint32_t kIdescSum = tc::idesc_bf16_f32(kBM, kBN, 1, 1);
constexpr size_t kSumSmem = 1024 + (size_t)kStages * kStageBytes + 256;

struct SumParams {
    CUtensorMap tmE;   // {d_out, K} bf16, box {64, 64}, 128B swizzle
    CUtensorMap tmA;   // {d_in,  K} bf16, box {64, 64}, 128B swizzle
    int64_t K, T, d_in, d_out;
    int m_blocks, n_blocks;
    const float* c;
    unsigned* status;
    float* G;
    int64_t coord_off;
    float scale;       // sigma * C
    float inv_L;       // 1 / L
    uint64_t seed, step;
    int box3d;                      // 1: one 3D TMA copy per operand tile (64-column chunks as the outer dimension)
    // split of the last partial wave (records mode only; see next_work)
    int full_tiles;                 // tiles done whole, strided over the grid
    int nsplit;                     // record ranges per remaining tile (1: no split)
    float* scratch;                 // [grid][kBN][kBM] partial sums of the split tiles
    unsigned long long* counters;   // [ntiles - full_tiles] arrivals, (epoch << 32) | count
    unsigned epoch;                 // this launch's tag for the counters
};

__device__ __forceinline__ void tile_coords(int tile, int m_blocks, int n_blocks, int& mb, int& nb) {
    // groups of 8 row blocks, column blocks fastest inside a group: the tiles
    // running together share their E and A column blocks in L2
    constexpr int GM = 8;
    const int per_group = GM * n_blocks;
    const int g = tile / per_group;
    const int first = g * GM;
    const int gm = min(GM, m_blocks - first);
    const int r = tile - g * per_group;
    mb = first + r % gm;
    nb = r / gm;
}

// ------------------------------------------------------------ work split
// With records (B > 1), a CTA pair does the whole tiles pair, pair + npairs,
// ... below full_tiles.  When the tile count leaves a partial last wave of R
// tiles, the remaining tiles are each cut into nsplit = npairs / R ranges of
// records, all run at once: pair b < R * nsplit takes tile full_tiles + b % R,
// records of range b / R.  The pairs working on one range read the same K
// rows of E and A at the same time, as a whole wave would.  Every range
// writes its partial sum to the CTA's scratch slot; the CTA that arrives last
// at the counter of its half of the tile adds the slots in range order and
// writes G (a fixed order, so the result does not depend on timing).
struct Work {
    int tile;
    int seg;            // record range of a split tile, -1 for a whole tile
    int64_t r0, r1;     // records [r0, r1)
};

// ====================================================== single-record sum
// One record of K rows with factor 1 (the clip factors are in the pre-scaled
// operand; a partial last K tile is zero-filled by TMA), one CTA per 128 x
// 256 tile, tiles strided over the CTAs, the whole K accumulated in TMEM (two
// buffers, so a tile's epilogue overlaps the next tile's MMAs).  Warps 2-17:
// four per TMEM lane quarter, each owning 64 of the 256 columns (sixteen
// epilogue warps keep enough chains in flight for the Philox / Box-Muller
// epilogue).
constexpr int kEpiWarps = 16;
constexpr int kColsPerWarp = kBN / (kEpiWarps / 4);
constexpr int kFoldThreads = 32 * (2 + kEpiWarps);

struct FoldSmem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t p_full[2];
    uint64_t p_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// z for 8 consecutive coordinates starting at kb
__device__ __forceinline__ void noise8(uint64_t seed, uint64_t step, uint64_t kb, float (&z)[8]) {
    if ((kb & 3u) == 0) {
        noise_blocks<2>(seed, step, kb >> 2, z);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) z[j] = noise_at(seed, step, kb + j);
    }
}

// S[4q .. 4q+3] += sigma C z at this thread's coordinates k0 + 4q .. k0 + 4q + 3
template <int NC>
__device__ __forceinline__ void add_noise_chunk_n(const SumParams& p, uint64_t k0, int q, float (&S)[NC]) {
    const uint64_t k = k0 + 4u * (uint64_t)q;
    float z[4];
    if ((k & 3u) == 0) {
        noise_blocks<1>(p.seed, p.step, k >> 2, z);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) z[j] = noise_at(p.seed, p.step, k + j);
    }
#pragma unroll
    for (int qq = 0; qq < NC / 4; ++qq)
        if (qq == q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) S[4 * qq + j] = fmaf(p.scale, z[j], S[4 * qq + j]);
        }
}

__global__ void __launch_bounds__(kFoldThreads, 1) k_clipped_sum_tc(const __grid_constant__ SumParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    FoldSmem* sh = reinterpret_cast<FoldSmem*>(tiles + (size_t)kStages * kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = p.m_blocks * p.n_blocks;
    const int nk = (int)((p.K + kBK - 1) / kBK);  // K tiles (zero-filled past K)
    volatile int* abort_flag = &sh->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&sh->full[s], 1);
            tc::mbar_init(&sh->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sh->p_full[b], 1);
            tc::mbar_init(&sh->p_empty[b], 32 * kEpiWarps);
        }
        tc::mbar_init(&sh->drain, 1);
        sh->abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&p.tmE);
        tc::tma_prefetch_desc(&p.tmA);
    }
    if (warp == 1) tc::tmem_alloc(&sh->tmem_base, kTmemCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    // everything above overlaps the previous kernel; its outputs (c, the
    // pre-scaled operand, the status word) are read only from here on
    grid_dep_wait();
    grid_dep_trigger();
    const bool skip = status_bad(p.status);

    if (!skip && warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            tc::StageRing<kStages> ring;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, p.m_blocks, p.n_blocks, mb, nb);
                for (int kt = 0; kt < nk; ++kt, ++it, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->empty[s], ring.ph ^ 1u, abort_flag, p.status)) goto sum_producer_done;
                    uint8_t* st = tiles + (size_t)s * kStageBytes;
                    tc::mbar_arrive_expect_tx(&sh->full[s], kStageBytes);
                    const int k0 = kt * kBK;
                    if (p.box3d) {
                        tc::tma_load_3d(st, &p.tmE, &sh->full[s], 0, k0, mb * (kBM / 64));
                        tc::tma_load_3d(st + kAStage, &p.tmA, &sh->full[s], 0, k0, nb * (kBN / 64));
                    } else {
                        tc::tma_load_2d(st, &p.tmE, &sh->full[s], mb * kBM, k0);
                        tc::tma_load_2d(st + 8192, &p.tmE, &sh->full[s], mb * kBM + 64, k0);
#pragma unroll
                        for (int q = 0; q < kBN / 64; ++q)
                            tc::tma_load_2d(st + kAStage + q * 8192, &p.tmA, &sh->full[s], nb * kBN + 64 * q, k0);
                    }
                }
            }
        sum_producer_done:
            for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
                tc::mbar_wait_drain(&sh->full[j % kStages], (j / kStages) & 1u);
        }
    } else if (!skip && warp == 1) {
        if (lane == 0) {
            uint32_t rc = 0;
            tc::StageRing<kStages> ring;
            const uint32_t tiles_u32 = tc::smem_u32(tiles);
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++rc) {
                const uint32_t b = rc & 1u, bph = (rc >> 1) & 1u;
                if (!tc::mbar_wait(&sh->p_empty[b], bph ^ 1u, abort_flag, p.status)) break;
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem + b * kAccCols;
                bool ok = true;
                for (int kt = 0; kt < nk; ++kt, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->full[s], ring.ph, abort_flag, p.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t sa = tiles_u32 + s * (uint32_t)kStageBytes;
                    const uint64_t ad = tc::smem_desc(sa, 8192, 1024, tc::SW_128B);
                    const uint64_t bd = tc::smem_desc(sa + kAStage, 8192, 1024, tc::SW_128B);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_bf16(d_tmem, tc::desc_advance(ad, kk * 2048), tc::desc_advance(bd, kk * 2048), kIdescSum,
                                     (kt | kk) != 0);
                    tc::mma_commit(&sh->empty[s]);
                }
                if (!ok) break;
                tc::mma_commit(&sh->p_full[b]);
            }
        }
    } else if (!skip && warp >= 2) {
        const int quarter = warp & 3;
        const int part = (warp - 2) >> 2;          // columns part*64 .. +63
        const int row = quarter * 32 + lane;
        uint32_t rc = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++rc) {
            // the noise does not depend on the sum: drawn while the tensor
            // cores are still accumulating this tile
            int mb, nb;
            tile_coords(tile, p.m_blocks, p.n_blocks, mb, nb);
            const int64_t m = (int64_t)mb * kBM + row;
            const int64_t n0 = (int64_t)nb * kBN + part * kColsPerWarp;
            float z[kColsPerWarp];
            if (m < p.d_out) {
#pragma unroll
                for (int ch = 0; ch < kColsPerWarp / 8; ++ch) {
                    float zc[8];
                    noise8(p.seed, p.step, (uint64_t)(p.coord_off + m * p.d_in + n0 + ch * 8), zc);
#pragma unroll
                    for (int j = 0; j < 8; ++j) z[ch * 8 + j] = zc[j];
                }
            }
            const uint32_t b = rc & 1u, bph = (rc >> 1) & 1u;
            if (!tc::mbar_wait_warp(&sh->p_full[b], bph, abort_flag, p.status)) break;
            tc::tc_fence_after();
            const float c0 = __ldca(p.c);
            const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + b * kAccCols + part * kColsPerWarp;
            float* out = p.G + m * p.d_in + n0;
#pragma unroll
            for (int ch = 0; ch < kColsPerWarp / 16; ++ch) {
                float v[16];
                tc::tmem_ld16(tb + ch * 16, v);
                if (m >= p.d_out) continue;
                const int64_t n = n0 + ch * 16;
                if (n + 16 <= p.d_in) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        float4 o;
                        o.x = (c0 * v[j] + p.scale * z[ch * 16 + j]) * p.inv_L;
                        o.y = (c0 * v[j + 1] + p.scale * z[ch * 16 + j + 1]) * p.inv_L;
                        o.z = (c0 * v[j + 2] + p.scale * z[ch * 16 + j + 2]) * p.inv_L;
                        o.w = (c0 * v[j + 3] + p.scale * z[ch * 16 + j + 3]) * p.inv_L;
                        *reinterpret_cast<float4*>(out + ch * 16 + j) = o;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (n + j < p.d_in) out[ch * 16 + j] = (c0 * v[j] + p.scale * z[ch * 16 + j]) * p.inv_L;
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sh->p_empty[b]);
        }
    }

    if (!skip && warp == 1 && lane == 0) {
        tc::mma_commit(&sh->drain);
        tc::mbar_wait_drain(&sh->drain, 0);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ================================= single-record sums of several layers
// Layers whose clip factors the clip kernel folded into a pre-scaled operand
// are sums over K = B*T rows with factor 1 (as k_clipped_sum_tc).
// Layers sharing K are summed in one persistent launch, k_sum_layers_pair_tc:
// their output tiles form one index space, strided over the CTA pairs, so a
// layer's tiles fill the SMs another layer's partial wave leaves idle, and
// the launch boundary between the layers is gone.
constexpr int kMaxSumLayers = 4;

struct SumLayer {
    CUtensorMap tmE;   // the layer's operands over the K rows (as SumParams)
    CUtensorMap tmA;
    int64_t d_in, d_out;
    int m_blocks, n_blocks;
    int box3d;
    float* G;
    int64_t coord_off;
};

struct LayersParams {
    int nlayers;
    int nk;                          // K tiles of every tile
    int tile_begin[kMaxSumLayers + 1];
    unsigned* status;
    float scale, inv_L;              // sigma * C, 1 / L
    uint64_t seed, step;
    SumLayer L[kMaxSumLayers];
};

// layer and tile within it of tile g of the launch
__device__ __forceinline__ int layer_of(const LayersParams& p, int g) {
    int l = 0;
    while (l + 1 < p.nlayers && p.tile_begin[l + 1] <= g) ++l;
    return l;
}

// ==================================== single-record sums on CTA pairs
// A 256 x 256 output tile per cluster of two CTAs and one
// tcgen05.mma.cta_group::2 per K step: CTA r stages columns [128 r, 128 r +
// 128) of the tile's E and A blocks (its half of M and of N), rank 0 issues
// the MMAs, and each CTA's TMEM receives its 128 rows of the tile (two
// buffers, so a tile's epilogue overlaps the next tile's MMAs).  Per SM the
// tensor cores do the same work per K step as a 128 x 256 tile of one CTA
// but stage two thirds of its bytes, which leaves room for six stages and a
// 2 KB staging block per epilogue warp.  Every tile of a pair but its first
// starts from its noise: the epilogue warps write sigma C z into the tile's
// TMEM buffer while the tensor cores accumulate the tile before it, and the
// MMAs accumulate onto it; the first tile's noise is drawn in its epilogue,
// 16 columns at a time, while the tensor cores accumulate the second.  The
// epilogue writes G = S / L through its staging block: a store instruction
// covers 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes, four
// times fewer (and whole-sector) L2 writes.
//
// Barriers: rank 0's full[s] counts both CTAs' copies (its producer expects
// the bytes of both halves); the MMA commits arrive on empty[s], p_full[b]
// and drain of both CTAs; the epilogue warps of both CTAs arrive on rank 0's
// p_empty[b].
//
// Eight epilogue warps, two per TMEM lane quarter, each owning 128 of the 256
// columns: with fewer warps drawing noise next to them, the TMA and MMA warps
// on the same schedulers keep pace (on the 1024 -> 4096 -> 1024 MLP with 4096
// records, sixteen warps took 61.4 us for both sums, eight take 59.4 us).
constexpr int kLEpiWarps = 8;
constexpr int kLColsPerWarp = kBN / (kLEpiWarps / 4);
constexpr int kLThreads = 32 * (2 + kLEpiWarps);
constexpr int kPairStages = 6;
constexpr int kHalf = 128;                    // M rows and N columns staged per CTA
constexpr int kPairTile = 2 * kHalf;          // output tile of the pair: 256 x 256
constexpr int kPairEStage = kHalf * kBK * 2;  // 2 boxes of 64 columns x 64 rows
constexpr int kPairStageBytes = 2 * kPairEStage;
constexpr uint32_t kIdescPair = tc::idesc_bf16_f32(kPairTile, kPairTile, 1, 1);
constexpr int kStagingBytes = kLEpiWarps * 32 * 16 * 4;  // 32 rows x 16 fp32 per epilogue warp
constexpr size_t kPairSmem = 1024 + (size_t)kPairStages * kPairStageBytes + kStagingBytes + 256;

struct PairSmem {
    uint64_t full[kPairStages];
    uint64_t empty[kPairStages];
    uint64_t p_full[2];
    uint64_t p_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(PairSmem) <= 256, "pair barriers exceed their shared-memory slot");


// sigma C z at this thread's 128 coordinates of tile g (row `row` of the
// CTA's half, the warp's column part), written into the warp's TMEM columns
// starting at tb: the accumulator of the tile then starts from its noise.
// Rows past d_out get zeros; columns past d_in get values that are never
// stored.  All lanes of the warp call it (the TMEM stores are warp-wide).
__device__ __forceinline__ void write_tile_noise(const LayersParams& p, int g, uint32_t rank, int row, int part,
                                                 uint32_t tb) {
    const int l = layer_of(p, g);
    const SumLayer& ly = p.L[l];
    int mb, nb;
    tile_coords(g - p.tile_begin[l], ly.m_blocks, ly.n_blocks, mb, nb);
    const int64_t m = (int64_t)mb * kPairTile + (int64_t)rank * kHalf + row;
    const int64_t n0 = (int64_t)nb * kPairTile + part * kLColsPerWarp;
#pragma unroll 1
    for (int ch = 0; ch < kLColsPerWarp / 16; ++ch) {
        float z[16];
        if (m < ly.d_out) {
            float za[8], zb[8];
            const uint64_t k = (uint64_t)(ly.coord_off + m * ly.d_in + n0 + ch * 16);
            noise8(p.seed, p.step, k, za);
            noise8(p.seed, p.step, k + 8, zb);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                z[j] = p.scale * za[j];
                z[8 + j] = p.scale * zb[j];
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) z[j] = 0.f;
        }
        tc::tmem_st16(tb + ch * 16, z);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kLThreads, 1)
    k_sum_layers_pair_tc(const __grid_constant__ LayersParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = tiles + (size_t)kPairStages * kPairStageBytes;
    PairSmem* sh = reinterpret_cast<PairSmem*>(staging + kStagingBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_ctarank();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int ntiles = p.tile_begin[p.nlayers];
    volatile int* abort_flag = &sh->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            tc::mbar_init(&sh->full[s], 1);
            tc::mbar_init(&sh->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sh->p_full[b], 1);
            tc::mbar_init(&sh->p_empty[b], 2 * kLEpiWarps);
        }
        tc::mbar_init(&sh->drain, 1);
        sh->abort_flag = 0;
        tc::fence_barrier_init();
        for (int l = 0; l < p.nlayers; ++l) {
            tc::tma_prefetch_desc(&p.L[l].tmE);
            tc::tma_prefetch_desc(&p.L[l].tmA);
        }
    }
    if (warp == 1) tc::tmem_alloc_pair(&sh->tmem_base, 2 * kAccCols);
    tc::tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either signals the other
    tc::cluster_sync();
    tc::tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    grid_dep_wait();
    grid_dep_trigger();
    const bool skip = status_bad(p.status);

    if (!skip && warp == 0) {
        if (lane == 0) {
            const uint32_t full0 = tc::mapa_shared(tc::smem_u32(&sh->full[0]), 0);
            uint32_t it = 0;
            tc::StageRing<kPairStages> ring;
            for (int g = pair; g < ntiles; g += npairs) {
                const int l = layer_of(p, g);
                const SumLayer& ly = p.L[l];
                int mb, nb;
                tile_coords(g - p.tile_begin[l], ly.m_blocks, ly.n_blocks, mb, nb);
                for (int kt = 0; kt < p.nk; ++kt, ++it, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->empty[s], ring.ph ^ 1u, abort_flag, p.status)) goto pair_producer_done;
                    uint8_t* st = tiles + (size_t)s * kPairStageBytes;
                    if (rank == 0) tc::mbar_arrive_expect_tx(&sh->full[s], 2 * kPairStageBytes);
                    const uint32_t fb = full0 + (uint32_t)(s * sizeof(uint64_t));
                    const int k0 = kt * kBK;
                    if (ly.box3d) {
                        tc::tma_load_3d_pair(st, &ly.tmE, fb, 0, k0, mb * (kPairTile / 64) + (int)rank * (kHalf / 64));
                        tc::tma_load_3d_pair(st + kPairEStage, &ly.tmA, fb, 0, k0,
                                             nb * (kPairTile / 64) + (int)rank * (kHalf / 64));
                    } else {
                        const int xe = mb * kPairTile + (int)rank * kHalf, xa = nb * kPairTile + (int)rank * kHalf;
                        tc::tma_load_2d_pair(st, &ly.tmE, fb, xe, k0);
                        tc::tma_load_2d_pair(st + 8192, &ly.tmE, fb, xe + 64, k0);
                        tc::tma_load_2d_pair(st + kPairEStage, &ly.tmA, fb, xa, k0);
                        tc::tma_load_2d_pair(st + kPairEStage + 8192, &ly.tmA, fb, xa + 64, k0);
                    }
                }
            }
        pair_producer_done:
            // rank 0 waits for the copies of both CTAs still in flight; rank 1's
            // copies complete on rank 0's barriers before the final cluster barrier
            if (rank == 0)
                for (uint32_t j = it > kPairStages ? it - kPairStages : 0; j < it; ++j)
                    tc::mbar_wait_drain(&sh->full[j % kPairStages], (j / kPairStages) & 1u);
        }
    } else if (!skip && warp == 1) {
        if (lane == 0 && rank == 0) {
            uint32_t rc = 0;
            tc::StageRing<kPairStages> ring;
            const uint32_t tiles_u32 = tc::smem_u32(tiles);
            bool ok = true;
            for (int g = pair; g < ntiles && ok; g += npairs, ++rc) {
                const uint32_t b = rc & 1u, bph = (rc >> 1) & 1u;
                // buffer 1 has one more phase: the epilogue releases it once at
                // the start, after writing the pair's second tile's noise into it
                if (!tc::mbar_wait(&sh->p_empty[b], b ? bph : (bph ^ 1u), abort_flag, p.status)) break;
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem + b * kAccCols;
                // every tile but the pair's first accumulates onto its noise
                const uint32_t acc0 = (rc >= 1 && p.scale != 0.f) ? 1u : 0u;
                for (int kt = 0; kt < p.nk; ++kt, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->full[s], ring.ph, abort_flag, p.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t sa = tiles_u32 + s * (uint32_t)kPairStageBytes;
                    const uint64_t ad = tc::smem_desc(sa, 8192, 1024, tc::SW_128B);
                    const uint64_t bd = tc::smem_desc(sa + kPairEStage, 8192, 1024, tc::SW_128B);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_bf16_pair(d_tmem, tc::desc_advance(ad, kk * 2048), tc::desc_advance(bd, kk * 2048),
                                          kIdescPair, acc0 | (uint32_t)((kt | kk) != 0));
                    tc::mma_commit_pair(&sh->empty[s], 0x3);
                }
                if (!ok) break;
                tc::mma_commit_pair(&sh->p_full[b], 0x3);
            }
        }
    } else if (!skip && warp >= 2) {
        const int quarter = warp & 3;
        const int part = (warp - 2) >> 2;          // columns part*64 .. +63
        const int row = quarter * 32 + lane;
        const uint32_t pe0 = tc::mapa_shared(tc::smem_u32(&sh->p_empty[0]), 0);
        const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16) + part * kLColsPerWarp;
        const bool noisy = p.scale != 0.f;
        // the pair's second tile starts from its noise, written into buffer 1
        // while the tensor cores accumulate the first tile
        if (noisy && pair + npairs < ntiles) write_tile_noise(p, pair + npairs, rank, row, part, tq + kAccCols);
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(pe0 + (uint32_t)sizeof(uint64_t));
        uint32_t rc = 0;
        for (int g = pair; g < ntiles; g += npairs, ++rc) {
            const int l = layer_of(p, g);
            const SumLayer& ly = p.L[l];
            int mb, nb;
            tile_coords(g - p.tile_begin[l], ly.m_blocks, ly.n_blocks, mb, nb);
            const int64_t m = (int64_t)mb * kPairTile + (int64_t)rank * kHalf + row;
            const int64_t n0 = (int64_t)nb * kPairTile + part * kLColsPerWarp;
            const uint32_t b = rc & 1u, bph = (rc >> 1) & 1u;
            if (!tc::mbar_wait_warp(&sh->p_full[b], bph, abort_flag, p.status)) break;
            tc::tc_fence_after();
            const uint32_t tb = tq + b * kAccCols;
            // the pair's first tile takes its noise here, 16 coordinates at a
            // time, while the tensor cores accumulate the next tile; the others
            // already hold theirs
            const bool add_noise = noisy && rc == 0;
            // the warp's 32 rows x 16 columns pass through its staging block so
            // that each store instruction writes 8 rows x 64 contiguous bytes
            const int64_t m_top = m - lane;
            float4* stg = reinterpret_cast<float4*>(staging) + (warp - 2) * 128;
#pragma unroll 1
            for (int ch = 0; ch < kLColsPerWarp / 16; ++ch) {
                float v[16];
                tc::tmem_ld16(tb + ch * 16, v);
                if (add_noise) {
                    float za[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, zb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    if (m < ly.d_out) {
                        const uint64_t k = (uint64_t)(ly.coord_off + m * ly.d_in + n0 + ch * 16);
                        noise8(p.seed, p.step, k, za);
                        noise8(p.seed, p.step, k + 8, zb);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[j] = v[j] + p.scale * za[j];
                        v[8 + j] = v[8 + j] + p.scale * zb[j];
                    }
                }
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    float4 o;
                    o.x = v[4 * j4] * p.inv_L;
                    o.y = v[4 * j4 + 1] * p.inv_L;
                    o.z = v[4 * j4 + 2] * p.inv_L;
                    o.w = v[4 * j4 + 3] * p.inv_L;
                    stg[lane * 4 + (j4 ^ ((lane >> 1) & 3))] = o;
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = i * 8 + (lane >> 2), q = lane & 3;
                    const float4 o = stg[r * 4 + (q ^ ((r >> 1) & 3))];
                    const int64_t mr = m_top + r;
                    const int64_t n = n0 + ch * 16 + q * 4;
                    if (mr < ly.d_out) {
                        float* dst = ly.G + mr * ly.d_in + n;
                        if (n + 4 <= ly.d_in) {
                            *reinterpret_cast<float4*>(dst) = o;
                        } else {
                            if (n < ly.d_in) dst[0] = o.x;
                            if (n + 1 < ly.d_in) dst[1] = o.y;
                            if (n + 2 < ly.d_in) dst[2] = o.z;
                        }
                    }
                }
                __syncwarp();
            }
            // buffer b is read; the tile two places later in the pair's list
            // reuses it and starts from its noise
            if (noisy && g + 2 * npairs < ntiles) write_tile_noise(p, g + 2 * npairs, rank, row, part, tb);
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(pe0 + (uint32_t)(b * sizeof(uint64_t)));
        }
    }

    if (!skip && warp == 1 && lane == 0) {
        if (rank == 0) tc::mma_commit_pair(&sh->drain, 0x3);
        tc::mbar_wait_drain(&sh->drain, 0);
    }
    tc::tc_fence_before();
    __syncthreads();
    // neither CTA leaves (nor frees its TMEM) while the pair's MMAs, copies or
    // arrivals may still touch it
    tc::cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tmem, 2 * kAccCols);
    }
}

// ============================================== per-record fold on CTA pairs
// T % 64 == 0 and B > 1: every record spans whole 64-row K tiles.  The tensor
// cores accumulate each record's unscaled partial P_i = E_i^T A_i in TMEM
// (two buffers) and the epilogue warps fold S += c_i * P_i in fp32
// registers: the clip factor is applied exactly, without rounding a scaled
// operand back to bf16.  Clusters of two CTAs with the operand staging and
// MMAs of k_sum_layers_pair_tc: 256 x 256 output tiles, each CTA staging its
// 128 columns of E and A per K step, its TMEM receiving its 128 rows of every
// record's partial, its epilogue warps folding those rows.  The record-range
// split of the last partial wave (see "work split") works per pair tile; each
// CTA of a pair keeps its half's partial sum in its own scratch slot, and the
// arrival counters are per (tile, half), so the CTA arriving last among the
// ranges of a half adds that half's slots in range order.
//
// Eight epilogue warps, two per TMEM lane quarter, each folding 128 of the
// 256 columns into 128 fp32 registers (with sixteen warps of 64 columns the
// dense 4096 x 4096 layer's sum took 2.8% longer); the tile's noise joins S
// four columns at a time after each of the first 32 records.
constexpr int kFEpiWarps = 8;
constexpr int kFColsPerWarp = kBN / (kFEpiWarps / 4);
constexpr int kFThreads = 32 * (2 + kFEpiWarps);
constexpr int kFNoiseChunks = kFColsPerWarp / 4;
constexpr int kFoldPairStages = 6;

struct FoldPairSmem {
    uint64_t full[kFoldPairStages];
    uint64_t empty[kFoldPairStages];
    uint64_t p_full[2];
    uint64_t p_empty[2];
    uint64_t drain;
    uint64_t fix_in;
    uint64_t fix_out;
    uint32_t tmem_base;
    int abort_flag;
    int fix_last;
};
static_assert(sizeof(FoldPairSmem) <= 256, "pair fold barriers exceed their shared-memory slot");
constexpr size_t kFoldPairSmem = 1024 + (size_t)kFoldPairStages * kPairStageBytes + 256;

// next_work over CTA pairs: whole pair tiles pair, pair + npairs, ... below
// full_tiles, then (with nsplit > 1) pair < R * nsplit takes record range
// pair / R of the remaining tile full_tiles + pair % R
__device__ __forceinline__ bool next_pair_work(const SumParams& p, int ntiles, int64_t B, int pair, int npairs,
                                               int& cursor, Work& w) {
    if (cursor < p.full_tiles) {
        w.tile = cursor;
        w.seg = -1;
        w.r0 = 0;
        w.r1 = B;
        cursor += npairs;
        return true;
    }
    if (cursor == INT_MAX || p.nsplit < 2) return false;
    cursor = INT_MAX;
    const int R = ntiles - p.full_tiles;
    if (pair >= R * p.nsplit) return false;
    w.tile = p.full_tiles + pair % R;
    w.seg = pair / R;
    w.r0 = (int64_t)w.seg * B / p.nsplit;
    w.r1 = (int64_t)(w.seg + 1) * B / p.nsplit;
    return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFThreads, 1)
    k_clipped_sum_fold_pair_tc(const __grid_constant__ SumParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    FoldPairSmem* sh = reinterpret_cast<FoldPairSmem*>(tiles + (size_t)kFoldPairStages * kPairStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_ctarank();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int ntiles = p.m_blocks * p.n_blocks;
    const int kpr = (int)((p.T + kBK - 1) / kBK);
    const int64_t B = p.K / p.T;
    volatile int* abort_flag = &sh->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFoldPairStages; ++s) {
            tc::mbar_init(&sh->full[s], 1);
            tc::mbar_init(&sh->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sh->p_full[b], 1);
            tc::mbar_init(&sh->p_empty[b], 2 * kFEpiWarps);
        }
        tc::mbar_init(&sh->drain, 1);
        tc::mbar_init(&sh->fix_in, 32 * kFEpiWarps);
        tc::mbar_init(&sh->fix_out, 1);
        sh->abort_flag = 0;
        sh->fix_last = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&p.tmE);
        tc::tma_prefetch_desc(&p.tmA);
    }
    if (warp == 1) tc::tmem_alloc_pair(&sh->tmem_base, 2 * kAccCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();
    tc::tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    grid_dep_wait();
    grid_dep_trigger();
    const bool skip = status_bad(p.status);

    if (!skip && warp == 0) {
        if (lane == 0) {
            const uint32_t full0 = tc::mapa_shared(tc::smem_u32(&sh->full[0]), 0);
            uint32_t it = 0;
            tc::StageRing<kFoldPairStages> ring;
            int cursor = pair;
            Work wk;
            while (next_pair_work(p, ntiles, B, pair, npairs, cursor, wk)) {
                int mb, nb;
                tile_coords(wk.tile, p.m_blocks, p.n_blocks, mb, nb);
                const int kt_end = (int)(wk.r1 * kpr);
                for (int kt = (int)(wk.r0 * kpr); kt < kt_end; ++kt, ++it, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->empty[s], ring.ph ^ 1u, abort_flag, p.status)) goto fold_pair_producer_done;
                    uint8_t* st = tiles + (size_t)s * kPairStageBytes;
                    if (rank == 0) tc::mbar_arrive_expect_tx(&sh->full[s], 2 * kPairStageBytes);
                    const uint32_t fb = full0 + (uint32_t)(s * sizeof(uint64_t));
                    const int k0 = kt * kBK;
                    if (p.box3d) {
                        tc::tma_load_3d_pair(st, &p.tmE, fb, 0, k0, mb * (kPairTile / 64) + (int)rank * (kHalf / 64));
                        tc::tma_load_3d_pair(st + kPairEStage, &p.tmA, fb, 0, k0,
                                             nb * (kPairTile / 64) + (int)rank * (kHalf / 64));
                    } else {
                        const int xe = mb * kPairTile + (int)rank * kHalf, xa = nb * kPairTile + (int)rank * kHalf;
                        tc::tma_load_2d_pair(st, &p.tmE, fb, xe, k0);
                        tc::tma_load_2d_pair(st + 8192, &p.tmE, fb, xe + 64, k0);
                        tc::tma_load_2d_pair(st + kPairEStage, &p.tmA, fb, xa, k0);
                        tc::tma_load_2d_pair(st + kPairEStage + 8192, &p.tmA, fb, xa + 64, k0);
                    }
                }
            }
        fold_pair_producer_done:
            if (rank == 0)
                for (uint32_t j = it > kFoldPairStages ? it - kFoldPairStages : 0; j < it; ++j)
                    tc::mbar_wait_drain(&sh->full[j % kFoldPairStages], (j / kFoldPairStages) & 1u);
        }
    } else if (!skip && warp == 1) {
        if (lane == 0 && rank == 0) {
            uint32_t rc = 0;
            tc::StageRing<kFoldPairStages> ring;
            const uint32_t tiles_u32 = tc::smem_u32(tiles);
            int cursor = pair;
            Work wk;
            while (next_pair_work(p, ntiles, B, pair, npairs, cursor, wk)) {
                bool ok = true;
                for (int64_t i = wk.r0; i < wk.r1 && ok; ++i, ++rc) {
                    const uint32_t b = rc & 1u, bph = (rc >> 1) & 1u;
                    if (!tc::mbar_wait(&sh->p_empty[b], bph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t d_tmem = tmem + b * kAccCols;
                    for (int kt = 0; kt < kpr; ++kt, ring.next()) {
                        const uint32_t s = ring.s;
                        if (!tc::mbar_wait(&sh->full[s], ring.ph, abort_flag, p.status)) { ok = false; break; }
                        tc::tc_fence_after();
                        const uint32_t sa = tiles_u32 + s * (uint32_t)kPairStageBytes;
                        const uint64_t ad = tc::smem_desc(sa, 8192, 1024, tc::SW_128B);
                        const uint64_t bd = tc::smem_desc(sa + kPairEStage, 8192, 1024, tc::SW_128B);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc::mma_bf16_pair(d_tmem, tc::desc_advance(ad, kk * 2048), tc::desc_advance(bd, kk * 2048),
                                              kIdescPair, (kt | kk) != 0);
                        tc::mma_commit_pair(&sh->empty[s], 0x3);
                    }
                    if (!ok) break;
                    tc::mma_commit_pair(&sh->p_full[b], 0x3);
                }
                if (!ok) break;
            }
        }
    } else if (!skip && warp >= 2) {
        const int quarter = warp & 3;
        const int part = (warp - 2) >> 2;          // columns part*64 .. +63
        const int row = quarter * 32 + lane;
        const uint32_t pe0 = tc::mapa_shared(tc::smem_u32(&sh->p_empty[0]), 0);
        uint32_t rc = 0, fix_phase = 0;
        int cursor = pair;
        Work wk;
        while (next_pair_work(p, ntiles, B, pair, npairs, cursor, wk)) {
            int mb, nb;
            tile_coords(wk.tile, p.m_blocks, p.n_blocks, mb, nb);
            const int64_t m = (int64_t)mb * kPairTile + (int64_t)rank * kHalf + row;
            const int64_t n0 = (int64_t)nb * kPairTile + part * kFColsPerWarp;
            const uint64_t k0 = (uint64_t)(p.coord_off + m * p.d_in + n0);   // this thread's first coordinate
            // the range holding the tile's first record also carries its noise
            const bool noisy = wk.r0 == 0 && m < p.d_out;
            float S[kFColsPerWarp];
#pragma unroll
            for (int j = 0; j < kFColsPerWarp; ++j) S[j] = 0.f;
            bool ok = true;
            for (int64_t i = wk.r0; i < wk.r1; ++i, ++rc) {
                const uint32_t b = rc & 1u, bph = (rc >> 1) & 1u;
                if (!tc::mbar_wait_warp(&sh->p_full[b], bph, abort_flag, p.status)) { ok = false; break; }
                tc::tc_fence_after();
                const float ci = __ldca(p.c + i);
                const uint32_t tb =
                    tmem + ((uint32_t)(quarter * 32) << 16) + b * kAccCols + part * kFColsPerWarp;
#pragma unroll
                for (int ch = 0; ch < kFColsPerWarp / 16; ++ch) {
                    float v[16];
                    tc::tmem_ld16(tb + ch * 16, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) S[ch * 16 + j] = fmaf(ci, v[j], S[ch * 16 + j]);
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(pe0 + (uint32_t)(b * sizeof(uint64_t)));
                if (noisy && i < kFNoiseChunks) add_noise_chunk_n<kFColsPerWarp>(p, k0, (int)i, S);
            }
            if (!ok) break;
            if (noisy)
                for (int q = (int)(wk.r1 < kFNoiseChunks ? wk.r1 : kFNoiseChunks); q < kFNoiseChunks; ++q)
                    add_noise_chunk_n<kFColsPerWarp>(p, k0, q, S);
            if (wk.seg >= 0) {
                // split tile: this half's partial sum to the CTA's slot, then the half's counter
                const int R = ntiles - p.full_tiles;
                const int r = wk.tile - p.full_tiles;
                float* slot = p.scratch + (size_t)blockIdx.x * (kBM * kBN);
#pragma unroll
                for (int j = 0; j < kFColsPerWarp; ++j) slot[(size_t)(part * kFColsPerWarp + j) * kBM + row] = S[j];
                __threadfence();
                tc::mbar_arrive(&sh->fix_in);
                if (warp == 2 && lane == 0) {
                    int last = 0;
                    if (tc::mbar_wait(&sh->fix_in, fix_phase, abort_flag, p.status)) {
                        __threadfence();
                        unsigned long long* cp = p.counters + 2 * r + (int)rank;
                        unsigned long long seen = *(volatile unsigned long long*)cp, prev;
                        do {
                            prev = seen;
                            const unsigned long long want = (unsigned)(prev >> 32) == p.epoch
                                                                ? prev + 1
                                                                : ((unsigned long long)p.epoch << 32) | 1ull;
                            seen = atomicCAS(cp, prev, want);
                        } while (seen != prev);
                        const unsigned before = (unsigned)(prev >> 32) == p.epoch ? (unsigned)prev : 0u;
                        last = before + 1 == (unsigned)p.nsplit ? 1 : 0;
                        __threadfence();
                    }
                    *(volatile int*)&sh->fix_last = last;
                    tc::mbar_arrive(&sh->fix_out);
                }
                const bool waited = tc::mbar_wait_warp(&sh->fix_out, fix_phase, abort_flag, p.status);
                fix_phase ^= 1u;
                if (!waited) break;
                if (!*(volatile int*)&sh->fix_last) continue;
                // last arrival for this half: the ranges' partial sums in range order
#pragma unroll
                for (int j = 0; j < kFColsPerWarp; ++j) S[j] = 0.f;
                for (int sg = 0; sg < p.nsplit; ++sg) {
                    const float* src = p.scratch + (size_t)(2 * (r + sg * R) + (int)rank) * (kBM * kBN);
#pragma unroll
                    for (int j = 0; j < kFColsPerWarp; ++j)
                        S[j] += __ldcg(src + (size_t)(part * kFColsPerWarp + j) * kBM + row);
                }
            }
            if (m < p.d_out) {
#pragma unroll
                for (int ch = 0; ch < kFColsPerWarp / 8; ++ch) {
                    const int64_t n = n0 + ch * 8;
                    if (n >= p.d_in) continue;
                    float* out = p.G + m * p.d_in + n;
                    if (n + 8 <= p.d_in) {
#pragma unroll
                        for (int j = 0; j < 8; j += 4) {
                            float4 o;
                            o.x = S[ch * 8 + j] * p.inv_L;
                            o.y = S[ch * 8 + j + 1] * p.inv_L;
                            o.z = S[ch * 8 + j + 2] * p.inv_L;
                            o.w = S[ch * 8 + j + 3] * p.inv_L;
                            *reinterpret_cast<float4*>(out + j) = o;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (n + j < p.d_in) out[j] = S[ch * 8 + j] * p.inv_L;
                    }
                }
            }
        }
    }

    if (!skip && warp == 1 && lane == 0) {
        if (rank == 0) tc::mma_commit_pair(&sh->drain, 0x3);
        tc::mbar_wait_drain(&sh->drain, 0);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tmem, 2 * kAccCols);
    }
}

// ============================================================ host side
bool encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
            const uint32_t* box, CUtensorMapSwizzle swz) {
    const EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t gd[3], gs[2];
    cuuint32_t bd[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bd[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bd,
                          es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// SMs of the current device
int sm_count_cached() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

bool tc_sum_supported(int dtype, int64_t d_in, int64_t d_out, int has_bias) {
    (void)has_bias;
    return dtype == DT_BF16 && d_in % 8 == 0 && d_out % 8 == 0 && d_in >= 64 && d_out >= 64;
}

bool tc_encode_sum(const GradTask& t, int64_t B, CUtensorMap* maps3) {
    const int64_t K = B * t.T;
    if (t.d_in % 64 == 0 && t.d_out % 64 == 0) {
        // {64 columns, K rows, 64-column chunks}: one copy brings a whole
        // tile (E: 128 columns; A: 256 columns, or 128 for a CTA of a pair)
        const uint32_t be[3] = {64, (uint32_t)kBK, (uint32_t)(kBM / 64)};
        const uint32_t ba[3] = {64, (uint32_t)kBK, (uint32_t)(kBN / 64)};
        const uint32_t bh[3] = {64, (uint32_t)kBK, (uint32_t)(kHalf / 64)};
        const uint64_t de[3] = {64, (uint64_t)K, (uint64_t)(t.d_out / 64)};
        const uint64_t se[2] = {(uint64_t)t.d_out * 2, 128};
        const uint64_t da[3] = {64, (uint64_t)K, (uint64_t)(t.d_in / 64)};
        const uint64_t sa[2] = {(uint64_t)t.d_in * 2, 128};
        return encode(&maps3[0], t.E, 3, de, se, be, CU_TENSOR_MAP_SWIZZLE_128B) &&
               encode(&maps3[1], t.A, 3, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_128B) &&
               encode(&maps3[2], t.A, 3, da, sa, bh, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    const uint32_t box[2] = {64, (uint32_t)kBK};
    const uint64_t de[2] = {(uint64_t)t.d_out, (uint64_t)K};
    const uint64_t se[1] = {(uint64_t)t.d_out * 2};
    const uint64_t da[2] = {(uint64_t)t.d_in, (uint64_t)K};
    const uint64_t sa[1] = {(uint64_t)t.d_in * 2};
    if (!encode(&maps3[0], t.E, 2, de, se, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&maps3[1], t.A, 2, da, sa, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    maps3[2] = maps3[1];
    return true;
}

size_t fold_scratch_floats(int sms) { return (size_t)sms * kBM * kBN; }

int device_sm_count() { return sm_count_cached(); }

// Clusters of two CTAs of a pair kernel resident at once on the current
// device (queried once per device and kernel, kept in `cache`; half the SM
// count if the query fails).
static int pair_clusters_cached(const void* kern, int threads, int smem, std::atomic<int> (&cache)[64]) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)sm_count_cached());
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = sm_count_cached() / 2;
        if (n < 1) n = 1;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// records mode (B > 1, T % 64 == 0) on CTA pairs; work == nullptr: every
// tile is done whole by one pair
static cudaError_t launch_fold_pair(const GradTask& t, const float* c, unsigned* status, const StepScalars& sc,
                                   const FoldWork* work, cudaStream_t s) {
    const void* kern = reinterpret_cast<const void*>(k_clipped_sum_fold_pair_tc);
    {
        const cudaError_t a = ensure_smem_limit(kern, (int)kFoldPairSmem);
        if (a != cudaSuccess) return a;
    }
    SumParams p;
    if (t.maps) {
        p.tmE = t.maps[0];
        p.tmA = t.maps[2];
    } else {
        CUtensorMap m[3];
        if (!tc_encode_sum(t, sc.B, m)) return cudaErrorInvalidValue;
        p.tmE = m[0];
        p.tmA = m[2];
    }
    p.K = sc.B * t.T;
    p.T = t.T;
    p.box3d = (t.d_in % 64 == 0 && t.d_out % 64 == 0) ? 1 : 0;
    p.d_in = t.d_in;
    p.d_out = t.d_out;
    p.m_blocks = (int)((t.d_out + kPairTile - 1) / kPairTile);
    p.n_blocks = (int)((t.d_in + kPairTile - 1) / kPairTile);
    p.c = c;
    p.status = status;
    p.G = t.G;
    p.coord_off = t.coord_off;
    p.scale = sc.sigma * sc.C;
    p.inv_L = 1.0f / sc.L;
    p.seed = sc.seed;
    p.step = sc.step;
    const int ntiles = p.m_blocks * p.n_blocks;
    static std::atomic<int> clusters[64];
    const int pairs = pair_clusters_cached(kern, kFThreads, (int)kFoldPairSmem, clusters);
    int npairs = ntiles < pairs ? ntiles : pairs;
    p.full_tiles = ntiles;
    p.nsplit = 1;
    p.scratch = nullptr;
    p.counters = nullptr;
    p.epoch = 0;
    if (work != nullptr && 2 * pairs <= sm_count_cached()) {
        // split the R pair tiles of a partial last wave into pairs / R record
        // ranges (each at least 8 K tiles) when the wave would leave over 4%
        // of the pair slots idle; a CTA's scratch slot and a (tile, half)
        // counter are indexed below the SM count
        const int R = ntiles % pairs;
        const int waves = (ntiles + pairs - 1) / pairs;
        const double idle = (double)((int64_t)waves * pairs - ntiles) / ((double)waves * pairs);
        const int64_t kpr = (t.T + kBK - 1) / kBK;
        int S = R > 0 ? pairs / R : 1;
        while (S > 1 && (sc.B / S) * kpr < 8) --S;
        if (R > 0 && S >= 2 && idle > 0.04) {
            p.full_tiles = ntiles - R;
            p.nsplit = S;
            p.scratch = work->scratch;
            p.counters = work->counters;
            p.epoch = work->epoch;
            npairs = pairs;
        }
    }
    const cudaError_t e = launch_dependent(k_clipped_sum_fold_pair_tc, dim3(2 * npairs), dim3(kFThreads), kFoldPairSmem, s, p);
    count_launch(KL_CLIPPED_SUM_FOLD_PAIR_TC);
    return e;
}

cudaError_t launch_clipped_sum_tc(const GradTask& t, const float* c, unsigned* status, const StepScalars& sc,
                                  const FoldWork* work, cudaStream_t s) {
    if (sc.B > 1) return launch_fold_pair(t, c, status, sc, work, s);
    // one record of t.T rows (with factor c[0])
    {
        const cudaError_t a = ensure_smem_limit(reinterpret_cast<const void*>(k_clipped_sum_tc), (int)kSumSmem);
        if (a != cudaSuccess) return a;
    }
    SumParams p;
    if (t.maps) {
        p.tmE = t.maps[0];
        p.tmA = t.maps[1];
    } else {
        CUtensorMap m[3];
        if (!tc_encode_sum(t, 1, m)) return cudaErrorInvalidValue;
        p.tmE = m[0];
        p.tmA = m[1];
    }
    p.K = t.T;
    p.T = t.T;
    p.box3d = (t.d_in % 64 == 0 && t.d_out % 64 == 0) ? 1 : 0;
    p.d_in = t.d_in;
    p.d_out = t.d_out;
    p.m_blocks = (int)((t.d_out + kBM - 1) / kBM);
    p.n_blocks = (int)((t.d_in + kBN - 1) / kBN);
    p.c = c;
    p.status = status;
    p.G = t.G;
    p.coord_off = t.coord_off;
    p.scale = sc.sigma * sc.C;
    p.inv_L = 1.0f / sc.L;
    p.seed = sc.seed;
    p.step = sc.step;
    p.full_tiles = p.m_blocks * p.n_blocks;
    p.nsplit = 1;
    p.scratch = nullptr;
    p.counters = nullptr;
    p.epoch = 0;
    const int ntiles = p.full_tiles;
    const int sms = sm_count_cached();
    const int grid = ntiles < sms ? ntiles : sms;
    const cudaError_t e = launch_dependent(k_clipped_sum_tc, dim3(grid), dim3(kFoldThreads), kSumSmem, s, p);
    count_launch(KL_CLIPPED_SUM_TC);
    return e;
}

cudaError_t launch_sum_layers_tc(const GradTask* tasks, int n, unsigned* status, const StepScalars& sc,
                                 cudaStream_t s) {
    if (n < 1 || n > kMaxSumLayers) return cudaErrorInvalidValue;
    const void* kern = reinterpret_cast<const void*>(k_sum_layers_pair_tc);
    {
        const cudaError_t a = ensure_smem_limit(kern, (int)kPairSmem);
        if (a != cudaSuccess) return a;
    }
    LayersParams p;
    p.nlayers = n;
    const int64_t K = tasks[0].T;   // one record of K rows with factor 1
    p.nk = (int)((K + kBK - 1) / kBK);
    int tiles = 0;
    for (int l = 0; l < n; ++l) {
        const GradTask& t = tasks[l];
        if (t.T != K) return cudaErrorInvalidValue;
        SumLayer& L = p.L[l];
        if (t.maps) {
            L.tmE = t.maps[0];
            L.tmA = t.maps[2];
        } else {
            CUtensorMap m[3];
            if (!tc_encode_sum(t, 1, m)) return cudaErrorInvalidValue;
            L.tmE = m[0];
            L.tmA = m[2];
        }
        L.d_in = t.d_in;
        L.d_out = t.d_out;
        L.m_blocks = (int)((t.d_out + kPairTile - 1) / kPairTile);
        L.n_blocks = (int)((t.d_in + kPairTile - 1) / kPairTile);
        L.box3d = (t.d_in % 64 == 0 && t.d_out % 64 == 0) ? 1 : 0;
        L.G = t.G;
        L.coord_off = t.coord_off;
        p.tile_begin[l] = tiles;
        tiles += L.m_blocks * L.n_blocks;
    }
    p.tile_begin[n] = tiles;
    p.status = status;
    p.scale = sc.sigma * sc.C;
    p.inv_L = 1.0f / sc.L;
    p.seed = sc.seed;
    p.step = sc.step;
    static std::atomic<int> clusters[64];
    const int pairs = pair_clusters_cached(kern, kLThreads, (int)kPairSmem, clusters);
    const int grid = 2 * (tiles < pairs ? tiles : pairs);
    const cudaError_t e = launch_dependent(k_sum_layers_pair_tc, dim3(grid), dim3(kLThreads), kPairSmem, s, p);
    count_launch(KL_SUM_LAYERS_PAIR_TC);
    return e;
}
