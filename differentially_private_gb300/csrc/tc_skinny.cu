// Materialized per-example gradients of low-rank (LoRA) factors on the
// tensor cores (tcgen05 + TMA), for layers where the chooser materializes
// (T^2 >= d_in * d_out) and one side is a rank r of 8 or 16:
//
//   g_i = E_i^T A_i,   ||g_i||_F^2,   and g_i kept for the weighted sum
//
// ("Privacy-Preserving Machine Learning", section "Differentially private
// stochastic gradient descent", phase 2: per-sample gradients).  With D the
// large side, X the [T, D] operand (A for LoRA-A, E for LoRA-B) and Y the
// [T, r] operand, the kernel computes g_i^T or g_i as X_i^T Y_i: M = 128
// columns of X per MMA, N = 16 (r padded with the TMA's zero fill), K = T.
//
// The 128-column blocks of D of every (layer, record) of the launch form one
// index space; each CTA takes a contiguous range of it, so the CTAs' loads
// differ by at most one block.  Work item = a run of at most item_cap blocks
// of one (layer, record) inside the CTA's range.  Stages walk an item k-tile
// by k-tile and, inside a k-tile, block by block, so the blocks of one
// 64-row slab are read back to back (whole rows of X in DRAM order).  Y has
// its own small ring and is loaded once per k-tile for all blocks.  Each
// block accumulates into its own 16 TMEM columns; items rotate through four
// accumulator sets.  One launch serves up to kMaxSkinnyGroup layers.
//
// The epilogue writes one partial squared norm per (record, block, epilogue
// warp) -- no barrier, no atomics: a record's norm depends only on its own
// rows ("Sensitivity Inflation from Cross-Record Precision Routing in
// Private Quantized Fine-Tuning", Proposition 2).
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 2-5 epilogue.
#include "common.cuh"
#include "launch.cuh"
#include "tc_common.cuh"

using namespace dpk;

namespace {

constexpr int kBM = 128, kBN = 16, kBK = 64;
constexpr int kXStages = 8;                 // 16 KB: 128 columns x 64 rows (two 64-column boxes)
constexpr int kYStages = 4;                 //  2 KB: 16 columns x 64 rows, 32-byte swizzle
constexpr int kXStage = kBM * kBK * 2;
constexpr int kYStage = kBN * kBK * 2;
constexpr int kMaxMb = 8;                   // column blocks per work item (TMEM columns of one set)
constexpr int kEpiGroup = 4;                // blocks whose TMEM columns the epilogue loads at once (tmem_ld16x4)
constexpr int kAccSets = 4;                 // the MMAs run up to three items ahead of the epilogue
constexpr uint32_t kTmemCols = 512;         // kAccSets * kMaxMb * kBN
constexpr int kThreads = 192;
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kBM, kBN, 1, 1);
constexpr size_t kSmem = 1024 + (size_t)kXStages * kXStage + (size_t)kYStages * kYStage + 8192 + 512;

struct SkinnyLayer {
    CUtensorMap tmX;   // {D, T, B}, box {64, 64, 1}, 128-byte swizzle
    CUtensorMap tmY;   // {r, T, B}, box {16, 64, 1}, 32-byte swizzle
    int64_t T, D, r;
    int x_is_A;        // 1: X = A (d_in = D, d_out = r); 0: X = E (d_out = D, d_in = r)
    int mblocks;       // 128-column blocks of D
    int item_cap;      // blocks per work item, at most kMaxMb
    float* partial;    // [B][mblocks * 4]
    float* gstore;     // [B][r * D] or nullptr
};

struct SkinnyParams {
    int nlayers;
    unsigned* status;
    // first block of each layer (+ the total): kept apart from the layer
    // records so that the search for a CTA's first layer reads a few cache
    // lines of the parameter bank, not one line per layer
    int64_t blk_begin[kMaxSkinnyGroup + 1];
    SkinnyLayer L[kMaxSkinnyGroup];
};

struct Smem {
    alignas(16) float gstage[4][32 * kBN];   // per epilogue warp: 32 rows x r of g before a coalesced store
    uint64_t full[kXStages];
    uint64_t empty[kXStages];
    uint64_t yfull[kYStages];
    uint64_t yempty[kYStages];
    uint64_t acc_full[kAccSets];
    uint64_t acc_empty[kAccSets];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int l_first;                             // layer of the CTA's first item
    int warm[32];                            // sink of the parameter-bank warm-up loads
};

static_assert(sizeof(Smem) <= 8192 + 512, "skinny kernel shared-memory budget");

// Layer of a block, found by a whole warp: lane i compares blk_begin[1 + i],
// blk_begin[33 + i] with the block (parallel parameter-bank reads instead of
// a chain of dependent ones) and the ballots count the layers starting at or
// before it.
__device__ __forceinline__ int warp_find_layer(const SkinnyParams& p, int64_t q, int lane) {
    int l = 0;
    for (int base = 1; base < p.nlayers; base += 32) {
        const int j = base + lane;
        l += __popc(__ballot_sync(0xffffffffu, j < p.nlayers && p.blk_begin[j] <= q));
    }
    return l;
}

struct ItemInfo {
    int rec, mb0, nmb, nk;
};

// The next item of a CTA's block range [q, hi): the run of blocks of one
// (layer, record) starting at block q, at most item_cap long.  Blocks of a
// CTA increase, so the layer cursor l only moves forward.
__device__ __forceinline__ bool next_item(const SkinnyParams& p, int64_t& q, int64_t hi, int& l, ItemInfo& in) {
    if (q >= hi) return false;
    while (l + 1 < p.nlayers && p.blk_begin[l + 1] <= q) ++l;
    const SkinnyLayer& ly = p.L[l];
    const int64_t local = q - p.blk_begin[l];
    in.rec = (int)(local / ly.mblocks);
    in.mb0 = (int)(local - (int64_t)in.rec * ly.mblocks);
    int n = ly.mblocks - in.mb0;
    if (n > ly.item_cap) n = ly.item_cap;
    if ((int64_t)n > hi - q) n = (int)(hi - q);
    in.nmb = n;
    in.nk = (int)((ly.T + kBK - 1) / kBK);
    q += n;
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) k_mat_skinny_tc(const __grid_constant__ SkinnyParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* xs = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ys = xs + (size_t)kXStages * kXStage;
    Smem* sh = reinterpret_cast<Smem*>(ys + (size_t)kYStages * kYStage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &sh->abort_flag;
    // each CTA takes one contiguous range of blocks: consecutive items share a
    // layer and its TMA descriptors
    const int64_t total = p.blk_begin[p.nlayers];
    const int64_t blk_lo = (int64_t)blockIdx.x * total / gridDim.x;
    const int64_t blk_hi = (int64_t)(blockIdx.x + 1) * total / gridDim.x;

    // Warp 0 sets up the barriers, finds its first layer and starts loading
    // at once; the other warps meet at named barrier 1, which warp 0 passes
    // with an arrive (no wait), while warp 1 allocates TMEM and warp 2 pulls
    // the layers' descriptors and parameter lines into the caches.
    constexpr uint32_t kSetupBar = 1;
    int l_first = 0;
    uint32_t tmem = 0;
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < kXStages; ++s) {
                tc::mbar_init(&sh->full[s], 1);
                tc::mbar_init(&sh->empty[s], 1);
            }
            for (int s = 0; s < kYStages; ++s) {
                tc::mbar_init(&sh->yfull[s], 1);
                tc::mbar_init(&sh->yempty[s], 1);
            }
            for (int a = 0; a < kAccSets; ++a) {
                tc::mbar_init(&sh->acc_full[a], 1);
                tc::mbar_init(&sh->acc_empty[a], 128);
            }
            tc::mbar_init(&sh->drain, 1);
            sh->abort_flag = 0;
            tc::fence_barrier_init();
        }
        __syncwarp();
        tc::named_bar_arrive(kSetupBar, kThreads);
        l_first = blk_lo < blk_hi ? warp_find_layer(p, blk_lo, lane) : 0;
    } else {
        if (warp == 1) tc::tmem_alloc(&sh->tmem_base, kTmemCols);
        if (warp == 2) {
            const int lf = blk_lo < blk_hi ? warp_find_layer(p, blk_lo, lane) : 0;
            const int ll = blk_lo < blk_hi ? warp_find_layer(p, blk_hi - 1, lane) : -1;
            if (lane == 0) sh->l_first = lf;
            int acc = 0;
            for (int l = lf + lane; l <= ll; l += 32) {
                tc::tma_prefetch_desc(&p.L[l].tmX);
                tc::tma_prefetch_desc(&p.L[l].tmY);
                acc += p.L[l].mblocks + (int)p.blk_begin[l];
            }
            sh->warm[lane] = acc;
        }
        tc::tc_fence_before();
        tc::named_bar_sync(kSetupBar, kThreads);
        tc::tc_fence_after();
        tmem = sh->tmem_base;
        l_first = sh->l_first;
    }
    // the set-up above (which reads only the parameters) may overlap the
    // previous kernel of the stream; A and E are read only after it completed
    grid_dep_wait();
    grid_dep_trigger();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0, yit = 0;
            int cur = l_first;
            int64_t q = blk_lo;
            ItemInfo in;
            // A and E are read once: evict them first, keep the stored g in L2
            const uint64_t stream_policy = tc::l2_evict_first();
            while (next_item(p, q, blk_hi, cur, in)) {
                const SkinnyLayer& ly = p.L[cur];
                for (int kt = 0; kt < in.nk; ++kt) {
                    const int qs = yit % kYStages;
                    const uint32_t qph = (yit / kYStages) & 1u;
                    if (!tc::mbar_wait(&sh->yempty[qs], qph ^ 1u, abort_flag, p.status)) goto producer_done;
                    tc::mbar_arrive_expect_tx(&sh->yfull[qs], kYStage);
                    tc::tma_load_3d_hint(ys + (size_t)qs * kYStage, &ly.tmY, &sh->yfull[qs], 0, kt * kBK, in.rec,
                                         stream_policy);
                    ++yit;
                    for (int m = 0; m < in.nmb; ++m, ++it) {
                        const int s = it % kXStages;
                        const uint32_t ph = (it / kXStages) & 1u;
                        if (!tc::mbar_wait(&sh->empty[s], ph ^ 1u, abort_flag, p.status)) goto producer_done;
                        uint8_t* st = xs + (size_t)s * kXStage;
                        const int col = (in.mb0 + m) * kBM;
                        tc::mbar_arrive_expect_tx(&sh->full[s], kXStage);
                        tc::tma_load_3d_hint(st, &ly.tmX, &sh->full[s], col, kt * kBK, in.rec, stream_policy);
                        tc::tma_load_3d_hint(st + 8192, &ly.tmX, &sh->full[s], col + 64, kt * kBK, in.rec,
                                             stream_policy);
                    }
                }
            }
        producer_done:
            // every copy this thread issued lands before the CTA may exit
            for (uint32_t j = it > kXStages ? it - kXStages : 0; j < it; ++j)
                tc::mbar_wait_drain(&sh->full[j % kXStages], (j / kXStages) & 1u);
            for (uint32_t j = yit > kYStages ? yit - kYStages : 0; j < yit; ++j)
                tc::mbar_wait_drain(&sh->yfull[j % kYStages], (j / kYStages) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, yit = 0, lt = 0;
            int cur = l_first;
            int64_t q = blk_lo;
            ItemInfo in;
            bool ok = true;
            while (ok && next_item(p, q, blk_hi, cur, in)) {
                const uint32_t a = lt % kAccSets, aph = (lt / kAccSets) & 1u;
                ++lt;
                if (!tc::mbar_wait(&sh->acc_empty[a], aph ^ 1u, abort_flag, p.status)) break;
                tc::tc_fence_after();
                for (int kt = 0; kt < in.nk && ok; ++kt) {
                    const int qs = yit % kYStages;
                    const uint32_t qph = (yit / kYStages) & 1u;
                    if (!tc::mbar_wait(&sh->yfull[qs], qph, abort_flag, p.status)) { ok = false; break; }
                    const uint32_t sy = tc::smem_u32(ys + (size_t)qs * kYStage);
                    for (int m = 0; m < in.nmb; ++m, ++it) {
                        const int s = it % kXStages;
                        const uint32_t ph = (it / kXStages) & 1u;
                        if (!tc::mbar_wait(&sh->full[s], ph, abort_flag, p.status)) { ok = false; break; }
                        tc::tc_fence_after();
                        const uint32_t sx = tc::smem_u32(xs + (size_t)s * kXStage);
                        const uint32_t d_tmem = tmem + a * (kMaxMb * kBN) + m * kBN;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            // X: 128-byte swizzled, 16 rows = two 1 KB groups; Y: 32-byte rows, 16 rows = 512 B
                            const uint64_t ad = tc::smem_desc(sx + kk * 2048, 8192, 1024, tc::SW_128B);
                            const uint64_t bd = tc::smem_desc(sy + kk * 512, 2048, 256, tc::SW_32B);
                            tc::mma_bf16(d_tmem, ad, bd, kIdesc, (kt | kk) != 0);
                        }
                        tc::mma_commit(&sh->empty[s]);
                    }
                    if (!ok) break;
                    tc::mma_commit(&sh->yempty[qs]);
                    ++yit;
                }
                if (!ok) break;
                tc::mma_commit(&sh->acc_full[a]);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;
        const int ew = warp - 2;
        uint32_t lt = 0;
        int cur = l_first;
        int64_t q = blk_lo;
        ItemInfo in;
        while (next_item(p, q, blk_hi, cur, in)) {
            const SkinnyLayer& ly = p.L[cur];
            const uint32_t a = lt % kAccSets, aph = (lt / kAccSets) & 1u;
            ++lt;
            if (!tc::mbar_wait_warp(&sh->acc_full[a], aph, abort_flag, p.status)) break;
            tc::tc_fence_after();
            const int64_t ncl = ly.r * ly.D;
            float* g = ly.gstore ? ly.gstore + (int64_t)in.rec * ncl : nullptr;
            float* part = ly.partial + (int64_t)in.rec * ly.mblocks * 4;
            for (int m0 = 0; m0 < in.nmb; m0 += kEpiGroup) {
                // the TMEM columns of up to four blocks at once (columns past the
                // item's blocks are read but unused; they stay inside the set)
                float v[kEpiGroup][16];
                tc::tmem_ld16x4(tmem + ((uint32_t)(quarter * 32) << 16) + a * (kMaxMb * kBN) + m0 * kBN, v);
                float ss[kEpiGroup];
#pragma unroll
                for (int b = 0; b < kEpiGroup; ++b) {
                    const int m = m0 + b;
                    ss[b] = 0.f;
                    if (m >= in.nmb) continue;
                    const int mb = in.mb0 + m;
                    const int64_t d = (int64_t)mb * kBM + row;
                    if (d < ly.D) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < ly.r) ss[b] = fmaf(v[b][j], v[b][j], ss[b]);
                    }
                    if (g && ly.x_is_A) {
                        // entry (j, d) of g [r x D]: for each j the warp's 32 rows d are contiguous
                        if (d < ly.D) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < ly.r) g[(int64_t)j * ly.D + d] = v[b][j];
                        }
                    } else if (g) {
                        // entry (d, j) of g [D x r]: the warp's 32 rows are one contiguous run of
                        // 32 r floats; stage it in shared memory, then store it as float4s
                        float* stage = sh->gstage[ew];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < ly.r) stage[lane * ly.r + j] = v[b][j];
                        __syncwarp();
                        const int64_t d0 = (int64_t)mb * kBM + quarter * 32;
                        const int64_t nvalid = min((int64_t)32, ly.D - d0) * ly.r;   // floats of this warp's run
                        float* dst = g + d0 * ly.r;
                        for (int qq = lane; qq * 4 < nvalid; qq += 32)
                            *reinterpret_cast<float4*>(dst + 4 * qq) = *reinterpret_cast<const float4*>(stage + 4 * qq);
                        __syncwarp();
                    }
                }
                // the blocks' warp sums, butterflies interleaved (same order per block as one warp_sum)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int b = 0; b < kEpiGroup; ++b) ss[b] += __shfl_xor_sync(0xffffffffu, ss[b], o);
                if (lane == 0) {
#pragma unroll
                    for (int b = 0; b < kEpiGroup; ++b)
                        if (m0 + b < in.nmb) part[(in.mb0 + m0 + b) * 4 + ew] = ss[b];
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sh->acc_empty[a]);
        }
    }

    if (warp == 1 && lane == 0) {
        // no MMA may still be writing TMEM when it is released
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

bool encode3d(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swz) {
    const EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t gd[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t gs[2] = {strides[0], strides[1]};
    cuuint32_t bd[3] = {box[0], box[1], box[2]};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gd, gs, bd, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// Blocks per work item of a layer: the record's blocks in the fewest runs of
// at most four (one TMEM load group of the epilogue), as even as possible.
int item_cap(int mblocks) {
    const int runs = (mblocks + kEpiGroup - 1) / kEpiGroup;
    return (mblocks + runs - 1) / runs;
}

}  // namespace

bool tc_skinny_supported(int dtype, int64_t d_in, int64_t d_out, int has_bias) {
    if (dtype != DT_BF16 || has_bias) return false;
    const int64_t r = d_in < d_out ? d_in : d_out;
    const int64_t D = d_in < d_out ? d_out : d_in;
    return (r == 8 || r == 16) && D % 8 == 0 && D >= 64;
}

int nslots_skinny(int64_t d_in, int64_t d_out) {
    const int64_t D = d_in < d_out ? d_out : d_in;
    return (int)((D + kBM - 1) / kBM) * 4;   // one partial per (block, epilogue warp)
}

bool tc_encode_skinny(const NormTask& t, int64_t B, CUtensorMap* maps2) {
    const bool x_is_A = t.d_in > t.d_out;
    const int64_t D = x_is_A ? t.d_in : t.d_out;
    const int64_t r = x_is_A ? t.d_out : t.d_in;
    const void* X = x_is_A ? t.A : t.E;
    const void* Y = x_is_A ? t.E : t.A;
    const uint64_t xd[3] = {(uint64_t)D, (uint64_t)t.T, (uint64_t)B};
    const uint64_t xs[2] = {(uint64_t)D * 2, (uint64_t)(D * t.T * 2)};
    const uint32_t xb[3] = {64, (uint32_t)kBK, 1};
    const uint64_t yd[3] = {(uint64_t)r, (uint64_t)t.T, (uint64_t)B};
    const uint64_t ysr[2] = {(uint64_t)r * 2, (uint64_t)(r * t.T * 2)};
    const uint32_t yb[3] = {16, (uint32_t)kBK, 1};
    return encode3d(&maps2[0], X, xd, xs, xb, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode3d(&maps2[1], Y, yd, ysr, yb, CU_TENSOR_MAP_SWIZZLE_32B);
}

cudaError_t launch_mat_skinny_tc(const NormTask* tasks, int n, int64_t B, unsigned* status, cudaStream_t s) {
    {
        const cudaError_t a = ensure_smem_limit(reinterpret_cast<const void*>(k_mat_skinny_tc), (int)kSmem);
        if (a != cudaSuccess) return a;
    }
    thread_local SkinnyParams p;   // host staging of the parameter block; each launch copies it
    const int sms = sm_count();
    for (int base = 0; base < n; base += kMaxSkinnyGroup) {
        p.nlayers = n - base < kMaxSkinnyGroup ? n - base : kMaxSkinnyGroup;
        p.status = status;
        int64_t blocks = 0;
        for (int i = 0; i < p.nlayers; ++i) {
            const NormTask& t = tasks[base + i];
            SkinnyLayer& L = p.L[i];
            const bool x_is_A = t.d_in > t.d_out;
            L.x_is_A = x_is_A ? 1 : 0;
            L.D = x_is_A ? t.d_in : t.d_out;
            L.r = x_is_A ? t.d_out : t.d_in;
            L.T = t.T;
            L.mblocks = (int)((L.D + kBM - 1) / kBM);
            L.item_cap = item_cap(L.mblocks);
            p.blk_begin[i] = blocks;
            L.partial = t.partial;
            L.gstore = t.gstore;
            blocks += B * L.mblocks;
            if (t.maps) {
                L.tmX = t.maps[0];
                L.tmY = t.maps[1];
            } else {
                CUtensorMap m[2];
                if (!tc_encode_skinny(t, B, m)) return cudaErrorInvalidValue;
                L.tmX = m[0];
                L.tmY = m[1];
            }
        }
        p.blk_begin[p.nlayers] = blocks;
        const int grid = (int)(blocks < sms ? blocks : sms);
        const cudaError_t e = launch_dependent(k_mat_skinny_tc, dim3(grid), dim3(kThreads), kSmem, s, p);
        count_launch(KL_MAT_SKINNY_TC);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
