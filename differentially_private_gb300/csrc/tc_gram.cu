// Ghost norm on the tensor cores (tcgen05 + TMA), for layers with T > 1:
//
//   ||E_i^T A_i||_F^2 = <A_i A_i^T, E_i E_i^T>     (+ 1^T E_i E_i^T 1 for a bias)
//
// obtained without forming the per-example gradient ("Privacy-Preserving
// Machine Learning", section "Differentially private stochastic gradient
// descent", phase 2: ghost clipping).  Both T x T Grams are symmetric, so
// only the upper triangle is computed: work item = (record i, 128-row block
// p, 256-column block q) with p <= 2q + 1.  The two 128x128 halves of the
// tile get weight 2 above the diagonal, 1 on it and 0 below.  GA accumulates
// over d_in and GE over d_out in two TMEM accumulators; the epilogue reduces
// sum_{s,t} w GA[s,t] GE[s,t] (+ w GE[s,t]) to one partial per epilogue warp.
// A record's partials depend only on its own rows and the shapes, so its
// norm is the same for any batch ("Sensitivity Inflation from Cross-Record
// Precision Routing in Private Quantized Fine-Tuning", Proposition 2).
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 2-5 epilogue.
#include "common.cuh"
#include "launch.cuh"
#include "tc_common.cuh"

using namespace dpk;

namespace {

constexpr int kGM = 128, kGN = 256, kGK = 64, kGStages = 4;
constexpr int kGAStage = kGM * kGK * 2;   // 16 KB: 128 rows x 64 features, 128B swizzle
constexpr int kGBStage = kGN * kGK * 2;   // 32 KB: 256 rows
constexpr int kGStageBytes = kGAStage + kGBStage;
constexpr int kGThreads = 192;
constexpr uint32_t kIdescGram = tc::idesc_bf16_f32(kGM, kGN, 0, 0);
constexpr uint32_t kIdescGramHalf = tc::idesc_bf16_f32(kGM, kGN / 2, 0, 0);
constexpr size_t kGramSmem = 1024 + (size_t)kGStages * kGStageBytes + 256;

struct GramParams {
    CUtensorMap tmA;   // {d_in, T, B}, box {64, 128, 1}, 128B swizzle
    CUtensorMap tmE;   // {d_out, T, B}
    int64_t T, d_in, d_out;
    int has_bias;
    int np, nq;        // 128-row blocks, 256-column blocks of the Gram
    int tiles_per_rec;
    int total_items;
    float* partial;    // [B][tiles_per_rec * 4]
    unsigned* status;
};

struct GramSmem {
    uint64_t full[kGStages];
    uint64_t empty[kGStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// tile index t of a record -> (p, q), enumerating p-major the tiles with p <= 2q + 1
__device__ __forceinline__ void gram_tile(int t, int np, int nq, int& p, int& q) {
    for (p = 0; p < np; ++p) {
        const int qmin = p >> 1;   // smallest q with 2q + 1 >= p
        const int cnt = nq - qmin;
        if (t < cnt) {
            q = qmin + t;
            return;
        }
        t -= cnt;
    }
    p = np - 1;
    q = nq - 1;
}

__global__ void __launch_bounds__(kGThreads, 1) k_ghost_gram_tc(const __grid_constant__ GramParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GramSmem* sh = reinterpret_cast<GramSmem*>(tiles + (size_t)kGStages * kGStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkA = (int)((p.d_in + kGK - 1) / kGK);
    const int nkE = (int)((p.d_out + kGK - 1) / kGK);
    volatile int* abort_flag = &sh->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            tc::mbar_init(&sh->full[s], 1);
            tc::mbar_init(&sh->empty[s], 1);
        }
        tc::mbar_init(&sh->acc_full, 1);
        tc::mbar_init(&sh->acc_empty, 128);
        tc::mbar_init(&sh->drain, 1);
        sh->abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&p.tmA);
        tc::tma_prefetch_desc(&p.tmE);
    }
    if (warp == 1) tc::tmem_alloc(&sh->tmem_base, 512);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    // the set-up above may overlap the previous kernel of the stream; A and E
    // are read only after it completed
    grid_dep_wait();
    grid_dep_trigger();

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            tc::StageRing<kGStages> ring;
            for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
                const int rec = item / p.tiles_per_rec;
                int pb, qb;
                gram_tile(item % p.tiles_per_rec, p.np, p.nq, pb, qb);
                // the left 128 columns of the tile lie below the diagonal when p = 2q + 1:
                // they are neither loaded nor multiplied.  On the diagonal the row block p
                // is one of the two halves of the column block q, so it is loaded once:
                // p = 2q uses the left half as A, p = 2q + 1 its own rows as the right half
                const bool left = pb <= 2 * qb;
                const bool diag = pb == 2 * qb;
                const uint32_t bytes = diag ? 2u * kGAStage : (left ? kGStageBytes : kGAStage);
                for (int kt = 0; kt < nkA + nkE; ++kt, ++it, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->empty[s], ring.ph ^ 1u, abort_flag, p.status)) goto gram_producer_done;
                    uint8_t* st = tiles + (size_t)s * kGStageBytes;
                    const CUtensorMap* tm = kt < nkA ? &p.tmA : &p.tmE;
                    const int k0 = (kt < nkA ? kt : kt - nkA) * kGK;
                    tc::mbar_arrive_expect_tx(&sh->full[s], bytes);
                    if (!diag) tc::tma_load_3d(st, tm, &sh->full[s], k0, pb * kGM, rec);
                    if (left) {
                        tc::tma_load_3d(st + kGAStage, tm, &sh->full[s], k0, qb * kGN, rec);
                        tc::tma_load_3d(st + kGAStage + kGAStage, tm, &sh->full[s], k0, qb * kGN + 128, rec);
                    }
                }
            }
        gram_producer_done:
            for (uint32_t j = it > kGStages ? it - kGStages : 0; j < it; ++j)
                tc::mbar_wait_drain(&sh->full[j % kGStages], (j / kGStages) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t lt = 0;
            tc::StageRing<kGStages> ring;
            const uint32_t tiles_u32 = tc::smem_u32(tiles);
            for (int item = blockIdx.x; item < p.total_items; item += gridDim.x, ++lt) {
                int pb, qb;
                gram_tile(item % p.tiles_per_rec, p.np, p.nq, pb, qb);
                const bool left = pb <= 2 * qb;
                const bool diag = pb == 2 * qb;
                // full tile: N = 256 from the first B row; right half only: N = 128, its B rows
                // being the A rows; on the diagonal A is the B block's left half
                const uint32_t idesc = left ? kIdescGram : kIdescGramHalf;
                const uint32_t aoff = diag ? (uint32_t)kGAStage : 0u;
                const uint32_t boff = left ? (uint32_t)kGAStage : 0u;
                const uint32_t coff = left ? 0u : 128u;
                if (!tc::mbar_wait(&sh->acc_empty, (lt & 1u) ^ 1u, abort_flag, p.status)) break;
                tc::tc_fence_after();
                bool ok = true;
                for (int kt = 0; kt < nkA + nkE; ++kt, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->full[s], ring.ph, abort_flag, p.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t sa = tiles_u32 + s * (uint32_t)kGStageBytes;
                    const bool phaseA = kt < nkA;
                    const uint32_t d_tmem = tmem + (phaseA ? 0u : 256u) + coff;
                    const int kl = phaseA ? kt : kt - nkA;
                    // K-major, 128B swizzle: 16 features = 32 bytes inside the swizzle row
                    const uint64_t ad = tc::smem_desc(sa + aoff, 16, 1024, tc::SW_128B);
                    const uint64_t bd = tc::smem_desc(sa + boff, 16, 1024, tc::SW_128B);
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk)
                        tc::mma_bf16(d_tmem, tc::desc_advance(ad, kk * 32), tc::desc_advance(bd, kk * 32), idesc,
                                     (kl | kk) != 0);
                    tc::mma_commit(&sh->empty[s]);
                }
                if (!ok) break;
                tc::mma_commit(&sh->acc_full);
            }
        }
    } else {
        const int quarter = warp & 3;
        const int ew = warp - 2;
        uint32_t lt = 0;
        for (int item = blockIdx.x; item < p.total_items; item += gridDim.x, ++lt) {
            const int rec = item / p.tiles_per_rec;
            const int tl = item % p.tiles_per_rec;
            int pb, qb;
            gram_tile(tl, p.np, p.nq, pb, qb);
            if (!tc::mbar_wait_warp(&sh->acc_full, lt & 1u, abort_flag, p.status)) break;
            tc::tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16);
            const float bias = p.has_bias ? 1.f : 0.f;
            float acc = 0.f;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const int bcol = 2 * qb + half;   // 128-column block of this half
                const float w = pb < bcol ? 2.f : (pb == bcol ? 1.f : 0.f);
                if (w == 0.f) continue;          // uniform across the CTA
                float part = 0.f;
#pragma unroll 1
                for (int g = 0; g < 2; ++g) {
                    // 64 columns of GA and of GE, four loads and one wait each
                    float ga[4][16], ge[4][16];
                    const uint32_t col = half * 128 + g * 64;
                    tc::tmem_ld16x4(tb + col, ga);
                    tc::tmem_ld16x4(tb + 256 + col, ge);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int j = 0; j < 16; ++j) part = fmaf(ga[c][j] + bias, ge[c][j], part);
                }
                acc = fmaf(w, part, acc);
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sh->acc_empty);
            acc = warp_sum(acc);
            if (lane == 0) p.partial[(int64_t)rec * (p.tiles_per_rec * 4) + tl * 4 + ew] = acc;
        }
    }

    if (warp == 1 && lane == 0) {
        tc::mma_commit(&sh->drain);
        tc::mbar_wait_drain(&sh->drain, 0);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

bool encode_bf16(CUtensorMap* m, const void* base, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box) {
    const EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t gd[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t gs[2] = {strides[0], strides[1]};
    cuuint32_t bd[3] = {box[0], box[1], box[2]};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gd, gs, bd, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gram_tiles_per_rec(int64_t T) {
    const int np = (int)((T + kGM - 1) / kGM), nq = (int)((T + kGN - 1) / kGN);
    int n = 0;
    for (int pb = 0; pb < np; ++pb) n += nq - (pb >> 1);
    return n;
}

}  // namespace

bool tc_encode_gram(const NormTask& t, int64_t B, CUtensorMap* maps2) {
    const uint32_t box[3] = {64, (uint32_t)kGM, 1};
    const uint64_t da[3] = {(uint64_t)t.d_in, (uint64_t)t.T, (uint64_t)B};
    const uint64_t sa[2] = {(uint64_t)t.d_in * 2, (uint64_t)(t.d_in * t.T * 2)};
    const uint64_t de[3] = {(uint64_t)t.d_out, (uint64_t)t.T, (uint64_t)B};
    const uint64_t se[2] = {(uint64_t)t.d_out * 2, (uint64_t)(t.d_out * t.T * 2)};
    return encode_bf16(&maps2[0], t.A, da, sa, box) && encode_bf16(&maps2[1], t.E, de, se, box);
}

bool tc_gram_supported(int dtype, int64_t T, int64_t d_in, int64_t d_out) {
    return dtype == DT_BF16 && T > 1 && d_in % 8 == 0 && d_out % 8 == 0 && d_in >= 64 && d_out >= 64;
}

int nslots_gram(int64_t T) { return gram_tiles_per_rec(T) * 4; }

cudaError_t launch_ghost_gram_tc(const NormTask& t, int64_t B, unsigned* status, cudaStream_t s) {
    {
        const cudaError_t a = ensure_smem_limit(reinterpret_cast<const void*>(k_ghost_gram_tc), (int)kGramSmem);
        if (a != cudaSuccess) return a;
    }
    GramParams p;
    if (t.maps) {
        p.tmA = t.maps[0];
        p.tmE = t.maps[1];
    } else {
        CUtensorMap m[2];
        if (!tc_encode_gram(t, B, m)) return cudaErrorInvalidValue;
        p.tmA = m[0];
        p.tmE = m[1];
    }
    p.T = t.T;
    p.d_in = t.d_in;
    p.d_out = t.d_out;
    p.has_bias = t.has_bias;
    p.np = (int)((t.T + kGM - 1) / kGM);
    p.nq = (int)((t.T + kGN - 1) / kGN);
    p.tiles_per_rec = gram_tiles_per_rec(t.T);
    p.total_items = (int)(B * p.tiles_per_rec);
    p.partial = t.partial;
    p.status = status;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = p.total_items < sms ? p.total_items : sms;
    const cudaError_t e = launch_dependent(k_ghost_gram_tc, dim3(grid), dim3(kGThreads), kGramSmem, s, p);
    count_launch(KL_GHOST_GRAM_TC);
    return e;
}
