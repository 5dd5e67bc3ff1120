// Record-owned LLM.int8 forward of a frozen layer ("Sensitivity Inflation
// from Cross-Record Precision Routing in Private Quantized Fine-Tuning",
// section 4.2, Eq. 6 and Algorithm 1; Appendix A):
//
//   O_r  = { j : |A_ij| >= tau for some row i of record r }   (segmented)
//   U    = union of the O_r                                    (batched routing)
//   s_i  = max over j with |A_ij| < tau of |A_ij|              (row-local scale)
//   Q_ij = rint((127 A_ij) / s_i) if j not in O, else 0        (O = O_r of the row, or U)
//   Y    = half( ((float(Q Wq^T) * s_i) * sW_n) / 16129 + sum_{j in O} A_ij What_nj )
//
// so that a row's output depends only on its own record's data (record
// isolation, Proposition 2) in record-owned mode, and on the whole batch in
// the batched mode LLM.int8 ships with.  The correction runs over the set's
// columns in ascending order, one fused multiply-add each.
//
// The integer product Q Wq^T is exact.  On GB300 the int8 tensor rate is a
// small fraction of the bf16 one (cuBLAS: 155 against 1904 dense TOPS on an
// 8192^3 product), so the product runs on the bf16 tensor cores instead:
// int8 codes are exact in bf16, their products (at most 127^2 = 16129) are
// exact in the fp32 accumulator, and so is every partial sum of at most 1024
// products (below 2^24).  K is cut into chunks of 1024 accumulated in their
// own TMEM columns; the epilogue adds the chunks in int32.  Layers with K
// above 4096 take a dp4a kernel on the CUDA cores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dp_clip.h"
#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "tc_common.cuh"

namespace {

constexpr int kTM = 64, kTN = 64, kTK = 64;

__global__ void k_int8_quantize_weight(const __half* __restrict__ W, int64_t N, int64_t K, int8_t* __restrict__ Wq,
                                       float* __restrict__ sW, __half* __restrict__ What) {
    const int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= N) return;
    const __half* w = W + n * K;
    float m = 0.f;
    for (int64_t j = lane; j < K; j += 32) m = fmaxf(m, fabsf(__half2float(w[j])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    for (int64_t j = lane; j < K; j += 32) {
        // the dequantized weight comes from the integer code (a code of 0 is +0)
        const int q = m > 0.f ? (int)rintf((127.0f * __half2float(w[j])) / m) : 0;
        Wq[n * K + j] = (int8_t)q;
        What[n * K + j] = __float2half_rn(((float)q * m) / 127.0f);
    }
    if (lane == 0) sW[n] = m;
}

// One warp per row i: the row's outlier bits (|a| >= tau) per 32-column word,
// ORed into its record's set and into the union (only nonzero words: the
// sets and the union start at zero), and its scale s_i = max |a| over the
// entries below tau.  Lane l reads 8-column groups l, l + 32, ...; the four
// lanes of a word combine their bits by shuffles.
__global__ void k_int8_rowscan(const __half* __restrict__ A, int64_t n, int64_t K, int64_t rows, int64_t words,
                               float tau, uint32_t* __restrict__ sets, uint32_t* __restrict__ uni,
                               float* __restrict__ scales, unsigned* __restrict__ status, int vec) {
    const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (status && i == 0 && lane == 0) *status = 0u;   // the tensor-core product's wait status
    if (i >= n) return;
    const __half* a = A + i * K;
    uint32_t* set = sets + (i / rows) * words;
    const int64_t groups = (K + 7) / 8;
    float m = 0.f;
    for (int64_t g0 = 0; g0 < groups; g0 += 32) {
        const int64_t g = g0 + lane;
        uint32_t bits = 0u;
        if (g < groups) {
            float v[8];
            if (vec) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4*>(a + g * 8));
                const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __half22float2(h[q]);
                    v[2 * q] = f.x;
                    v[2 * q + 1] = f.y;
                }
            } else {
#pragma unroll
                for (int b = 0; b < 8; ++b) v[b] = g * 8 + b < K ? __half2float(a[g * 8 + b]) : 0.f;
            }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const float x = fabsf(v[b]);
                if (x >= tau) bits |= 1u << b;
                else m = fmaxf(m, x);
            }
        }
        // the group's 8 bits at their place in the 32-column word, ORed over the word's 4 lanes
        bits <<= 8 * (lane & 3);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
        const int64_t w = g / 4;
        if ((lane & 3) == 0 && bits && w < words) {
            atomicOr(set + w, bits);
            atomicOr(uni + w, bits);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) scales[i] = m;
}

struct Int8Args {
    const __half* A;
    int64_t n, K, rows, words;
    const int8_t* Wq;
    const float* sW;
    const __half* What;
    int64_t N;
    int record_owned;
    const uint32_t* sets;
    const uint32_t* uni;
    const float* s;
    __half* Y;
};

__device__ __forceinline__ const uint32_t* row_set(const Int8Args& p, int64_t i) {
    return p.record_owned ? p.sets + (i / p.rows) * p.words : p.uni;
}

// 64 x 64 output tile per block of 256 threads, 4 x 4 outputs per thread;
// A is quantized while it is staged in shared memory
__global__ void __launch_bounds__(256) k_int8_gemm(const Int8Args p) {
    __shared__ int32_t Qs[kTM][kTK / 4 + 1];
    __shared__ int32_t Ws[kTN][kTK / 4 + 1];
    const int tid = threadIdx.x;
    const int64_t i0 = (int64_t)blockIdx.y * kTM, n0 = (int64_t)blockIdx.x * kTN;
    const int tr = tid / 16, tc = tid % 16;    // rows i0 + 4 tr .. , outputs n0 + 4 tc ..
    int32_t acc[4][4] = {};
    for (int64_t k0 = 0; k0 < p.K; k0 += kTK) {
        // stage: thread t packs 4 consecutive K entries of one A row and of one W row, 4 times
        for (int e = tid; e < kTM * (kTK / 4); e += 256) {
            const int r = e / (kTK / 4), k4 = e % (kTK / 4);
            const int64_t i = i0 + r;
            uint32_t packed = 0u, wpacked = 0u;
            if (i < p.n) {
                const uint32_t* set = row_set(p, i);
                const float s = p.s[i];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int64_t j = k0 + 4 * k4 + b;
                    int q = 0;
                    if (j < p.K && s > 0.f && !((set[j >> 5] >> (j & 31)) & 1u))
                        q = (int)rintf((127.0f * __half2float(p.A[i * p.K + j])) / s);
                    packed |= (uint32_t)(q & 0xff) << (8 * b);
                }
            }
            Qs[r][k4] = (int32_t)packed;
            const int64_t nn = n0 + r;
            if (nn < p.N) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int64_t j = k0 + 4 * k4 + b;
                    const int w = j < p.K ? (int)p.Wq[nn * p.K + j] : 0;
                    wpacked |= (uint32_t)(w & 0xff) << (8 * b);
                }
            }
            Ws[r][k4] = (int32_t)wpacked;
        }
        __syncthreads();
#pragma unroll 4
        for (int k4 = 0; k4 < kTK / 4; ++k4) {
            int32_t qa[4], wb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                qa[u] = Qs[4 * tr + u][k4];
                wb[u] = Ws[4 * tc + u][k4];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = __dp4a(qa[u], wb[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + 4 * tr + u;
        if (i >= p.n) continue;
        const float s = p.s[i];
        const uint32_t* set = row_set(p, i);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int64_t nn = n0 + 4 * tc + v;
            if (nn >= p.N) continue;
            const float deq = (((float)acc[u][v] * s) * p.sW[nn]) / 16129.0f;
            float corr = 0.f;
            for (int64_t w = 0; w < p.words; ++w) {
                uint32_t bits = set[w];
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1u;
                    const int64_t j = w * 32 + b;
                    corr = fmaf(__half2float(p.A[i * p.K + j]), __half2float(p.What[nn * p.K + j]), corr);
                }
            }
            p.Y[i * p.N + nn] = __float2half_rn(deq + corr);
        }
    }
}

// ------------------------------------------------ tensor-core integer product
// Workspace of one forward call (every region 256-byte aligned): the outlier
// sets, the row scales, the sets as ascending column lists, a status word,
// and the bf16 codes of A and of the weights, rows padded to Kp = K rounded
// up to 8 (16-byte rows for TMA).
struct Int8Workspace {
    int64_t sets, scales, lists, status, qa, qw, total, Kp;
    static int64_t pad(int64_t b) { return (b + 255) / 256 * 256; }
    static Int8Workspace layout(int64_t n, int64_t K, int64_t N, int64_t records) {
        Int8Workspace w;
        const int64_t words = (K + 31) / 32;
        w.Kp = (K + 7) / 8 * 8;
        w.sets = 0;
        w.scales = w.sets + pad((records + 1) * words * 4);
        w.lists = w.scales + pad(n * 4);
        w.status = w.lists + pad((records + 1) * (K + 1) * 4);
        w.qa = w.status + 256;
        w.qw = w.qa + pad(n * w.Kp * 2);
        w.total = w.qw + pad(N * w.Kp * 2);
        return w;
    }
};

constexpr int kQChunk = 1024;                  // products per exact fp32 partial sum
constexpr int kQM = 128, kQK = 64, kQStages = 4;
constexpr int kQEpiWarps = 16;
constexpr int kQPre = 2;                       // set columns whose half weights are loaded ahead (one per half-warp)
static_assert(kQPre == 2, "the epilogue hands the preloaded half weights around as two half-warps");
constexpr int kQThreads = 32 * (2 + kQEpiWarps);
constexpr int kQAStage = kQM * kQK * 2;        // 16 KB: 128 rows x 64 codes, 128-byte swizzle
constexpr int kQBStageMax = 256 * kQK * 2;     // 32 KB: up to 256 weight rows
constexpr int kQStageBytes = kQAStage + kQBStageMax;
constexpr size_t kQSmem = 1024 + (size_t)kQStages * kQStageBytes + 256;

// One warp per set (the records' sets, then the union): its columns in
// ascending order, lists[t][0] = count, lists[t][1 ..] = columns.
__device__ void set_list(const uint32_t* __restrict__ sets, int64_t words, int64_t K, int64_t t,
                         int* __restrict__ lists) {
    const int lane = threadIdx.x & 31;
    const uint32_t* bits = sets + t * words;
    int* out = lists + t * (K + 1);
    int cnt = 0;
    for (int64_t w = 0; w < words; ++w) {
        const uint32_t word = bits[w];                 // the same word for every lane
        const bool mine = (word >> lane) & 1u;
        const uint32_t below = word & ((1u << lane) - 1u);
        if (mine) out[1 + cnt + __popc(below)] = (int)(w * 32 + lane);
        cnt += __popc(word);
    }
    if (lane == 0) out[0] = cnt;
}

// The first list_blocks blocks write the sets' column lists (a warp per
// set); the others the bf16 codes, one thread per 8 columns of a row: rows
// 0 .. n-1 of A as Q_ij (0 in the row's outlier columns or when s_i = 0),
// then the rows of the weights' int8 codes; columns K .. Kp-1 zero.  Each
// thread writes 16 bytes.
__global__ void k_int8_codes(const __half* __restrict__ A, int64_t n, int64_t K, int64_t Kp, int64_t rows,
                             int64_t words, int record_owned, const uint32_t* __restrict__ sets,
                             const uint32_t* __restrict__ uni, const float* __restrict__ scales,
                             const int8_t* __restrict__ Wq, int64_t N, __nv_bfloat16* __restrict__ qa,
                             __nv_bfloat16* __restrict__ qw, int64_t nsets, int* __restrict__ lists,
                             int list_blocks, int vec) {
    if ((int)blockIdx.x < list_blocks) {
        const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
        if (t < nsets) set_list(sets, words, K, t, lists);
        return;
    }
    const int64_t gpr = Kp / 8;                        // groups per row
    const int64_t total = (n + N) * gpr;
    const int64_t nthreads = (int64_t)(gridDim.x - list_blocks) * blockDim.x;
    for (int64_t t = (int64_t)(blockIdx.x - list_blocks) * blockDim.x + threadIdx.x; t < total; t += nthreads) {
        const int64_t r = t / gpr, j0 = (t - r * gpr) * 8;
        __align__(16) __nv_bfloat16 out[8];
        if (r < n) {
            const uint32_t* set = record_owned ? sets + (r / rows) * words : uni;
            const float s = __ldg(scales + r);
            const uint32_t word = j0 < K ? __ldg(set + (j0 >> 5)) : 0u;
            // the group's eight entries, one 16-byte load when the rows are whole aligned vectors
            __align__(16) __half a8[8];
            if (vec) {
                *reinterpret_cast<uint4*>(a8) = __ldg(reinterpret_cast<const uint4*>(A + r * K + j0));
            } else {
#pragma unroll
                for (int b = 0; b < 8; ++b) a8[b] = j0 + b < K ? A[r * K + j0 + b] : __float2half(0.f);
            }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int64_t j = j0 + b;
                int q = 0;
                if (j < K && s > 0.f && !((word >> (j & 31)) & 1u))
                    q = (int)rintf((127.0f * __half2float(a8[b])) / s);
                out[b] = __float2bfloat16_rn((float)q);
            }
            *reinterpret_cast<uint4*>(qa + r * Kp + j0) = *reinterpret_cast<const uint4*>(out);
        } else {
            const int64_t nn = r - n;
#pragma unroll
            for (int b = 0; b < 8; ++b) out[b] = __float2bfloat16_rn(j0 + b < K ? (float)Wq[nn * K + j0 + b] : 0.f);
            *reinterpret_cast<uint4*>(qw + nn * Kp + j0) = *reinterpret_cast<const uint4*>(out);
        }
    }
}

struct QGemmParams {
    CUtensorMap tmA;     // codes of A: {K, n}, row pitch Kp, box {64, 128}, 128-byte swizzle
    CUtensorMap tmW;     // codes of W: {K, N}, row pitch Kp, box {64, NT}
    int64_t n, N, K;
    int NT;              // output columns per tile (256 or 128)
    int nch;             // K chunks of kQChunk, each in its own TMEM columns
    int nk;              // 64-wide K tiles
    int m_tiles, n_tiles;
    int64_t rows, records;
    int record_owned;
    const __half* A;
    const __half* What;
    const float* s;
    const float* sW;
    const int* lists;
    __half* Y;
    int y_vec;           // Y rows start on 16-byte boundaries (N % 8 == 0)
    unsigned* status;
};

struct QSmem {
    uint64_t full[kQStages];
    uint64_t empty[kQStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Y = half(dequant(Q Wq^T) + correction) for 128 x NT output tiles, strided
// over the CTAs.  Warp 0: TMA producer; warp 1: TMEM owner and MMA issuer
// (tcgen05.mma kind::f16, bf16 x bf16 -> fp32, M = 128, N = NT, both operands
// K-major); warps 2-17: epilogue, a thread per output row and column quarter.
__global__ void __launch_bounds__(kQThreads, 1) k_int8_gemm_tc(const __grid_constant__ QGemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    QSmem* sh = reinterpret_cast<QSmem*>(tiles + (size_t)kQStages * kQStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = p.m_tiles * p.n_tiles;
    const int bstage = p.NT * kQK * 2;
    volatile int* abort_flag = &sh->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            tc::mbar_init(&sh->full[s], 1);
            tc::mbar_init(&sh->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sh->acc_full[b], 1);
            tc::mbar_init(&sh->acc_empty[b], 32 * kQEpiWarps);
        }
        tc::mbar_init(&sh->drain, 1);
        sh->abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&p.tmA);
        tc::tma_prefetch_desc(&p.tmW);
    }
    if (warp == 1) tc::tmem_alloc(&sh->tmem_base, 512);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    // two accumulators (the next tile's MMAs run during this tile's epilogue)
    // when a tile's chunks fit in half of the 512 TMEM columns
    const uint32_t nbuf = p.nch * p.NT <= 256 ? 2u : 1u;
    // the codes come from the kernel before this one on the stream
    dpk::grid_dep_wait();
    dpk::grid_dep_trigger();

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            tc::StageRing<kQStages> ring;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                const int mb = tile / p.n_tiles, nb = tile % p.n_tiles;
                for (int kt = 0; kt < p.nk; ++kt, ++it, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->empty[s], ring.ph ^ 1u, abort_flag, p.status)) goto q_producer_done;
                    uint8_t* st = tiles + (size_t)s * kQStageBytes;
                    tc::mbar_arrive_expect_tx(&sh->full[s], (uint32_t)(kQAStage + bstage));
                    tc::tma_load_2d(st, &p.tmA, &sh->full[s], kt * kQK, mb * kQM);
                    tc::tma_load_2d(st + kQAStage, &p.tmW, &sh->full[s], kt * kQK, nb * p.NT);
                }
            }
        q_producer_done:
            for (uint32_t j = it > kQStages ? it - kQStages : 0; j < it; ++j)
                tc::mbar_wait_drain(&sh->full[j % kQStages], (j / kQStages) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16_f32(kQM, p.NT, 0, 0);
            const uint32_t tiles_u32 = tc::smem_u32(tiles);
            const int kt_per_chunk = kQChunk / kQK;
            uint32_t lt = 0;
            tc::StageRing<kQStages> ring;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
                const uint32_t b = lt % nbuf, use = lt / nbuf;
                if (!tc::mbar_wait(&sh->acc_empty[b], (use & 1u) ^ 1u, abort_flag, p.status)) break;
                tc::tc_fence_after();
                bool ok = true;
                for (int kt = 0; kt < p.nk; ++kt, ring.next()) {
                    const uint32_t s = ring.s;
                    if (!tc::mbar_wait(&sh->full[s], ring.ph, abort_flag, p.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const int ch = kt / kt_per_chunk, kl = kt - ch * kt_per_chunk;
                    const uint32_t d_tmem = tmem + b * 256u + (uint32_t)(ch * p.NT);
                    const uint32_t sa = tiles_u32 + s * (uint32_t)kQStageBytes;
                    const uint64_t ad = tc::smem_desc(sa, 16, 1024, tc::SW_128B);
                    const uint64_t bd = tc::smem_desc(sa + kQAStage, 16, 1024, tc::SW_128B);
#pragma unroll
                    for (int kk = 0; kk < kQK / 16; ++kk)
                        tc::mma_bf16(d_tmem, tc::desc_advance(ad, kk * 32), tc::desc_advance(bd, kk * 32), idesc,
                                     (kl | kk) != 0);
                    tc::mma_commit(&sh->empty[s]);
                }
                if (!ok) break;
                tc::mma_commit(&sh->acc_full[b]);
            }
        }
    } else {
        // four warps per TMEM lane quarter, each taking a quarter of the tile's
        // columns, 16 at a time (the divisions of the dequantization are many
        // dependent instructions: sixteen warps keep the schedulers busy).
        // Everything the epilogue reads from global memory -- the row's scale,
        // its set's first kQPre columns and their A entries, the weights'
        // scales and (when the warp's rows share one set) the half weights of
        // those set columns in the warp's columns -- is loaded while the tensor
        // cores work, one value per lane, and handed around by shuffles.
        const int quarter = warp & 3;
        const int part = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const int cols = p.NT / 4;
        const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t lt = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
            const int mb = tile / p.n_tiles, nb = tile % p.n_tiles;
            const int64_t i = (int64_t)mb * kQM + row;
            const bool valid = i < p.n;
            const float si = valid ? p.s[i] : 0.f;
            const int64_t set = p.record_owned ? (valid ? i / p.rows : 0) : p.records;
            const int* list = p.lists + set * (p.K + 1);
            const int cnt = valid ? list[0] : 0;
            int jj[kQPre];
            float av[kQPre];
#pragma unroll
            for (int u = 0; u < kQPre; ++u) {
                jj[u] = u < cnt ? list[1 + u] : 0;   // column 0 stands in for an absent entry
                av[u] = u < cnt ? __half2float(p.A[i * p.K + jj[u]]) : 0.f;
            }
            const int64_t cbase = (int64_t)nb * p.NT + part * cols;   // the warp's first column
            const float swv0 = cbase + lane < p.N ? __ldg(p.sW + cbase + lane) : 0.f;
            const float swv1 = cols > 32 && cbase + 32 + lane < p.N ? __ldg(p.sW + cbase + 32 + lane) : 0.f;
            // the rows of a warp usually belong to one record (or all take the union):
            // then lane l holds, for each 16-column group g, the half weight of column
            // 16 g + (l mod 16) and set column l / 16
            // (every lane takes part in each shuffle: none sits behind a short-circuit)
            const int cnt_l0 = __shfl_sync(0xffffffffu, cnt, 0);
            const int jj0_l0 = __shfl_sync(0xffffffffu, jj[0], 0);
            const int jj1_l0 = __shfl_sync(0xffffffffu, jj[1], 0);
            const bool shared_set = __all_sync(0xffffffffu, cnt == cnt_l0 && jj[0] == jj0_l0 && jj[1] == jj1_l0);
            float wpre[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int64_t nn = cbase + 16 * g + (lane & 15);
                const int u = lane >> 4;
                wpre[g] = shared_set && u < cnt && 16 * g < cols && nn < p.N
                              ? __half2float(p.What[nn * p.K + (u ? jj[1] : jj[0])])
                              : 0.f;
            }
            const uint32_t b = lt % nbuf, use = lt / nbuf;
            if (!tc::mbar_wait_warp(&sh->acc_full[b], use & 1u, abort_flag, p.status)) break;
            tc::tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < cols; c0 += 16) {
                // every partial sum is an integer below 2^24, exact in fp32
                int acc[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = 0;
                for (int ch = 0; ch < p.nch; ++ch) {
                    float v[16];
                    tc::tmem_ld16(tq + b * 256u + (uint32_t)(ch * p.NT + part * cols + c0), v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] += __float2int_rz(v[j]);
                }
                const int64_t n0 = cbase + c0;
                if (n0 < p.N) {   // uniform across the warp; rows past n have an empty set
                    // the correction over the row's set in ascending column order: the
                    // first kQPre columns' weights loaded together, the rest one by one
                    float corr[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) corr[j] = 0.f;
                    if (shared_set) {
                        const int g = c0 >> 4;
                        const float wg = g == 0 ? wpre[0] : (g == 1 ? wpre[1] : (g == 2 ? wpre[2] : wpre[3]));
#pragma unroll
                        for (int u = 0; u < kQPre; ++u) {
                            if (u < cnt) {
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    corr[j] = fmaf(av[u], __shfl_sync(0xffffffffu, wg, 16 * u + j), corr[j]);
                            }
                        }
                    }
                    for (int c = shared_set ? kQPre : 0; c < cnt; ++c) {
                        const int jc = list[1 + c];
                        const float a = __half2float(p.A[i * p.K + jc]);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (n0 + j < p.N) corr[j] = fmaf(a, __half2float(p.What[(n0 + j) * p.K + jc]), corr[j]);
                    }
                    __align__(16) __half y[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        // the weight's scale of column n0 + j, from the lane that loaded it
                        const int cc = c0 + j;
                        const float sw = __shfl_sync(0xffffffffu, (cc & 32) ? swv1 : swv0, cc & 31);
                        const float deq = (((float)acc[j] * si) * sw) / 16129.0f;
                        y[j] = __float2half_rn(deq + corr[j]);
                    }
                    if (valid) {
                        __half* dst = p.Y + i * p.N + n0;
                        if (p.y_vec && n0 + 16 <= p.N) {
                            reinterpret_cast<uint4*>(dst)[0] = reinterpret_cast<const uint4*>(y)[0];
                            reinterpret_cast<uint4*>(dst)[1] = reinterpret_cast<const uint4*>(y)[1];
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (n0 + j < p.N) dst[j] = y[j];
                        }
                    }
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sh->acc_empty[b]);
        }
        // a wait that gave up leaves this CTA's tiles undone: they read NaN
        if (*abort_flag) {
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                const int mb = tile / p.n_tiles, nb = tile % p.n_tiles;
                const int64_t i = (int64_t)mb * kQM + row;
                if (i >= p.n) continue;
                for (int c = part * cols; c < (part + 1) * cols; ++c) {
                    const int64_t nn = (int64_t)nb * p.NT + c;
                    if (nn < p.N) p.Y[i * p.N + nn] = __float2half_rn(__int_as_float(0x7fc00000));
                }
            }
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

bool encode_codes(CUtensorMap* m, const void* base, int64_t K, int64_t Kp, int64_t rows, uint32_t box_rows) {
    const EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t gd[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t gs[1] = {(cuuint64_t)(Kp * 2)};
    cuuint32_t bd[2] = {(cuuint32_t)kQK, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gd, gs, bd, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int64_t dp_int8_workspace_bytes(int64_t n, int64_t K, int64_t N, int64_t rows_per_record) {
    if (n < 1 || K < 1 || N < 1 || rows_per_record < 1 || n % rows_per_record) return -1;
    return Int8Workspace::layout(n, K, N, n / rows_per_record).total;
}

extern "C" dp_status dp_int8_quantize_weight(const void* W, int64_t N, int64_t K, int8_t* Wq, float* sW, void* What,
                                             void* stream) {
    NvtxRange nvtx_range("dp_int8_quantize_weight");
    if (!W || !Wq || !sW || !What) return DP_ERR_INVALID_ARG;
    if (N < 1 || K < 1) return DP_ERR_SHAPE;
    const int64_t blocks = (N + 7) / 8;
    k_int8_quantize_weight<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __half*>(W), N, K, Wq, sW, static_cast<__half*>(What));
    count_launch(KL_INT8_QUANTIZE_WEIGHT);
    return cudaGetLastError() == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}

extern "C" dp_status dp_int8_forward(const void* A, int64_t n, int64_t K, int64_t rows_per_record, const int8_t* Wq,
                                     const float* sW, const void* What, int64_t N, float tau, int record_owned,
                                     void* Y, void* workspace, void* stream) {
    NvtxRange nvtx_range("dp_int8_forward");
    if (!A || !Wq || !sW || !What || !Y || !workspace) return DP_ERR_INVALID_ARG;
    if (n < 1 || K < 1 || N < 1 || rows_per_record < 1 || n % rows_per_record) return DP_ERR_SHAPE;
    if (!(tau > 0.f)) return DP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return DP_ERR_INVALID_ARG;
    if (n >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= 133000) return DP_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t words = (K + 31) / 32;
    const int64_t records = n / rows_per_record;
    const Int8Workspace lay = Int8Workspace::layout(n, K, N, records);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint32_t* sets = reinterpret_cast<uint32_t*>(ws + lay.sets);
    uint32_t* uni = sets + records * words;
    float* scales = reinterpret_cast<float*>(ws + lay.scales);
    if (cudaMemsetAsync(sets, 0, (size_t)(records + 1) * words * 4, s) != cudaSuccess) return DP_ERR_CUDA;
    const bool tensor_cores = K <= 4 * kQChunk;
    unsigned* status = reinterpret_cast<unsigned*>(ws + lay.status);
    // rows of whole 16-byte vectors on 16-byte boundaries are read as such
    const int vec = (K % 8 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0) ? 1 : 0;
    k_int8_rowscan<<<(unsigned)((n + 7) / 8), 256, 0, s>>>(static_cast<const __half*>(A), n, K, rows_per_record, words,
                                                           tau, sets, uni, scales, tensor_cores ? status : nullptr,
                                                           vec);
    count_launch(KL_INT8_ROWSCAN);
    if (!tensor_cores) {
        // beyond four exact chunks per tile: the integer product on the CUDA cores
        Int8Args p;
        p.A = static_cast<const __half*>(A);
        p.n = n;
        p.K = K;
        p.rows = rows_per_record;
        p.words = words;
        p.Wq = Wq;
        p.sW = sW;
        p.What = static_cast<const __half*>(What);
        p.N = N;
        p.record_owned = record_owned ? 1 : 0;
        p.sets = sets;
        p.uni = uni;
        p.s = scales;
        p.Y = static_cast<__half*>(Y);
        k_int8_gemm<<<dim3((unsigned)((N + kTN - 1) / kTN), (unsigned)((n + kTM - 1) / kTM)), 256, 0, s>>>(p);
        count_launch(KL_INT8_GEMM);
        return cudaGetLastError() == cudaSuccess ? DP_OK : DP_ERR_CUDA;
    }
    int* lists = reinterpret_cast<int*>(ws + lay.lists);
    __nv_bfloat16* qa = reinterpret_cast<__nv_bfloat16*>(ws + lay.qa);
    __nv_bfloat16* qw = reinterpret_cast<__nv_bfloat16*>(ws + lay.qw);
    {
        const int64_t groups = (n + N) * (lay.Kp / 8);
        int64_t grid = (groups + 255) / 256;
        const int64_t cap = (int64_t)device_sm_count() * 16;
        if (grid > cap) grid = cap;
        const int64_t list_blocks = (records + 1 + 7) / 8;   // a warp per set, 8 warps per block
        k_int8_codes<<<(unsigned)(list_blocks + grid), 256, 0, s>>>(
            static_cast<const __half*>(A), n, K, lay.Kp, rows_per_record, words, record_owned ? 1 : 0, sets, uni,
            scales, Wq, N, qa, qw, records + 1, lists, (int)list_blocks, vec);
    }
    count_launch(KL_INT8_CODES);
    QGemmParams p;
    p.nch = (int)((K + kQChunk - 1) / kQChunk);
    p.NT = p.nch <= 2 ? 256 : 128;
    if (!encode_codes(&p.tmA, qa, K, lay.Kp, n, kQM) || !encode_codes(&p.tmW, qw, K, lay.Kp, N, (uint32_t)p.NT))
        return DP_ERR_CUDA;
    p.n = n;
    p.N = N;
    p.K = K;
    p.nk = (int)((K + kQK - 1) / kQK);
    p.m_tiles = (int)((n + kQM - 1) / kQM);
    p.n_tiles = (int)((N + p.NT - 1) / p.NT);
    p.rows = rows_per_record;
    p.records = records;
    p.record_owned = record_owned ? 1 : 0;
    p.A = static_cast<const __half*>(A);
    p.What = static_cast<const __half*>(What);
    p.s = scales;
    p.sW = sW;
    p.lists = lists;
    p.Y = static_cast<__half*>(Y);
    p.y_vec = (N % 8 == 0 && (reinterpret_cast<uintptr_t>(Y) & 15u) == 0) ? 1 : 0;
    p.status = status;
    {
        const cudaError_t a = ensure_smem_limit(reinterpret_cast<const void*>(k_int8_gemm_tc), (int)kQSmem);
        if (a != cudaSuccess) return DP_ERR_CUDA;
    }
    const int64_t ntiles = (int64_t)p.m_tiles * p.n_tiles;
    const int sms = device_sm_count();
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    const cudaError_t e = launch_dependent(k_int8_gemm_tc, dim3(grid), dim3(kQThreads), kQSmem, s, p);
    count_launch(KL_INT8_GEMM_TC);
    return e == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}
