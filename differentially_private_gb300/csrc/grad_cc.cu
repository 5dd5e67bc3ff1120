// Clip factors (with the pre-scaled operand copies of single-record
// tensor-core sums), the reweighted clipped sum with its noise epilogue on the
// CUDA cores, the weighted sum of stored per-example gradients, and the
// standalone noise generator.
//
//   n2_i = sum over layers (registration order) of the layer's partials
//   c_i  = 1 if sqrt(n2_i) <= C, else C / sqrt(n2_i) rounded toward zero
//   G    = (sum_i c_i g_i + sigma C z) / L
// ("Privacy-Preserving Machine Learning", section "Differentially private
// stochastic gradient descent", phases 3-5; "Differential Privacy in
// Fine-Tuning (DP-SGD)", "Per-Sample Gradient Clipping" and "Calibrated
// Gaussian Noise Addition"; "Sensitivity Inflation from Cross-Record
// Precision Routing in Private Quantized Fine-Tuning", Eq. 2 and Eq. 3.)
#include "common.cuh"
#include "launch.cuh"

using namespace dpk;

namespace {

// --------------------------------------------------------------- clipping
// The partial slots of a record, all layers in registration order, form one
// flat index space of total_slots entries; slot j of record i lives at
// slots[j].base[i * slots[j].stride] (a table the host builds once per layer
// set).  A group of G threads serves one record: thread t sums slots t,
// t + G, t + 2G, ... in ascending order, kClipLoads loads in flight at a
// time, then a fixed-order butterfly (G = 32, a warp per record) or block
// reduction (G = blockDim) combines the threads.  G depends on total_slots
// only, never on B, so a record's norm does not depend on the batch.
constexpr int kClipLoads = 8;
constexpr int kScalePre = 8;          // pre-scale units a thread fetches before the dependency wait
constexpr int kClipMaxThreads = 512;
constexpr int kClipWarpBlock = 256;   // warp-per-record mode: 8 records per block

// G = smallest power of two with G * kClipLoads >= total_slots, at least a
// warp and at most kClipMaxThreads; it depends on the shapes only
int clip_group(int64_t total_slots) {
    int G = 32;
    while (G < kClipMaxThreads && (int64_t)G * kClipLoads < total_slots) G *= 2;
    return G;
}

// c * (8 bf16), rounded to bf16 (the pre-scaled operand of the tensor-core sum)
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float c) {
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w[i]);
        const float2 f = __bfloat1622float2(h);
        h = __floats2bfloat162_rn(f.x * c, f.y * c);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return v;
}

// Unit x (16 bytes) of record rec's rows over the pre-scale jobs, jobs in order.
__device__ __forceinline__ bool scale_unit(const ClipParams& p, int64_t x, int64_t rec, const uint4** src,
                                           uint4** dst) {
    for (int j = 0; j < p.nscale; ++j) {
        const int64_t n = p.scale[j].units;
        if (x < n) {
            *src = p.scale[j].src + rec * n + x;
            *dst = p.scale[j].dst + rec * n + x;
            return true;
        }
        x -= n;
    }
    return false;
}

// Besides n2 and c, the record's group of G threads writes the pre-scaled
// copies c_i * X_i of the operands of the layers whose tensor-core sum runs
// as one record (p.scale): those operands were written before the norm
// kernels ran, so each thread fetches its first units of them before the
// dependency wait and scales them as soon as c_i is known.
template <bool kWarpPerRecord>
__global__ void __launch_bounds__(kClipMaxThreads) k_clip(const ClipParams p, float* __restrict__ n2_out,
                                                          float* __restrict__ c_out, float* __restrict__ n2_user,
                                                          float* __restrict__ c_user, unsigned* __restrict__ status) {
    __shared__ float red[32];
    const int64_t rec = kWarpPerRecord ? (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)
                                       : (int64_t)blockIdx.x;
    const int t = kWarpPerRecord ? (int)(threadIdx.x & 31) : (int)threadIdx.x;
    const int G = kWarpPerRecord ? 32 : (int)blockDim.x;
    int64_t units = 0;
    for (int j = 0; j < p.nscale; ++j) units += p.scale[j].units;
    uint4 pre[kScalePre];
#pragma unroll
    for (int k = 0; k < kScalePre; ++k) {
        const uint4* src;
        uint4* dst;
        if (rec < p.B && scale_unit(p, t + (int64_t)k * G, rec, &src, &dst)) pre[k] = __ldcs(src);
    }
    // the slot table of the first round: written by the host before an earlier
    // step when p.slots_ready, so it is read before the dependency wait
    SlotRef ref0[kClipLoads];
    if (p.slots_ready && rec < p.B) {
#pragma unroll
        for (int u = 0; u < kClipLoads; ++u) {
            const int64_t j = t + (int64_t)u * G;
            if (j < p.total_slots) ref0[u] = p.slots[j];
        }
    }
    grid_dep_wait();
    grid_dep_trigger();
    if (p.status_next && blockIdx.x == 0 && threadIdx.x == 0) *p.status_next = 0u;
    float s = 0.f;
    if (rec < p.B) {   // uniform per warp in warp mode; always true in block mode
        for (int64_t j0 = t; j0 < p.total_slots; j0 += (int64_t)G * kClipLoads) {
            float v[kClipLoads];
#pragma unroll
            for (int u = 0; u < kClipLoads; ++u) {
                const int64_t j = j0 + (int64_t)u * G;
                v[u] = 0.f;
                if (j < p.total_slots) {
                    const SlotRef r = p.slots_ready && j0 == t ? ref0[u] : p.slots[j];
                    v[u] = __ldcg(r.base + rec * r.stride);
                }
            }
#pragma unroll
            for (int u = 0; u < kClipLoads; ++u) s += v[u];
        }
    }
    if (kWarpPerRecord) {
        if (rec >= p.B) return;
        s = warp_sum(s);
    } else {
        s = block_sum(s, red);
    }
    // every thread of the group holds the same s, so the same c
    const bool finite = isfinite(s);
    // C / n rounded toward zero keeps c * n <= C in float arithmetic
    const float c = !finite ? 0.f : (sqrtf(s) <= p.C ? 1.0f : __fdiv_rz(p.C, sqrtf(s)));
    if (t == 0) {
        if (!finite) atomicOr(status, 1u);
        n2_out[rec] = s;
        c_out[rec] = c;
        if (n2_user) n2_user[rec] = s;
        if (c_user) c_user[rec] = c;
    }
#pragma unroll
    for (int k = 0; k < kScalePre; ++k) {
        const uint4* src;
        uint4* dst;
        if (scale_unit(p, t + (int64_t)k * G, rec, &src, &dst)) *dst = scale_bf16x8(pre[k], c);
    }
    for (int64_t x = t + (int64_t)kScalePre * G; x < units; x += G) {
        const uint4* src;
        uint4* dst;
        scale_unit(p, x, rec, &src, &dst);
        *dst = scale_bf16x8(__ldcs(src), c);
    }
}

// Every layer of the step is a T == 1 bf16 layer: the norm kernel and the
// clip kernel in one launch.  A block of eight warps serves R = max(1, 8 / n)
// records: each warp takes (record, layer) items and forms the layer's partial
// from the sums of squares of the a and e rows in the norm kernel's order
// (vector l, l + 32, ... of each row for lane l), the partials meet in shared
// memory, and a warp per record combines them with the butterfly the clip
// kernel applies to one slot per lane -- so n2 and c are bitwise those of the
// two-kernel path.  A warp whose row is a pre-scaled operand keeps that row's
// vectors in registers and writes c_i times them once c_i is known (when every
// such row fits kKeepUnits vectors per lane; otherwise the block re-reads them).
constexpr int kFusedWarps = 8;

__global__ void __launch_bounds__(32 * kFusedWarps, 4) k_norm_clip_t1(const ClipParams p, const T1Group g,
                                                                   float* __restrict__ n2_out,
                                                                   float* __restrict__ c_out,
                                                                   float* __restrict__ n2_user,
                                                                   float* __restrict__ c_user,
                                                                   unsigned* __restrict__ status) {
    using T = __nv_bfloat16;
    __shared__ float part[kFusedWarps][32];
    __shared__ float cs[kFusedWarps];
    // A and E may come from the kernel just before this one on the stream
    grid_dep_wait();
    grid_dep_trigger();
    if (p.status_next && blockIdx.x == 0 && threadIdx.x == 0) *p.status_next = 0u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = g.n >= kFusedWarps ? 1 : kFusedWarps / g.n;
    const int64_t rec0 = (int64_t)blockIdx.x * R;
    // the row kept for pre-scaling by this warp's last item (at most one item
    // per warp when g.keep_x: the host allows it only for g.n <= kFusedWarps)
    uint4 keep[kKeepUnits];
    int keep_r = -1;
    uint4* keep_dst = nullptr;
    int64_t keep_n4 = 0;
    for (int item = warp; item < R * g.n; item += kFusedWarps) {
        const int r = item / g.n, l = item - r * g.n;
        const int64_t rec = rec0 + r;
        if (rec >= p.B) continue;
        const auto& ly = g.L[l];
        const uint4* a = (const uint4*)ly.A + rec * (ly.d_in / 8);
        const uint4* e = (const uint4*)ly.E + rec * (ly.d_out / 8);
        float sa, se;
        if (g.keep_x && ly.scale_job >= 0) {
            const uint4* x = ly.x_is_a ? a : e;
            const int64_t n4 = ly.x_is_a ? ly.d_in / 8 : ly.d_out / 8;
#pragma unroll
            for (int j = 0; j < kKeepUnits; ++j)
                if (lane + 32 * j < n4) keep[j] = __ldg(x + lane + 32 * j);
            const float so = warp_sum(sumsq_vec<T>(ly.x_is_a ? e : a, ly.x_is_a ? ly.d_out / 8 : ly.d_in / 8, lane));
            float sx = 0.f;
#pragma unroll
            for (int j = 0; j < kKeepUnits; ++j) {
                if (lane + 32 * j < n4) {
                    const T* q = (const T*)&keep[j];
#pragma unroll
                    for (int u = 0; u < 8; ++u) { const float f = (float)q[u]; sx = fmaf(f, f, sx); }
                }
            }
            sx = warp_sum(sx);
            sa = ly.x_is_a ? sx : so;
            se = ly.x_is_a ? so : sx;
            keep_r = r;
            keep_dst = p.scale[ly.scale_job].dst + rec * n4;
            keep_n4 = n4;
        } else {
            sa = warp_sum(sumsq_vec<T>(a, ly.d_in / 8, lane));
            se = warp_sum(sumsq_vec<T>(e, ly.d_out / 8, lane));
        }
        if (lane == 0) part[r][l] = t1_partial(sa, se, ly.has_bias);
    }
    __syncthreads();
    if (warp < R && rec0 + warp < p.B) {
        const int64_t rec = rec0 + warp;
        const float s = warp_sum(lane < g.n ? part[warp][lane] : 0.f);
        const bool finite = isfinite(s);
        // C / n rounded toward zero keeps c * n <= C in float arithmetic
        const float c = !finite ? 0.f : (sqrtf(s) <= p.C ? 1.0f : __fdiv_rz(p.C, sqrtf(s)));
        if (lane == 0) {
            if (!finite) atomicOr(status, 1u);
            n2_out[rec] = s;
            c_out[rec] = c;
            if (n2_user) n2_user[rec] = s;
            if (c_user) c_user[rec] = c;
            cs[warp] = c;
        }
    }
    if (p.nscale == 0) return;
    __syncthreads();
    if (g.keep_x) {
        if (keep_r >= 0) {
            const float c = cs[keep_r];
#pragma unroll
            for (int j = 0; j < kKeepUnits; ++j)
                if (lane + 32 * j < keep_n4) keep_dst[lane + 32 * j] = scale_bf16x8(keep[j], c);
        }
        return;
    }
    int64_t units = 0;
    for (int j = 0; j < p.nscale; ++j) units += p.scale[j].units;
    const int nrec = p.B - rec0 < R ? (int)(p.B - rec0) : R;
    for (int64_t x = threadIdx.x; x < (int64_t)nrec * units; x += blockDim.x) {
        const int r = (int)(x / units);
        const uint4* src;
        uint4* dst;
        scale_unit(p, x - (int64_t)r * units, rec0 + r, &src, &dst);
        *dst = scale_bf16x8(__ldg(src), cs[r]);
    }
}

// --------------------------------------------- stored-gradient weighted sum
struct WsumParams {
    int n;
    GradTask t[kMaxGroup];
};

// acc += c_i g_i[p .. p+3] for records i .. i+N-1 in ascending order, all N loads issued first
template <int N>
__device__ __forceinline__ void wsum_round(const float4* g4, int64_t stride4, const float* c, int64_t i,
                                           float4& acc) {
    float4 v[N];
    float cv[N];
#pragma unroll
    for (int u = 0; u < N; ++u) {
        v[u] = __ldcg(g4 + (i + u) * stride4);
        cv[u] = __ldca(c + i + u);
    }
#pragma unroll
    for (int u = 0; u < N; ++u) {
        acc.x = fmaf(cv[u], v[u].x, acc.x);
        acc.y = fmaf(cv[u], v[u].y, acc.y);
        acc.z = fmaf(cv[u], v[u].z, acc.z);
        acc.w = fmaf(cv[u], v[u].w, acc.w);
    }
}

// blockIdx.y = layer of the group; each thread owns one Philox block of the
// layer's coordinates (up to 4 coordinates) and sums c_i g_i[p] over records
// in ascending order.
__global__ void __launch_bounds__(256) k_grad_wsum(const WsumParams P, const float* __restrict__ c,
                                                   const unsigned* __restrict__ status, StepScalars sc) {
    const GradTask& t = P.t[blockIdx.y];
    const int64_t ncl = t.d_out * t.d_in + (t.has_bias ? t.d_out : 0);
    const int64_t j0 = t.coord_off >> 2;
    const int64_t j_last = (t.coord_off + ncl - 1) >> 2;
    const float scale = sc.sigma * sc.C;
    const bool vec = ((t.coord_off | ncl) & 3) == 0;   // Philox blocks = aligned float4 of G and g_i
    int64_t j = j0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // the first block's noise depends on no earlier kernel: drawn before waiting for them
    float4 z4 = j <= j_last ? noise4(sc.seed, sc.step, (uint64_t)j) : make_float4(0.f, 0.f, 0.f, 0.f);
    grid_dep_wait();
    grid_dep_trigger();
    if (status_bad(status)) return;
    for (bool first = true; j <= j_last; j += (int64_t)gridDim.x * blockDim.x, first = false) {
        if (!first) z4 = noise4(sc.seed, sc.step, (uint64_t)j);
        if (vec) {
            const int64_t p = 4 * j - t.coord_off;
            const float4* g4 = reinterpret_cast<const float4*>(t.gstore + p);
            const int64_t stride4 = ncl / 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            int64_t i = 0;
            // records in ascending order; sixteen (then eight) records' loads in flight per thread
            for (; i + 16 <= sc.B; i += 16) wsum_round<16>(g4, stride4, c, i, acc);
            for (; i + 8 <= sc.B; i += 8) wsum_round<8>(g4, stride4, c, i, acc);
            for (; i < sc.B; ++i) {
                const float4 v = __ldcg(g4 + i * stride4);
                const float ci = __ldca(c + i);
                acc.x = fmaf(ci, v.x, acc.x);
                acc.y = fmaf(ci, v.y, acc.y);
                acc.z = fmaf(ci, v.z, acc.z);
                acc.w = fmaf(ci, v.w, acc.w);
            }
            float4 o;
            o.x = (acc.x + scale * z4.x) / sc.L;
            o.y = (acc.y + scale * z4.y) / sc.L;
            o.z = (acc.z + scale * z4.z) / sc.L;
            o.w = (acc.w + scale * z4.w) / sc.L;
            *reinterpret_cast<float4*>(t.G + p) = o;
        } else {
            const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t p = 4 * j + q - t.coord_off;
                if (p < 0 || p >= ncl) continue;
                float acc = 0.f;
                for (int64_t i = 0; i < sc.B; ++i) acc = fmaf(__ldca(c + i), __ldcg(t.gstore + i * ncl + p), acc);
                t.G[p] = (acc + scale * zz[q]) / sc.L;
            }
        }
    }
}

// ---------------------------------------- reweighted E^T diag(c) A (CUDA core)
constexpr int kBM = 64, kBN = 64, kBK = 32;
constexpr int kGemmLoads = kBK * kBM / 256;   // elements of each operand a thread stages per chunk

// One 64 x 64 tile of G per block, K in chunks of 32 rows.  A and E were
// written before the step's first kernel (at least two launches back), so
// the block fetches its first chunk before the dependency wait, which guards
// only c and the status word; each later chunk (with its clip factors) is
// fetched into registers while the block computes on the one before.
template <int DT>
__global__ void __launch_bounds__(256) k_grad_gemm_cc(const GradTask t, const float* __restrict__ c,
                                                      const unsigned* __restrict__ status, StepScalars sc) {
    using Tt = typename Elem<DT>::T;
    __shared__ float Es[kBK][kBM];
    __shared__ float As[kBK][kBN];
    const int tid = threadIdx.x;
    const int tr = tid >> 4, tc = tid & 15;
    const int64_t m0 = (int64_t)blockIdx.y * kBM, n0 = (int64_t)blockIdx.x * kBN;
    const int64_t K = sc.B * t.T;
    const Tt* E = (const Tt*)t.E;
    const Tt* A = (const Tt*)t.A;
    // the thread's places of a chunk: row idx >> 6, column idx & 63, idx = tid + 256 r
    float er[kGemmLoads], ar[kGemmLoads], cr[kGemmLoads];
    auto fetch = [&](int64_t k0, bool with_c) {
#pragma unroll
        for (int r = 0; r < kGemmLoads; ++r) {
            const int idx = tid + 256 * r;
            const int64_t k = k0 + (idx >> 6);
            const int col = idx & 63;
            er[r] = (k < K && m0 + col < t.d_out) ? Elem<DT>::ld(E + k * t.d_out + m0 + col) : 0.f;
            ar[r] = (k < K && n0 + col < t.d_in) ? Elem<DT>::ld(A + k * t.d_in + n0 + col) : 0.f;
            if (with_c) cr[r] = k < K ? __ldca(c + k / t.T) : 0.f;
        }
    };
    fetch(0, false);
    grid_dep_wait();
    grid_dep_trigger();
    if (status_bad(status)) return;
#pragma unroll
    for (int r = 0; r < kGemmLoads; ++r) {
        const int64_t k = (tid + 256 * r) >> 6;
        cr[r] = k < K ? __ldca(c + k / t.T) : 0.f;
    }
    float acc[4][4] = {};
    float bsum = 0.f;
    const bool do_bias = t.has_bias && blockIdx.x == 0;
    for (int64_t k0 = 0; k0 < K; k0 += kBK) {
#pragma unroll
        for (int r = 0; r < kGemmLoads; ++r) {
            const int idx = tid + 256 * r;
            const int kk = idx >> 6, col = idx & 63;
            Es[kk][col] = cr[r] * er[r];
            As[kk][col] = ar[r];
        }
        __syncthreads();
        if (k0 + kBK < K) fetch(k0 + kBK, true);
#pragma unroll 8
        for (int kk = 0; kk < kBK; ++kk) {
            float ev[4], av[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ev[i] = Es[kk][tr * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) av[j] = As[kk][tc * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ev[i], av[j], acc[i][j]);
        }
        if (do_bias && tid < kBM) {
            for (int kk = 0; kk < kBK; ++kk) bsum += Es[kk][tid];
        }
        __syncthreads();
    }
    // the epilogue stays rolled: small launches of this kernel run with a
    // cold instruction cache, where code size is time
    const float scale = sc.sigma * sc.C;
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + tr * 4 + i;
        if (m >= t.d_out) continue;
        const int64_t nb = n0 + tc * 4;
        const uint64_t kb = (uint64_t)(t.coord_off + m * t.d_in + nb);
        float z[4];
        if ((kb & 3u) == 0 && nb + 4 <= t.d_in) {
            // the four coordinates are one Philox block
            const float4 z4 = noise4(sc.seed, sc.step, kb >> 2);
            z[0] = z4.x;
            z[1] = z4.y;
            z[2] = z4.z;
            z[3] = z4.w;
        } else {
#pragma unroll 1
            for (int j = 0; j < 4; ++j) z[j] = nb + j < t.d_in ? noise_at(sc.seed, sc.step, kb + j) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = nb + j;
            if (n >= t.d_in) continue;
            t.G[m * t.d_in + n] = (acc[i][j] + scale * z[j]) / sc.L;
        }
    }
    if (do_bias && tid < kBM && m0 + tid < t.d_out) {
        const int64_t p = t.d_out * t.d_in + m0 + tid;
        const float z = noise_at(sc.seed, sc.step, (uint64_t)(t.coord_off + p));
        t.G[p] = (bsum + scale * z) / sc.L;
    }
}

// The same sum for outputs too small to occupy the GPU with 64 x 64 tiles:
// one 16 x 16 tile per block, one output per thread, K in chunks of 128 rows
// (the first fetched before the dependency wait, as above).  A block whose
// tile starts the row holds the bias sums of its 16 rows.
constexpr int kSmallTile = 16, kSmallBK = 128;
constexpr int kSmallLoads = kSmallBK * kSmallTile / 256;   // elements of each operand a thread stages per chunk

template <int DT>
__global__ void __launch_bounds__(256) k_grad_gemm_small(const GradTask t, const float* __restrict__ c,
                                                         const unsigned* __restrict__ status, StepScalars sc) {
    using Tt = typename Elem<DT>::T;
    __shared__ float Es[kSmallBK][kSmallTile];
    __shared__ float As[kSmallBK][kSmallTile];
    const int tid = threadIdx.x;
    const int tr = tid >> 4, tc = tid & 15;   // output row and column within the tile
    const int64_t m0 = (int64_t)blockIdx.y * kSmallTile, n0 = (int64_t)blockIdx.x * kSmallTile;
    const int64_t K = sc.B * t.T;
    const Tt* E = (const Tt*)t.E;
    const Tt* A = (const Tt*)t.A;
    // the thread's places of a chunk: row idx >> 4, column idx & 15, idx = tid + 256 r
    float er[kSmallLoads], ar[kSmallLoads], cr[kSmallLoads];
    auto fetch = [&](int64_t k0, bool with_c) {
#pragma unroll
        for (int r = 0; r < kSmallLoads; ++r) {
            const int idx = tid + 256 * r;
            const int64_t k = k0 + (idx >> 4);
            const int col = idx & 15;
            er[r] = (k < K && m0 + col < t.d_out) ? Elem<DT>::ld(E + k * t.d_out + m0 + col) : 0.f;
            ar[r] = (k < K && n0 + col < t.d_in) ? Elem<DT>::ld(A + k * t.d_in + n0 + col) : 0.f;
            if (with_c) cr[r] = k < K ? __ldca(c + k / t.T) : 0.f;
        }
    };
    fetch(0, false);
    grid_dep_wait();
    grid_dep_trigger();
    if (status_bad(status)) return;
#pragma unroll
    for (int r = 0; r < kSmallLoads; ++r) {
        const int64_t k = (tid + 256 * r) >> 4;
        cr[r] = k < K ? __ldca(c + k / t.T) : 0.f;
    }
    float acc = 0.f, bsum = 0.f;
    const bool do_bias = t.has_bias && blockIdx.x == 0;
    for (int64_t k0 = 0; k0 < K; k0 += kSmallBK) {
#pragma unroll
        for (int r = 0; r < kSmallLoads; ++r) {
            const int idx = tid + 256 * r;
            Es[idx >> 4][idx & 15] = cr[r] * er[r];
            As[idx >> 4][idx & 15] = ar[r];
        }
        __syncthreads();
        if (k0 + kSmallBK < K) fetch(k0 + kSmallBK, true);
#pragma unroll 16
        for (int kk = 0; kk < kSmallBK; ++kk) acc = fmaf(Es[kk][tr], As[kk][tc], acc);
        if (do_bias && tid < kSmallTile) {
            for (int kk = 0; kk < kSmallBK; ++kk) bsum += Es[kk][tid];
        }
        __syncthreads();
    }
    const float scale = sc.sigma * sc.C;
    const int64_t m = m0 + tr, n = n0 + tc;
    if (m < t.d_out && n < t.d_in) {
        const float z = noise_at(sc.seed, sc.step, (uint64_t)(t.coord_off + m * t.d_in + n));
        t.G[m * t.d_in + n] = (acc + scale * z) / sc.L;
    }
    if (do_bias && tid < kSmallTile && m0 + tid < t.d_out) {
        const int64_t p = t.d_out * t.d_in + m0 + tid;
        const float z = noise_at(sc.seed, sc.step, (uint64_t)(t.coord_off + p));
        t.G[p] = (bsum + scale * z) / sc.L;
    }
}

// --------------------------------------------- bias part of the clipped sum
// sb[m] = sum_k c[k / T] E[k, m] (ascending k), then G = (sb + sigma C z) / L
// at the layer's bias coordinates.  Used beside the tensor-core weight sum.
template <int DT>
__global__ void __launch_bounds__(256) k_bias_sum(const GradTask t, const float* __restrict__ c,
                                                  const unsigned* __restrict__ status, StepScalars sc) {
    using Tt = typename Elem<DT>::T;
    grid_dep_wait();
    grid_dep_trigger();
    if (status_bad(status)) return;
    const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= t.d_out) return;
    const Tt* E = (const Tt*)t.E;
    const int64_t K = sc.B * t.T;
    float acc = 0.f;
    for (int64_t k = 0; k < K; ++k) acc = fmaf(__ldca(c + k / t.T), Elem<DT>::ld(E + k * t.d_out + m), acc);
    const int64_t p = t.d_out * t.d_in + m;
    t.G[p] = (acc + sc.sigma * sc.C * noise_at(sc.seed, sc.step, (uint64_t)(t.coord_off + p))) / sc.L;
}

// ------------------------------------- clip factor folded into the operand
// X'[k, :] = bf16(c[k / T] * X[k, :]), X the operand (A or E) with fewer
// columns, for the tensor-core clipped sum of layers whose records do not
// span whole 64-row tiles (T = 1 included).
// One thread per 8 consecutive elements of a row (d % 8 == 0); the product is
// formed in fp32 and rounded to nearest.
__global__ void __launch_bounds__(256) k_prescale_rows(const uint4* __restrict__ E, uint4* __restrict__ E2,
                                                       const float* __restrict__ c, int64_t K, int64_t T,
                                                       int64_t d8) {
    grid_dep_wait();
    grid_dep_trigger();
    const int64_t n = K * d8;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = q / d8;
        const float ck = __ldca(c + k / T);
        uint4 v = __ldcs(E + q);
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w[i]);
            const float2 f = __bfloat1622float2(h);
            h = __floats2bfloat162_rn(f.x * ck, f.y * ck);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        E2[q] = v;
    }
}

// ------------------------------------------- noise on a coordinate range
// G[j] = (S[j] + scale z_{k0 + j}) / L for 0 <= j < n: the noise and the
// normalizer applied to a contiguous range of global coordinates (one rank's
// shard of the summed clipped gradient when the records are split over
// ranks).  One thread per noise block (4 coordinates) of the range; vector
// loads and stores when k0 % 4 == 0 and both arrays are 16-byte aligned.
template <bool VEC>
__global__ void __launch_bounds__(256) k_noise_shard(const float* __restrict__ S, float* __restrict__ G, uint64_t k0,
                                                     int64_t n, float scale, float L, uint64_t seed, uint64_t step) {
    const uint64_t jb = k0 >> 2;
    const int64_t nblocks = (int64_t)((k0 + (uint64_t)n - 1) >> 2) - (int64_t)jb + 1;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t j = jb + (uint64_t)b;
        const float4 z = noise4(seed, step, j);
        const float zz[4] = {z.x, z.y, z.z, z.w};
        const int64_t p0 = (int64_t)(4 * j - k0);   // index in S of the block's first coordinate
        if (VEC && p0 + 3 < n) {
            const float4 v = __ldcs(reinterpret_cast<const float4*>(S + p0));
            float4 o;
            o.x = (v.x + scale * zz[0]) / L;
            o.y = (v.y + scale * zz[1]) / L;
            o.z = (v.z + scale * zz[2]) / L;
            o.w = (v.w + scale * zz[3]) / L;
            __stcs(reinterpret_cast<float4*>(G + p0), o);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t p = p0 + q;
                if (p >= 0 && p < n) G[p] = (S[p] + scale * zz[q]) / L;
            }
        }
    }
}

// ------------------------------------------------------- noise test hook
// The Box-Muller map of the noise on given word pairs (words[2i], words[2i+1])
// -> (z[2i], z[2i+1]): the same device function as every noise draw.
__global__ void k_box_muller(const uint2* __restrict__ words, int64_t npairs, float2* __restrict__ z) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npairs;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint2 w = words[i];
        z[i] = box_muller(w.x, w.y);
    }
}

__global__ void k_philox_normals(uint64_t seed, uint64_t step, uint64_t k0, int64_t n,
                                 uint32_t* __restrict__ raw, float* __restrict__ z) {
    const int64_t jb = (int64_t)(k0 >> 2);
    const int64_t nblocks = (int64_t)((k0 + n - 1) >> 2) - jb + 1;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t j = (uint64_t)(jb + b);
        const uint4 w = noise_block(seed, step, j);
        if (raw) {
            raw[4 * b + 0] = w.x;
            raw[4 * b + 1] = w.y;
            raw[4 * b + 2] = w.z;
            raw[4 * b + 3] = w.w;
        }
        if (z) {
            const float2 p0 = box_muller(w.x, w.y);
            const float2 p1 = box_muller(w.z, w.w);
            const float v[4] = {p0.x, p0.y, p1.x, p1.y};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t k = (int64_t)(4 * j + q) - (int64_t)k0;
                if (k >= 0 && k < n) z[k] = v[q];
            }
        }
    }
}

}  // namespace

cudaError_t launch_clip(const ClipParams& p, float* n2, float* c, float* n2_user, float* c_user,
                        unsigned* status, cudaStream_t s) {
    cudaError_t e;
    const int G = clip_group(p.total_slots);
    if (G == 32) {
        const int per_block = kClipWarpBlock / 32;
        const unsigned grid = (unsigned)((p.B + per_block - 1) / per_block);
        e = launch_dependent(k_clip<true>, dim3(grid), dim3(kClipWarpBlock), 0, s, p, n2, c, n2_user, c_user, status);
    } else {
        e = launch_dependent(k_clip<false>, dim3((unsigned)p.B), dim3(G), 0, s, p, n2, c, n2_user, c_user, status);
    }
    count_launch(KL_CLIP);
    return e;
}

cudaError_t launch_norm_clip_t1(const ClipParams& p, const T1Group& g, float* n2, float* c, float* n2_user,
                                float* c_user, unsigned* status, cudaStream_t s) {
    const int R = g.n >= kFusedWarps ? 1 : kFusedWarps / g.n;   // records per block
    const unsigned grid = (unsigned)((p.B + R - 1) / R);
    const cudaError_t e = launch_dependent(k_norm_clip_t1, dim3(grid), dim3(32 * kFusedWarps), 0, s, p, g, n2, c,
                                           n2_user, c_user, status);
    count_launch(KL_NORM_CLIP_T1);
    return e;
}

cudaError_t launch_grad_wsum(const GradTask* tasks, int n, const float* c, const unsigned* status,
                             const StepScalars& sc, cudaStream_t s) {
    for (int base = 0; base < n; base += kMaxGroup) {
        WsumParams P;
        P.n = n - base < kMaxGroup ? n - base : kMaxGroup;
        int64_t maxblk = 1;
        for (int i = 0; i < P.n; ++i) {
            P.t[i] = tasks[base + i];
            const GradTask& t = P.t[i];
            const int64_t ncl = t.d_out * t.d_in + (t.has_bias ? t.d_out : 0);
            const int64_t nb = ((t.coord_off + ncl - 1) >> 2) - (t.coord_off >> 2) + 1;
            maxblk = nb > maxblk ? nb : maxblk;
        }
        int64_t gx = (maxblk + 255) / 256;
        if (gx > 4096) gx = 4096;
        const cudaError_t e = launch_dependent(k_grad_wsum, dim3((unsigned)gx, (unsigned)P.n), dim3(256), 0, s, P, c,
                                               status, sc);
        count_launch(KL_GRAD_WSUM);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_grad_gemm_cc(const GradTask& t, const float* c, const unsigned* status,
                                const StepScalars& sc, cudaStream_t s) {
    const dim3 grid((unsigned)((t.d_in + kBN - 1) / kBN), (unsigned)((t.d_out + kBM - 1) / kBM));
    if (grid.x * grid.y < 16) {
        // too few 64 x 64 tiles to spread over the SMs: 16 x 16 tiles
        const dim3 g16((unsigned)((t.d_in + kSmallTile - 1) / kSmallTile),
                       (unsigned)((t.d_out + kSmallTile - 1) / kSmallTile));
        const cudaError_t e =
            t.dtype == DT_F32 ? launch_dependent(k_grad_gemm_small<DT_F32>, g16, dim3(256), 0, s, t, c, status, sc)
                              : launch_dependent(k_grad_gemm_small<DT_BF16>, g16, dim3(256), 0, s, t, c, status, sc);
        count_launch(KL_GRAD_GEMM_SMALL);
        return e;
    }
    const cudaError_t e = t.dtype == DT_F32
                              ? launch_dependent(k_grad_gemm_cc<DT_F32>, grid, dim3(256), 0, s, t, c, status, sc)
                              : launch_dependent(k_grad_gemm_cc<DT_BF16>, grid, dim3(256), 0, s, t, c, status, sc);
    count_launch(KL_GRAD_GEMM_CC);
    return e;
}

cudaError_t launch_bias_sum(const GradTask& t, const float* c, const unsigned* status, const StepScalars& sc,
                            cudaStream_t s) {
    const unsigned grid = (unsigned)((t.d_out + 255) / 256);
    const cudaError_t e = t.dtype == DT_F32
                              ? launch_dependent(k_bias_sum<DT_F32>, dim3(grid), dim3(256), 0, s, t, c, status, sc)
                              : launch_dependent(k_bias_sum<DT_BF16>, dim3(grid), dim3(256), 0, s, t, c, status, sc);
    count_launch(KL_BIAS_SUM);
    return e;
}

cudaError_t launch_prescale_rows(const void* E, void* E2, const float* c, int64_t K, int64_t T, int64_t d,
                                 cudaStream_t s) {
    const int64_t n = K * (d / 8);
    int64_t grid = (n + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dependent(k_prescale_rows, dim3((unsigned)grid), dim3(256), 0, s,
                                           (const uint4*)E, (uint4*)E2, c, K, T, d / 8);
    count_launch(KL_PRESCALE_ROWS);
    return e;
}

cudaError_t launch_box_muller(const uint32_t* words, int64_t npairs, float* z, cudaStream_t s) {
    if (npairs <= 0) return cudaSuccess;
    int64_t grid = (npairs + 255) / 256;
    if (grid > 152 * 64) grid = 152 * 64;
    k_box_muller<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<const uint2*>(words), npairs,
                                                reinterpret_cast<float2*>(z));
    count_launch(KL_BOX_MULLER);
    return cudaGetLastError();
}

cudaError_t launch_philox_normals(uint64_t seed, uint64_t step, uint64_t k0, int64_t n,
                                  uint32_t* raw, float* z, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t nblocks = (int64_t)((k0 + n - 1) >> 2) - (int64_t)(k0 >> 2) + 1;
    int64_t grid = (nblocks + 255) / 256;
    if (grid > 152 * 64) grid = 152 * 64;
    k_philox_normals<<<(unsigned)grid, 256, 0, s>>>(seed, step, k0, n, raw, z);
    count_launch(KL_PHILOX_NORMALS);
    return cudaGetLastError();
}

cudaError_t launch_noise_shard(const float* S, float* G, uint64_t k0, int64_t n, float scale, float L,
                               uint64_t seed, uint64_t step, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t nblocks = (int64_t)((k0 + (uint64_t)n - 1) >> 2) - (int64_t)(k0 >> 2) + 1;
    int64_t grid = (nblocks + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;   // 8 resident blocks of 256 threads per SM
    if (grid > cap) grid = cap;
    const bool vec = (k0 & 3u) == 0 && (reinterpret_cast<uintptr_t>(S) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
    if (vec) k_noise_shard<true><<<(unsigned)grid, 256, 0, s>>>(S, G, k0, n, scale, L, seed, step);
    else k_noise_shard<false><<<(unsigned)grid, 256, 0, s>>>(S, G, k0, n, scale, L, seed, step);
    count_launch(KL_NOISE_SHARD);
    return cudaGetLastError();
}
