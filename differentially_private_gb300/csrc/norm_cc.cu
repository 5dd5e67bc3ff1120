// Per-example squared-norm kernels on the CUDA cores.
//
//  * T == 1 closed form (ghost path of a non-sequence layer):
//      ||e a^T||_F^2 = ||a||^2 ||e||^2, plus ||e||^2 for a bias.
//  * Ghost norm for T > 1 by tiled Grams:
//      ||E_i^T A_i||_F^2 = <A_i A_i^T, E_i E_i^T>, bias 1^T E_i E_i^T 1.
//  * Materialized norm: g_i = E_i^T A_i tile by tile, ||g_i||_F^2, optionally
//    storing g_i (and the bias gradient sum_t E_i[t]) for the clipped sum.
// Ghost clipping obtains the clip factor without forming every full
// per-example gradient ("Privacy-Preserving Machine Learning", section
// "Differentially private stochastic gradient descent", phase 2).
//
// Every kernel writes per-(record, tile) partial sums to its own slots; no
// atomics.  A record's partials depend on its own rows and on the shapes
// only, so its norm is bitwise the same for any batch ("Sensitivity
// Inflation from Cross-Record Precision Routing in Private Quantized
// Fine-Tuning", Proposition 2).
#include "common.cuh"
#include "launch.cuh"

using namespace dpk;

namespace {

constexpr int kGT = 32;   // Gram / gradient tile edge

// ------------------------------------------------------------------ T == 1
// Several T == 1 layers in one launch (bf16, rows of whole 16-byte vectors):
// blockIdx.y selects the layer, one warp per record.

__global__ void __launch_bounds__(256) k_norm_t1_group(const T1Group g) {
    using T = __nv_bfloat16;
    // may start while the previous kernel of the stream runs: A and E are read
    // only after it completed
    grid_dep_wait();
    grid_dep_trigger();
    const auto& ly = g.L[blockIdx.y];
    const int64_t rec = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (rec >= g.B) return;
    const float sa = warp_sum(sumsq_vec<T>((const uint4*)ly.A + rec * (ly.d_in / 8), ly.d_in / 8, lane));
    const float se = warp_sum(sumsq_vec<T>((const uint4*)ly.E + rec * (ly.d_out / 8), ly.d_out / 8, lane));
    if (lane == 0) ly.partial[rec] = t1_partial(sa, se, ly.has_bias);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(256) k_norm_t1(const void* __restrict__ Av, const void* __restrict__ Ev,
                                                 int64_t B, int64_t d_in, int64_t d_out, int has_bias,
                                                 float* __restrict__ partial) {
    using T = typename Elem<DT>::T;
    const int64_t rec = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (rec >= B) return;
    const T* a = (const T*)Av + rec * d_in;
    const T* e = (const T*)Ev + rec * d_out;
    float sa = 0.f, se = 0.f;
    if constexpr (VEC) {
        sa = sumsq_vec<T>((const uint4*)a, d_in / (16 / (int)sizeof(T)), lane);
        se = sumsq_vec<T>((const uint4*)e, d_out / (16 / (int)sizeof(T)), lane);
    } else {
        for (int64_t k = lane; k < d_in; k += 32) { const float f = Elem<DT>::ld(a + k); sa = fmaf(f, f, sa); }
        for (int64_t k = lane; k < d_out; k += 32) { const float f = Elem<DT>::ld(e + k); se = fmaf(f, f, se); }
    }
    sa = warp_sum(sa);
    se = warp_sum(se);
    if (lane == 0) partial[rec] = t1_partial(sa, se, has_bias);
}

// ------------------------------------------------------------ ghost Gram
// Upper-triangular tile (p, q), p <= q, of the T x T Gram matrices.
__device__ __forceinline__ void tri_tile(int tile, int nt, int& p, int& q) {
    p = 0;
    int rem = tile;
    while (rem >= nt - p) { rem -= nt - p; ++p; }
    q = p + rem;
}

// Accumulate the 32x32 Gram tile X[rows p] . X[rows q]^T over the feature axis.
template <int DT>
__device__ __forceinline__ void gram_tile(const typename Elem<DT>::T* X, int64_t T, int64_t d, int p, int q,
                                          float (*Xs)[kGT + 1], float (*Ys)[kGT + 1], float acc[4]) {
    const int tid = threadIdx.x, lane = tid & 31, ty = tid >> 5;
    for (int64_t k0 = 0; k0 < d; k0 += kGT) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int idx = tid + 256 * r;
            const int row = idx >> 5, col = idx & 31;
            const int64_t s = (int64_t)p * kGT + row, t = (int64_t)q * kGT + row, k = k0 + col;
            Xs[row][col] = (s < T && k < d) ? Elem<DT>::ld(X + s * d + k) : 0.f;
            Ys[row][col] = (t < T && k < d) ? Elem<DT>::ld(X + t * d + k) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kGT; ++kk) {
            const float y = Ys[lane][kk];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(Xs[ty + 8 * j][kk], y, acc[j]);
        }
        __syncthreads();
    }
}

template <int DT>
__global__ void __launch_bounds__(256) k_norm_ghost_cc(const void* __restrict__ Av, const void* __restrict__ Ev,
                                                       int64_t T, int64_t d_in, int64_t d_out, int has_bias,
                                                       float* __restrict__ partial, int nslots) {
    using Tt = typename Elem<DT>::T;
    __shared__ float Xs[kGT][kGT + 1];
    __shared__ float Ys[kGT][kGT + 1];
    __shared__ float red[32];
    const int nt = (int)((T + kGT - 1) / kGT);
    const int64_t rec = (int64_t)blockIdx.x / nslots;
    const int tile = (int)((int64_t)blockIdx.x % nslots);
    int p, q;
    tri_tile(tile, nt, p, q);
    const Tt* A = (const Tt*)Av + rec * T * d_in;
    const Tt* E = (const Tt*)Ev + rec * T * d_out;
    float ga[4] = {0.f, 0.f, 0.f, 0.f}, ge[4] = {0.f, 0.f, 0.f, 0.f};
    gram_tile<DT>(A, T, d_in, p, q, Xs, Ys, ga);
    gram_tile<DT>(E, T, d_out, p, q, Xs, Ys, ge);
    // rows/cols outside [0, T) hold zeros in both Grams, so they add nothing
    float v = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) v += ga[j] * ge[j] + (has_bias ? ge[j] : 0.f);
    if (p != q) v *= 2.f;   // tile (q, p) of the symmetric product is the same
    v = block_sum(v, red);
    if (threadIdx.x == 0) partial[rec * nslots + tile] = v;
}

// ------------------------------------------------------ materialized norm
template <int DT>
__global__ void __launch_bounds__(256) k_norm_mat_cc(const void* __restrict__ Av, const void* __restrict__ Ev,
                                                     int64_t T, int64_t d_in, int64_t d_out, int has_bias,
                                                     float* __restrict__ partial, int nslots,
                                                     float* __restrict__ gstore) {
    using Tt = typename Elem<DT>::T;
    __shared__ float Es[kGT][kGT + 1];
    __shared__ float As[kGT][kGT + 1];
    __shared__ float red[32];
    const int tid = threadIdx.x, lane = tid & 31, ty = tid >> 5;
    const int ntn = (int)((d_in + kGT - 1) / kGT);
    const int64_t rec = (int64_t)blockIdx.x / nslots;
    const int slot = (int)((int64_t)blockIdx.x % nslots);
    const int mt = slot / ntn, ntile = slot % ntn;
    const int64_t m0 = (int64_t)mt * kGT, n0 = (int64_t)ntile * kGT;
    const Tt* A = (const Tt*)Av + rec * T * d_in;
    const Tt* E = (const Tt*)Ev + rec * T * d_out;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float bsum = 0.f;   // bias gradient of row m0 + lane (tiles with ntile == 0, warp 0)
    for (int64_t t0 = 0; t0 < T; t0 += kGT) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int idx = tid + 256 * r;
            const int row = idx >> 5, col = idx & 31;
            const int64_t t = t0 + row;
            Es[row][col] = (t < T && m0 + col < d_out) ? Elem<DT>::ld(E + t * d_out + m0 + col) : 0.f;
            As[row][col] = (t < T && n0 + col < d_in) ? Elem<DT>::ld(A + t * d_in + n0 + col) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int tt = 0; tt < kGT; ++tt) {
            const float a = As[tt][lane];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(Es[tt][ty + 8 * j], a, acc[j]);
        }
        if (has_bias && ntile == 0 && ty == 0) {
            for (int tt = 0; tt < kGT; ++tt) bsum += Es[tt][lane];
        }
        __syncthreads();
    }
    const int64_t ncl = d_out * d_in + (has_bias ? d_out : 0);
    float v = 0.f;
    const int64_t n = n0 + lane;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t m = m0 + ty + 8 * j;
        if (m < d_out && n < d_in) {
            v = fmaf(acc[j], acc[j], v);
            if (gstore) gstore[rec * ncl + m * d_in + n] = acc[j];
        }
    }
    if (has_bias && ntile == 0 && ty == 0 && m0 + lane < d_out) {
        v = fmaf(bsum, bsum, v);
        if (gstore) gstore[rec * ncl + d_out * d_in + m0 + lane] = bsum;
    }
    v = block_sum(v, red);
    if (tid == 0) partial[rec * nslots + slot] = v;
}

// ------------------------------------------------------ per-layer totals
__global__ void k_layer_sqnorm(const float* __restrict__ partial, int nslots, int64_t B, float* __restrict__ out) {
    const int64_t rec = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (rec >= B) return;
    float s = 0.f;
    for (int j = lane; j < nslots; j += 32) s += partial[rec * nslots + j];
    s = warp_sum(s);
    if (lane == 0) out[rec] = s;
}

// The same, for partials whose producers report a wait that gave up in
// *status: every total is NaN when the word is not zero.
__global__ void k_layer_sqnorm_status(const float* __restrict__ partial, int nslots, int64_t B,
                                      float* __restrict__ out, const unsigned* __restrict__ status) {
    const int64_t rec = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (rec >= B) return;
    float s = 0.f;
    for (int j = lane; j < nslots; j += 32) s += partial[rec * nslots + j];
    s = warp_sum(s);
    if (lane == 0) out[rec] = status_bad(status) ? __int_as_float(0x7fc00000) : s;
}

inline int ntri(int64_t T) {
    const int64_t nt = (T + kGT - 1) / kGT;
    return (int)(nt * (nt + 1) / 2);
}

}  // namespace

int nslots_cc(int kernel, int64_t T, int64_t d_in, int64_t d_out) {
    switch (kernel) {
        case NK_T1: return 1;
        case NK_GHOST_CC: return ntri(T);
        case NK_MAT_CC: return (int)(((d_out + kGT - 1) / kGT) * ((d_in + kGT - 1) / kGT));
        default: return -1;
    }
}

cudaError_t launch_norm_t1(const NormTask& t, int64_t B, cudaStream_t s) {
    const int threads = 256;
    const int64_t blocks = (B * 32 + threads - 1) / threads;
    const size_t esz = t.dtype == DT_F32 ? 4 : 2;
    const bool vec = ((t.d_in * esz) % 16 == 0) && ((t.d_out * esz) % 16 == 0);
    if (t.dtype == DT_F32) {
        if (vec) k_norm_t1<DT_F32, true><<<(unsigned)blocks, threads, 0, s>>>(t.A, t.E, B, t.d_in, t.d_out, t.has_bias, t.partial);
        else k_norm_t1<DT_F32, false><<<(unsigned)blocks, threads, 0, s>>>(t.A, t.E, B, t.d_in, t.d_out, t.has_bias, t.partial);
    } else {
        if (vec) k_norm_t1<DT_BF16, true><<<(unsigned)blocks, threads, 0, s>>>(t.A, t.E, B, t.d_in, t.d_out, t.has_bias, t.partial);
        else k_norm_t1<DT_BF16, false><<<(unsigned)blocks, threads, 0, s>>>(t.A, t.E, B, t.d_in, t.d_out, t.has_bias, t.partial);
    }
    count_launch(KL_NORM_T1);
    return cudaGetLastError();
}

bool t1_groupable(const NormTask& t) { return t.dtype == DT_BF16 && t.d_in % 8 == 0 && t.d_out % 8 == 0; }

cudaError_t launch_norm_t1_group(const NormTask* tasks, int n, int64_t B, cudaStream_t s) {
    for (int base = 0; base < n; base += kMaxGroup) {
        T1Group g;
        g.n = n - base < kMaxGroup ? n - base : kMaxGroup;
        g.B = B;
        for (int i = 0; i < g.n; ++i) {
            const NormTask& t = tasks[base + i];
            g.L[i].A = t.A;
            g.L[i].E = t.E;
            g.L[i].d_in = t.d_in;
            g.L[i].d_out = t.d_out;
            g.L[i].has_bias = t.has_bias;
            g.L[i].partial = t.partial;
            g.L[i].scale_job = -1;
            g.L[i].x_is_a = 0;
        }
        g.keep_x = 0;
        const dim3 grid((unsigned)((B * 32 + 255) / 256), (unsigned)g.n);
        const cudaError_t e = launch_dependent(k_norm_t1_group, grid, dim3(256), 0, s, g);
        count_launch(KL_NORM_T1_GROUP);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_norm_ghost_cc(const NormTask& t, int64_t B, cudaStream_t s) {
    const dim3 grid((unsigned)(B * t.nslots));
    if (t.dtype == DT_F32)
        k_norm_ghost_cc<DT_F32><<<grid, 256, 0, s>>>(t.A, t.E, t.T, t.d_in, t.d_out, t.has_bias, t.partial, t.nslots);
    else
        k_norm_ghost_cc<DT_BF16><<<grid, 256, 0, s>>>(t.A, t.E, t.T, t.d_in, t.d_out, t.has_bias, t.partial, t.nslots);
    count_launch(KL_NORM_GHOST_CC);
    return cudaGetLastError();
}

cudaError_t launch_norm_mat_cc(const NormTask& t, int64_t B, cudaStream_t s) {
    const dim3 grid((unsigned)(B * t.nslots));
    if (t.dtype == DT_F32)
        k_norm_mat_cc<DT_F32><<<grid, 256, 0, s>>>(t.A, t.E, t.T, t.d_in, t.d_out, t.has_bias, t.partial, t.nslots, t.gstore);
    else
        k_norm_mat_cc<DT_BF16><<<grid, 256, 0, s>>>(t.A, t.E, t.T, t.d_in, t.d_out, t.has_bias, t.partial, t.nslots, t.gstore);
    count_launch(KL_NORM_MAT_CC);
    return cudaGetLastError();
}

cudaError_t launch_layer_sqnorm(const float* partial, int nslots, int64_t B, float* out, cudaStream_t s) {
    const int threads = 256;
    const int64_t blocks = (B * 32 + threads - 1) / threads;
    k_layer_sqnorm<<<(unsigned)blocks, threads, 0, s>>>(partial, nslots, B, out);
    count_launch(KL_LAYER_SQNORM);
    return cudaGetLastError();
}

cudaError_t launch_layer_sqnorm_checked(const float* partial, int nslots, int64_t B, float* out,
                                        const unsigned* status, cudaStream_t s) {
    const int threads = 256;
    const int64_t blocks = (B * 32 + threads - 1) / threads;
    k_layer_sqnorm_status<<<(unsigned)blocks, threads, 0, s>>>(partial, nslots, B, out, status);
    count_launch(KL_LAYER_SQNORM_STATUS);
    return cudaGetLastError();
}
