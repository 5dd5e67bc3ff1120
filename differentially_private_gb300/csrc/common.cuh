// Device helpers shared by the kernels of the library: element loads,
// warp reductions, the Philox4x32-10 generator and the Box-Muller map.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dpk {

// ---------------------------------------------------------------- elements
template <int DT> struct Elem;
template <> struct Elem<DT_F32> {
    using T = float;
    static __device__ __forceinline__ float ld(const float* p) { return __ldg(p); }
};
template <> struct Elem<DT_BF16> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }
};

// Sum over the 32 lanes with a fixed xor butterfly (same order on every call).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide sum of one value per thread, fixed order: warp butterflies, then
// warp 0 sums the warp totals in warp order.  `red` holds >= 32 floats.
// Every thread receives the total.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    if (warp == 0) {
        t = lane < nwarps ? red[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    t = red[0];
    __syncthreads();
    return t;
}

// Sum of squares of one row read as 16-byte vectors by a warp: lane l takes
// vectors l, l + 32, ... in that order (eight loads in flight per lane).
template <typename T>
__device__ __forceinline__ float sumsq_vec(const uint4* __restrict__ p, int64_t n4, int lane) {
    constexpr int PER = 16 / (int)sizeof(T);
    float s = 0.f;
    int64_t k = lane;
    for (; k + 224 < n4; k += 256) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldg(p + k + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const T* x = (const T*)&v[u];
#pragma unroll
            for (int q = 0; q < PER; ++q) { const float f = (float)x[q]; s = fmaf(f, f, s); }
        }
    }
    for (; k < n4; k += 32) {
        const uint4 v = __ldg(p + k);
        const T* x = (const T*)&v;
#pragma unroll
        for (int q = 0; q < PER; ++q) { const float f = (float)x[q]; s = fmaf(f, f, s); }
    }
    return s;
}

// The T == 1 closed form of one layer's squared norm from the two row sums of
// squares: ||a||^2 ||e||^2, plus ||e||^2 for a bias, as one fused multiply-add.
__device__ __forceinline__ float t1_partial(float sa, float se, int has_bias) {
    return fmaf(sa, se, has_bias ? se : 0.f);
}

// ---------------------------------------------------------------- Philox
// Philox-4x32 with ten rounds (Salmon, Moraes, Dror, Shaw, SC'11): each round
// multiplies counter words 0 and 2 by two fixed odd constants, keeps the low
// halves as the new words 3 and 1 and xors the high halves with the other
// counter words and the round key to form the new words 0 and 2; the key is
// advanced by the two Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t p0_lo = 0xD2511F53u * c.x;
        const uint32_t p0_hi = __umulhi(0xD2511F53u, c.x);
        const uint32_t p1_lo = 0xCD9E8D57u * c.z;
        const uint32_t p1_hi = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(p1_hi ^ c.y ^ k0, p1_lo, p0_hi ^ c.w ^ k1, p0_lo);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Words of noise block j (coordinates 4j .. 4j+3) of the (seed, step) stream.
__device__ __forceinline__ uint4 noise_block(uint64_t seed, uint64_t step, uint64_t j) {
    const uint4 ctr = make_uint4((uint32_t)j, (uint32_t)(j >> 32), (uint32_t)step, (uint32_t)(step >> 32));
    return philox4x32_10(ctr, (uint32_t)seed, (uint32_t)(seed >> 32));
}

// Box-Muller: u1 = ((xa >> 8) + 1) 2^-24 in (0, 1], u2 = (xb >> 8) 2^-24 in
// [0, 1), r = sqrt(-2 ln u1), (r cos 2 pi u2, r sin 2 pi u2).  Both uniforms
// are exact in float; the transcendental calls are CUDA's own.
__device__ __forceinline__ float2 box_muller(uint32_t xa, uint32_t xb) {
    const float u1 = (float)((xa >> 8) + 1u) * 0x1p-24f;
    const float u2 = (float)(xb >> 8) * 0x1p-24f;
    const float r = sqrtf(-2.0f * logf(u1));
    float s, c;
    sincospif(2.0f * u2, &s, &c);
    return make_float2(r * c, r * s);
}

// The four normals of block j.
__device__ __forceinline__ float4 noise4(uint64_t seed, uint64_t step, uint64_t j) {
    const uint4 w = noise_block(seed, step, j);
    const float2 a = box_muller(w.x, w.y);
    const float2 b = box_muller(w.z, w.w);
    return make_float4(a.x, a.y, b.x, b.y);
}

// The 4 NB normals of blocks j0 .. j0+NB-1.  The NB Philox evaluations run
// round by round side by side and the 2 NB Box-Muller pairs are independent,
// so a thread has several dependency chains in flight (the GEMM epilogues run
// with few warps per SM and would otherwise wait on one long chain).
template <int NB>
__device__ __forceinline__ void noise_blocks(uint64_t seed, uint64_t step, uint64_t j0, float (&z)[4 * NB]) {
    uint4 c[NB];
#pragma unroll
    for (int q = 0; q < NB; ++q) {
        const uint64_t j = j0 + q;
        c[q] = make_uint4((uint32_t)j, (uint32_t)(j >> 32), (uint32_t)step, (uint32_t)(step >> 32));
    }
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            const uint32_t p0_lo = 0xD2511F53u * c[q].x;
            const uint32_t p0_hi = __umulhi(0xD2511F53u, c[q].x);
            const uint32_t p1_lo = 0xCD9E8D57u * c[q].z;
            const uint32_t p1_hi = __umulhi(0xCD9E8D57u, c[q].z);
            c[q] = make_uint4(p1_hi ^ c[q].y ^ k0, p1_lo, p0_hi ^ c[q].w ^ k1, p0_lo);
        }
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
#pragma unroll
    for (int q = 0; q < NB; ++q) {
        const float2 a = box_muller(c[q].x, c[q].y);
        const float2 b = box_muller(c[q].z, c[q].w);
        z[4 * q] = a.x;
        z[4 * q + 1] = a.y;
        z[4 * q + 2] = b.x;
        z[4 * q + 3] = b.y;
    }
}

// The normal of one coordinate k (computes its whole block).
__device__ __forceinline__ float noise_at(uint64_t seed, uint64_t step, uint64_t k) {
    const uint4 w = noise_block(seed, step, k >> 2);
    const int lane = (int)(k & 3);
    const float2 p = lane < 2 ? box_muller(w.x, w.y) : box_muller(w.z, w.w);
    return (lane & 1) ? p.y : p.x;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream is still
// running.  grid_dep_wait() returns once that kernel has completed and its
// writes are visible (a no-op after a normal launch); nothing the previous
// kernels wrote may be read before it.  grid_dep_trigger() lets the next
// kernel of the stream begin launching; it is issued only after the wait, so
// a kernel that starts early can never overtake the kernel two places ahead.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Loads after grid_dep_wait().  Data another kernel wrote that each address
// of is read once (partial norms, stored per-example gradients) is loaded
// with __ldcg (L2 only).  The clip factors c_i are read by every warp of the
// grid: they are loaded with __ldca (cached in L1 as well), so that each SM
// fetches a line once instead of every warp sending a request to the same
// L2 line.

__device__ __forceinline__ bool status_bad(const unsigned* status) {
    return (*(volatile const unsigned*)status) != 0u;
}

}  // namespace dpk
