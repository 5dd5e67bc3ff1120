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
// the batched mode LLM.int8 ships with.  The integer product is exact
// (int32, dp4a on the CUDA cores: GB300's int8 tensor rate is low and the
// layer is a producer off the gradient hot path); the correction runs over
// the set's columns in ascending order, one fused multiply-add each.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dp_clip.h"
#include "internal.h"

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

// per (record, 32-column word): bit set when some row of the record has |a| >= tau
__global__ void k_int8_sets(const __half* __restrict__ A, int64_t K, int64_t rows, int64_t words, float tau,
                            uint32_t* __restrict__ sets, uint32_t* __restrict__ uni) {
    const int64_t r = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int64_t word = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (word >= words) return;
    const int64_t j = word * 32 + lane;
    bool hit = false;
    if (j < K)
        for (int64_t i = r * rows; i < (r + 1) * rows; ++i) hit |= fabsf(__half2float(A[i * K + j])) >= tau;
    const uint32_t bits = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) {
        sets[r * words + word] = bits;
        if (bits) atomicOr(uni + word, bits);
    }
}

// row-local scales: max |a| over the row's entries below tau
__global__ void k_int8_scales(const __half* __restrict__ A, int64_t n, int64_t K, float tau, float* __restrict__ s) {
    const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= n) return;
    float m = 0.f;
    for (int64_t j = lane; j < K; j += 32) {
        const float a = fabsf(__half2float(A[i * K + j]));
        if (a < tau) m = fmaxf(m, a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s[i] = m;
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

}  // namespace

extern "C" int64_t dp_int8_workspace_bytes(int64_t n, int64_t K, int64_t rows_per_record) {
    if (n < 0 || K < 1 || rows_per_record < 1 || n % rows_per_record) return -1;
    const int64_t words = (K + 31) / 32;
    const int64_t records = n / rows_per_record;
    const int64_t sets = ((records + 1) * words * 4 + 15) / 16 * 16;
    return sets + (n * 4 + 15) / 16 * 16;
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
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return DP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t words = (K + 31) / 32;
    const int64_t records = n / rows_per_record;
    uint32_t* sets = static_cast<uint32_t*>(workspace);
    uint32_t* uni = sets + records * words;
    float* scales = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                             ((records + 1) * words * 4 + 15) / 16 * 16);
    if (cudaMemsetAsync(uni, 0, (size_t)words * 4, s) != cudaSuccess) return DP_ERR_CUDA;
    k_int8_sets<<<dim3((unsigned)((words + 7) / 8), (unsigned)records), 256, 0, s>>>(
        static_cast<const __half*>(A), K, rows_per_record, words, tau, sets, uni);
    k_int8_scales<<<(unsigned)((n + 7) / 8), 256, 0, s>>>(static_cast<const __half*>(A), n, K, tau, scales);
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
    count_launch(KL_INT8_SETS);
    count_launch(KL_INT8_SCALES);
    count_launch(KL_INT8_GEMM);
    return cudaGetLastError() == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}
