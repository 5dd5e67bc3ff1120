// Records grouped by user for user-level clipping ("Privacy-Preserving
// Machine Learning", section "Differentially private stochastic gradient
// descent", the user-level construction: group records, build a vector per
// user, clip that vector).  A user's vector is the sum of its records'
// gradients, sum_i E_i^T A_i = E_u^T A_u with A_u, E_u the user's records
// stacked along T, so a user is one record of length k T for the rest of the
// library.  dp_pack_groups lays users with different record counts out as
// [U, kmax, T, d] (the missing records zero, which adds nothing to a norm or
// a sum).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dp_clip.h"
#include "internal.h"

namespace {

// one thread per 16-byte vector of the output; records of vec16 vectors
__global__ void k_pack_groups(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t B, int64_t vec16,
                              const int64_t* __restrict__ starts, int64_t U, int64_t kmax) {
    const int64_t total = U * kmax * vec16;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rec = q / vec16, off = q - rec * vec16;
        const int64_t u = rec / kmax, s = rec - u * kmax;
        const int64_t r = starts[u] + s;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < starts[u + 1] && r >= 0 && r < B) v = src[r * vec16 + off];
        dst[q] = v;
    }
}

__global__ void k_pack_groups_bytes(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t B,
                                    int64_t rec_bytes, const int64_t* __restrict__ starts, int64_t U, int64_t kmax) {
    const int64_t total = U * kmax * rec_bytes;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rec = q / rec_bytes, off = q - rec * rec_bytes;
        const int64_t u = rec / kmax, s = rec - u * kmax;
        const int64_t r = starts[u] + s;
        dst[q] = (r < starts[u + 1] && r >= 0 && r < B) ? src[r * rec_bytes + off] : (uint8_t)0;
    }
}

}  // namespace

extern "C" dp_status dp_pack_groups(const void* src, void* dst, int64_t B, int64_t T, int64_t d, int dtype,
                                    const int64_t* group_starts, int64_t U, int64_t kmax, void* stream) {
    NvtxRange nvtx_range("dp_pack_groups");
    if (!src || !dst || !group_starts) return DP_ERR_INVALID_ARG;
    if (dtype != DP_F32 && dtype != DP_BF16) return DP_ERR_INVALID_ARG;
    if (B < 0 || T < 1 || d < 1 || U < 0 || kmax < 0) return DP_ERR_SHAPE;
    const int64_t esz = dtype == DP_F32 ? 4 : 2;
    const int64_t rec_bytes = T * d * esz;
    const int64_t total = U * kmax * rec_bytes;
    if (total == 0) return DP_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool vec = rec_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    const int64_t items = vec ? total / 16 : total;
    int64_t grid = (items + 255) / 256;
    if (grid > 152 * 32) grid = 152 * 32;
    if (vec)
        k_pack_groups<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), B,
                                                   rec_bytes / 16, group_starts, U, kmax);
    else
        k_pack_groups_bytes<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint8_t*>(src),
                                                         static_cast<uint8_t*>(dst), B, rec_bytes, group_starts,
                                                         U, kmax);
    count_launch(KL_PACK_GROUPS);
    return cudaGetLastError() == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}
