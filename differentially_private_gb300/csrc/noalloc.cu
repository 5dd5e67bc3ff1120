// dp_layer_sqnorms_static: per-example squared gradient norms of one layer
// with no device allocation at all.
//
// Some callers cannot call cudaMalloc: a process that reserved all device
// memory for its own pool at start-up, a host program whose device memory
// is owned by another framework's allocator, or a latency-bound loop that
// cannot afford the device-wide synchronization cudaMalloc and cudaFree may
// perform.  For them this entry point runs the same norm kernels as
// dp_norm_accumulate (chosen by the same shape rule) but takes the partial
// sums those kernels write from a fixed array in this file, resolved once
// per device with cudaGetSymbolAddress.  The caller passes A, E and the
// output; nothing else is needed, no context either.
#include <mutex>

#include "../../include/dp_clip.h"
#include "internal.h"

namespace {

// Largest B * (partial slots per record) one call may need: 2^20 floats (4 MiB).
constexpr int64_t kStaticPartials = int64_t(1) << 20;

// The scratch itself.  Every GPU that loads the library holds it until exit.
static __device__ __align__(256) float g_static_partials[kStaticPartials];
// Status word the tensor-core kernels report a wait timeout into (padded to 256 bytes).
static __device__ __align__(256) unsigned g_static_status[64];

struct DeviceScratch {
    float* partials = nullptr;
    unsigned* status = nullptr;
    CUcontext ctx = nullptr;   // the context the addresses belong to
    bool ready = false;
};

constexpr int kMaxDevices = 128;
DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// cuCtxGetCurrent, fetched once through the runtime (the library does not
// link libcuda directly).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static const CtxGetCurrentFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (CtxGetCurrentFn) nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(ptr);
    }();
    return fn;
}

// Host code may not use the arrays' names as device addresses: resolve them
// for the current device, checking the return codes.  The addresses are
// kept per device and resolved again when the device's current context is
// not the one they were resolved in (after a cudaDeviceReset the module is
// loaded anew and the old addresses are stale).
dp_status scratch_for_current_device(DeviceScratch* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DP_ERR_CUDA;
    const CtxGetCurrentFn get = ctx_get_current();
    if (!get) return DP_ERR_CUDA;
    // no context may be current yet on this thread: the runtime binds the
    // device's primary context when the addresses are first resolved
    CUcontext cur = nullptr;
    if (get(&cur) != CUDA_SUCCESS) return DP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    DeviceScratch& s = g_scratch[dev];
    if (!s.ready || !cur || s.ctx != cur) {
        s.ready = false;
        void* p = nullptr;
        void* q = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_partials) != cudaSuccess) {
            cudaGetLastError();
            return DP_ERR_CUDA;
        }
        if (cudaGetSymbolAddress(&q, g_static_status) != cudaSuccess) {
            cudaGetLastError();
            return DP_ERR_CUDA;
        }
        if (get(&cur) != CUDA_SUCCESS || !cur) return DP_ERR_CUDA;
        s.partials = static_cast<float*>(p);
        s.status = static_cast<unsigned*>(q);
        s.ctx = cur;
        s.ready = true;
    }
    *out = s;
    return DP_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" dp_status dp_layer_sqnorms_static(const void* A, const void* E, int64_t B, int64_t T, int64_t d_in,
                                             int64_t d_out, int has_bias, dp_dtype dtype, float* sqnorm_out,
                                             void* stream) {
    NvtxRange nvtx_range("dp_layer_sqnorms_static");
    if (!A || !E || !sqnorm_out) return DP_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(E, 16) || !aligned(sqnorm_out, 4)) return DP_ERR_INVALID_ARG;
    if (dtype != DP_F32 && dtype != DP_BF16) return DP_ERR_INVALID_ARG;
    if (B < 1 || T < 1 || d_in < 1 || d_out < 1) return DP_ERR_SHAPE;
    const unsigned __int128 rows = (unsigned __int128)(uint64_t)B * (uint64_t)T;
    if (rows >= ((unsigned __int128)1 << 31)) return DP_ERR_SHAPE;
    if (rows * (uint64_t)(d_in > d_out ? d_in : d_out) >= ((unsigned __int128)1 << 62)) return DP_ERR_SHAPE;
    const int dt = dtype == DP_F32 ? DT_F32 : DT_BF16;
    int nslots = 0;
    const int kind = plan_norm_kernel(dt, T, d_in, d_out, has_bias ? 1 : 0, &nslots);
    if (nslots <= 0) return DP_ERR_UNSUPPORTED;
    // the fixed scratch bounds the request
    if ((unsigned __int128)(uint64_t)B * (uint64_t)nslots > (unsigned __int128)kStaticPartials) return DP_ERR_SHAPE;

    DeviceScratch sc;
    const dp_status st = scratch_for_current_device(&sc);
    if (st != DP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The partial slots are all overwritten.  The status word is zero here:
    // it starts at zero and every call clears it after reading it.

    NormTask t;
    t.A = A;
    t.E = E;
    t.T = T;
    t.d_in = d_in;
    t.d_out = d_out;
    t.has_bias = has_bias ? 1 : 0;
    t.dtype = dt;
    t.partial = sc.partials;
    t.nslots = nslots;
    t.gstore = nullptr;
    t.maps = nullptr;
    alignas(64) CUtensorMap maps[2];
    cudaError_t e = cudaSuccess;
    switch (kind) {
        case NK_T1: e = launch_norm_t1(t, B, s); break;
        case NK_GHOST_CC: e = launch_norm_ghost_cc(t, B, s); break;
        case NK_MAT_CC: e = launch_norm_mat_cc(t, B, s); break;
        case NK_GHOST_TC:
            if (!tc_encode_gram(t, B, maps)) return DP_ERR_CUDA;
            t.maps = maps;
            e = launch_ghost_gram_tc(t, B, sc.status, s);
            break;
        case NK_MAT_TC:
            if (!tc_encode_skinny(t, B, maps)) return DP_ERR_CUDA;
            t.maps = maps;
            e = launch_mat_skinny_tc(&t, 1, B, sc.status, s);
            break;
        default: return DP_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return DP_ERR_CUDA;
    // a wait of the tensor-core kernels that gave up left their partials
    // unwritten: the totals are then NaN, so the caller sees a non-finite norm
    if (launch_layer_sqnorm_checked(sc.partials, nslots, B, sqnorm_out, sc.status, s) != cudaSuccess)
        return DP_ERR_CUDA;
    if (cudaMemsetAsync(sc.status, 0, sizeof(unsigned), s) != cudaSuccess) return DP_ERR_CUDA;
    return DP_OK;
}

extern "C" dp_status dp_static_check_wait_timeout(uint32_t limit_ms, void* stream) {
    NvtxRange nvtx_range("dp_static_check_wait_timeout");
    if (limit_ms < 1 || limit_ms > 2000) return DP_ERR_INVALID_ARG;
    DeviceScratch sc;
    const dp_status st = scratch_for_current_device(&sc);
    if (st != DP_OK) return st;
    const cudaError_t e =
        launch_wait_expiry(sc.status, (uint64_t)limit_ms * 1000000ull, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}
