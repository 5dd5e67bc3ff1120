// Host runtime behind the C ABI of include/dp_clip.h: the context, the layer
// registry and coordinate layout, the ghost / materialize chooser, the step
// state machine, context-owned device scratch and kernel planning.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/dp_clip.h"
#include "internal.h"

namespace {

constexpr int kVersion = 100;  // 0.1.0

// Per-example gradients of a materialized layer are kept for the weighted sum
// when they take at most this many bytes; otherwise the clipped sum re-reads
// A and E.
constexpr uint64_t kStoreBudgetBytes = 8ull << 30;

enum Phase { IDLE = 0, OPEN = 1, CLIPPED = 2 };

struct Layer {
    int64_t d_in = 0, d_out = 0;
    int has_bias = 0;
    int dtype = DT_F32;
    int64_t coord_off = 0, ncoords = 0;
    // per step
    bool accumulated = false;
    int path = DP_PATH_GHOST;
    int norm_kernel = NK_T1;
    int grad_kernel = GK_GEMM_CC;
    const void* A = nullptr;
    const void* E = nullptr;
    int64_t T = 0;
    int nslots = 0;
    bool stored = false;
    // context-owned device buffers
    float* partial = nullptr;
    size_t partial_cap = 0;   // floats
    float* gstore = nullptr;
    size_t gstore_cap = 0;    // floats
    // c_i E_i in bf16 for the tensor-core sum of a layer whose T is not a
    // multiple of 64 (the clip factor folded into the operand before the sum)
    bool prescale = false;     // clip factors folded into a bf16 copy of one operand
    bool prescale_A = false;   // that operand is A (fewer columns than E), else E
    float* escaled = nullptr;  // the pre-scaled copy
    bool scaled_by_clip = false;   // this step's copy is written by the clip kernel
    size_t escaled_cap = 0;   // floats (two bf16 each)
    // TMA descriptors of the tensor-core kernels, encoded once per request
    // shape: reused while (A, E, T, B) stay the same from step to step
    struct MapKey {
        const void* A = nullptr;
        const void* E = nullptr;
        int64_t T = 0, B = 0;
        int kind = -1;
        bool operator==(const MapKey& o) const {
            return A == o.A && E == o.E && T == o.T && B == o.B && kind == o.kind;
        }
    } nkey, gkey;
    CUtensorMap nmaps[2];   // the type carries the alignment TMA needs
    CUtensorMap gmaps[3];
};

}  // namespace

struct dp_ctx {
    int device = 0;
    cudaStream_t stream = nullptr;
    int sm_count = 0;
    std::vector<Layer> layers;
    int64_t P = 0;
    Phase phase = IDLE;
    int64_t B = 0;
    double L = 1.0;
    float C = 1.0f;
    float* n2 = nullptr;
    float* c = nullptr;
    size_t bcap = 0;
    size_t ccap = 0;
    unsigned* status_words = nullptr; // two status words: steps alternate between them
    unsigned* status = nullptr;        // the current step's word
    int slot = 1;                      // index of the current step's word
    bool clean[2] = {true, true};      // the word is known to be zero for the next step that takes it
    float* one = nullptr;              // device constant 1.0f
    float* fold_scratch = nullptr;     // partial sums of split tiles of the tensor-core clipped sum
    unsigned long long* fold_counters = nullptr;   // their arrival counters (zeroed once)
    unsigned fold_epoch = 0;           // tag of the last clipped-sum launch
    SlotRef* d_slots = nullptr;        // clip kernel's flat view of every layer's partial slots
    size_t d_slots_cap = 0;
    std::vector<std::pair<const float*, int64_t>> slots_key;   // (partial, nslots) per layer d_slots was built from
    std::vector<SlotRef> h_slots;      // host copy of d_slots (the source of its last upload)
    // every layer of the step T == 1 and accumulated in one batch call without
    // per-layer outputs: their norms are deferred to the clip call, which runs
    // norms, clip factors and pre-scaled copies in one kernel
    bool t1_fused = false;
    std::vector<NormTask> t1_tasks;    // in registration order
    std::string err;
};

namespace {

// launch tag of the clipped-sum split counters; 0 is never used, so the
// zeroed counters match no launch
unsigned next_fold_epoch(dp_ctx* ctx) {
    if (++ctx->fold_epoch == 0) ++ctx->fold_epoch;
    return ctx->fold_epoch;
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

dp_status fail(dp_ctx* ctx, dp_status s, const char* fmt, ...) {
    if (ctx) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        ctx->err = buf;
    }
    return s;
}

dp_status cuda_fail(dp_ctx* ctx, cudaError_t e, const char* what) {
    return fail(ctx, DP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Grow a context-owned float buffer to at least n floats.  Synchronizes the
// stream before releasing the old buffer, which only happens when a step
// needs more room than any earlier one.
dp_status grow(dp_ctx* ctx, float** buf, size_t* cap, size_t n) {
    if (n <= *cap && *buf) return DP_OK;
    cudaError_t e;
    if (*buf) {
        e = cudaStreamSynchronize(ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
        cudaFree(*buf);
        *buf = nullptr;
        *cap = 0;
    }
    const size_t want = std::max<size_t>(n, 64);
    e = cudaMalloc(reinterpret_cast<void**>(buf), want * sizeof(float));
    if (e != cudaSuccess) {
        cudaGetLastError();
        *buf = nullptr;
        return fail(ctx, DP_ERR_OOM, "cudaMalloc of %zu bytes failed: %s", want * sizeof(float),
                    cudaGetErrorString(e));
    }
    *cap = want;
    return DP_OK;
}

int choose(int64_t T, int64_t d_in, int64_t d_out) {
    // exact T^2 < d_in * d_out on unsigned 128-bit products
    const unsigned __int128 t2 = (unsigned __int128)(uint64_t)T * (uint64_t)T;
    const unsigned __int128 dd = (unsigned __int128)(uint64_t)d_in * (uint64_t)d_out;
    return t2 < dd ? DP_PATH_GHOST : DP_PATH_MATERIALIZE;
}

// Kernel choice depends on the shapes and dtype only, never on B, so that a
// record's norm does not depend on the batch it is in.
void plan_norm(Layer& ly, int64_t T) {
    ly.path = choose(T, ly.d_in, ly.d_out);
    if (ly.path == DP_PATH_GHOST) {
        if (T == 1) ly.norm_kernel = NK_T1;
        else if (tc_gram_supported(ly.dtype, T, ly.d_in, ly.d_out)) ly.norm_kernel = NK_GHOST_TC;
        else ly.norm_kernel = NK_GHOST_CC;
    } else {
        ly.norm_kernel = tc_skinny_supported(ly.dtype, ly.d_in, ly.d_out, ly.has_bias) ? NK_MAT_TC : NK_MAT_CC;
    }
    ly.nslots = nslots_for(ly.norm_kernel, T, ly.d_in, ly.d_out);
}

NormTask make_norm_task(const Layer& ly) {
    NormTask t;
    t.A = ly.A;
    t.E = ly.E;
    t.T = ly.T;
    t.d_in = ly.d_in;
    t.d_out = ly.d_out;
    t.has_bias = ly.has_bias;
    t.dtype = ly.dtype;
    t.partial = ly.partial;
    t.nslots = ly.nslots;
    t.gstore = ly.stored ? ly.gstore : nullptr;
    t.maps = (ly.norm_kernel == NK_MAT_TC || ly.norm_kernel == NK_GHOST_TC) ? ly.nmaps : nullptr;
    return t;
}

dp_status launch_norm(dp_ctx* ctx, const Layer& ly) {
    const NormTask t = make_norm_task(ly);
    cudaError_t e = cudaSuccess;
    switch (ly.norm_kernel) {
        case NK_T1: e = launch_norm_t1(t, ctx->B, ctx->stream); break;
        case NK_GHOST_CC: e = launch_norm_ghost_cc(t, ctx->B, ctx->stream); break;
        case NK_MAT_CC: e = launch_norm_mat_cc(t, ctx->B, ctx->stream); break;
        case NK_MAT_TC: e = launch_mat_skinny_tc(&t, 1, ctx->B, ctx->status, ctx->stream); break;
        case NK_GHOST_TC: e = launch_ghost_gram_tc(t, ctx->B, ctx->status, ctx->stream); break;
        default: return fail(ctx, DP_ERR_UNSUPPORTED, "no norm kernel %d", ly.norm_kernel);
    }
    if (e != cudaSuccess) return cuda_fail(ctx, e, "norm kernel launch");
    return DP_OK;
}

// Validate one accumulate request without changing any state.
dp_status check_accumulate(dp_ctx* ctx, int id, const void* A, const void* E, int64_t T) {
    if (ctx->phase != OPEN)
        return fail(ctx, DP_ERR_STATE, "dp_norm_accumulate needs an open step before dp_clip_factors");
    if (id < 0 || id >= (int)ctx->layers.size()) return fail(ctx, DP_ERR_INVALID_ARG, "unknown layer id %d", id);
    if (ctx->layers[id].accumulated)
        return fail(ctx, DP_ERR_STATE, "layer %d was already accumulated in this step", id);
    if (T < 1) return fail(ctx, DP_ERR_SHAPE, "T must be >= 1 (got %lld)", (long long)T);
    if (!A || !E) return fail(ctx, DP_ERR_INVALID_ARG, "A and E must not be NULL");
    if (!aligned16(A) || !aligned16(E)) return fail(ctx, DP_ERR_INVALID_ARG, "A and E must be 16-byte aligned");
    const Layer& ly = ctx->layers[id];
    const unsigned __int128 rows = (unsigned __int128)(uint64_t)ctx->B * (uint64_t)T;
    if (rows * (uint64_t)std::max(ly.d_in, ly.d_out) >= ((unsigned __int128)1 << 62))
        return fail(ctx, DP_ERR_SHAPE, "B*T*d overflows");
    if (rows >= ((unsigned __int128)1 << 31)) return fail(ctx, DP_ERR_SHAPE, "B*T must be below 2^31");
    return DP_OK;
}

// Plan one layer's step work and size its context scratch; no launch.
dp_status prepare(dp_ctx* ctx, int id, const void* A, const void* E, int64_t T, Layer& plan) {
    Layer& ly = ctx->layers[id];
    plan = ly;
    plan.A = A;
    plan.E = E;
    plan.T = T;
    plan_norm(plan, T);
    if (plan.nslots <= 0) return fail(ctx, DP_ERR_UNSUPPORTED, "no norm plan for layer %d", id);
    dp_status st = grow(ctx, &ly.partial, &ly.partial_cap, (size_t)ctx->B * plan.nslots);
    if (st != DP_OK) return st;
    plan.partial = ly.partial;
    plan.partial_cap = ly.partial_cap;
    plan.stored = false;
    if (plan.path == DP_PATH_MATERIALIZE &&
        (uint64_t)ctx->B * (uint64_t)ly.ncoords * 4u <= kStoreBudgetBytes) {
        st = grow(ctx, &ly.gstore, &ly.gstore_cap, (size_t)ctx->B * ly.ncoords);
        if (st != DP_OK) return st;
        plan.gstore = ly.gstore;
        plan.gstore_cap = ly.gstore_cap;
        plan.stored = true;
    }
    if (plan.stored) plan.grad_kernel = GK_WSUM;
    else if (tc_sum_supported(plan.dtype, plan.d_in, plan.d_out, plan.has_bias)) plan.grad_kernel = GK_GEMM_TC;
    else plan.grad_kernel = GK_GEMM_CC;
    // descriptors of the tensor-core kernels, re-encoded only when the request changed
    if (plan.norm_kernel == NK_MAT_TC || plan.norm_kernel == NK_GHOST_TC) {
        Layer::MapKey key;
        key.A = A;
        key.E = E;
        key.T = T;
        key.B = ctx->B;
        key.kind = plan.norm_kernel;
        if (!(key == plan.nkey)) {
            plan.nkey = Layer::MapKey();
            NormTask t = make_norm_task(plan);
            t.maps = nullptr;
            const bool ok = plan.norm_kernel == NK_MAT_TC ? tc_encode_skinny(t, ctx->B, plan.nmaps)
                                                           : tc_encode_gram(t, ctx->B, plan.nmaps);
            if (!ok) return fail(ctx, DP_ERR_CUDA, "TMA descriptor encoding failed for layer %d", id);
            plan.nkey = key;
        }
    }
    plan.prescale = plan.grad_kernel == GK_GEMM_TC && T % 64 != 0;
    // c_i can scale either operand's rows: the narrower one is copied
    plan.prescale_A = plan.prescale && plan.d_in < plan.d_out;
    if (plan.prescale) {
        const int64_t dsc = plan.prescale_A ? plan.d_in : plan.d_out;
        st = grow(ctx, &ly.escaled, &ly.escaled_cap, ((size_t)ctx->B * T * dsc + 1) / 2);
        if (st != DP_OK) return st;
        plan.escaled = ly.escaled;
        plan.escaled_cap = ly.escaled_cap;
    }
    if (plan.grad_kernel == GK_GEMM_TC && !ctx->fold_scratch) {
        const int sms = device_sm_count();
        cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&ctx->fold_scratch), fold_scratch_floats(sms) * sizeof(float));
        if (e == cudaSuccess)
            e = cudaMalloc(reinterpret_cast<void**>(&ctx->fold_counters), (size_t)sms * sizeof(unsigned long long));
        if (e == cudaSuccess) e = cudaMemset(ctx->fold_counters, 0, (size_t)sms * sizeof(unsigned long long));
        if (e != cudaSuccess) {
            cudaGetLastError();
            cudaFree(ctx->fold_scratch);
            cudaFree(ctx->fold_counters);
            ctx->fold_scratch = nullptr;
            ctx->fold_counters = nullptr;
            return fail(ctx, DP_ERR_OOM, "allocation of the clipped-sum scratch failed");
        }
    }
    if (plan.grad_kernel == GK_GEMM_TC) {
        // the sum reads the pre-scaled copy as one record of B*T rows when prescaling
        const void* Asum = plan.prescale_A ? static_cast<const void*>(plan.escaled) : A;
        const void* Esum = plan.prescale && !plan.prescale_A ? static_cast<const void*>(plan.escaled) : E;
        Layer::MapKey key;
        key.A = Asum;
        key.E = Esum;
        key.T = T;
        key.B = ctx->B;
        key.kind = GK_GEMM_TC;
        if (!(key == plan.gkey)) {
            plan.gkey = Layer::MapKey();
            GradTask g{};
            g.A = Asum;
            g.E = Esum;
            g.T = T;
            g.d_in = plan.d_in;
            g.d_out = plan.d_out;
            if (!tc_encode_sum(g, ctx->B, plan.gmaps))
                return fail(ctx, DP_ERR_CUDA, "TMA descriptor encoding failed for layer %d", id);
            plan.gkey = key;
        }
    }
    return DP_OK;
}

dp_status finish(dp_ctx* ctx, int id, Layer& plan, float* sq) {
    if (sq) {
        const cudaError_t e = launch_layer_sqnorm(plan.partial, plan.nslots, ctx->B, sq, ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "layer norm launch");
    }
    plan.accumulated = true;
    ctx->layers[id] = plan;
    return DP_OK;
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
    static const EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({dev, kernel})) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({dev, kernel});
    return e;
}

static std::atomic<int64_t> g_launches{0};
static std::atomic<int64_t> g_kernel_launches[KL_COUNT];

// Names of the kernels, in KernelId order.
static const char* const kKernelNames[KL_COUNT] = {
    "k_norm_t1", "k_norm_t1_group", "k_norm_ghost_cc", "k_norm_mat_cc", "k_layer_sqnorm",
    "k_layer_sqnorm_status", "k_ghost_gram_tc", "k_mat_skinny_tc", "k_clip", "k_norm_clip_t1", "k_grad_wsum",
    "k_grad_gemm_small", "k_grad_gemm_cc", "k_bias_sum", "k_prescale_rows", "k_clipped_sum_fold_pair_tc",
    "k_clipped_sum_tc", "k_sum_layers_pair_tc", "k_noise_shard", "k_box_muller", "k_philox_normals",
    "k_pack_groups", "k_int8_quantize_weight", "k_int8_rowscan", "k_int8_gemm",
    "k_int8_codes", "k_int8_gemm_tc", "k_wait_expires",
};

void count_launch(KernelId k) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    g_kernel_launches[k].fetch_add(1, std::memory_order_relaxed);
}

NvtxRange::NvtxRange(const char* name) { nvtxRangePushA(name); }
NvtxRange::~NvtxRange() { nvtxRangePop(); }

int plan_norm_kernel(int dtype, int64_t T, int64_t d_in, int64_t d_out, int has_bias, int* nslots) {
    Layer ly;
    ly.d_in = d_in;
    ly.d_out = d_out;
    ly.has_bias = has_bias;
    ly.dtype = dtype;
    plan_norm(ly, T);
    *nslots = ly.nslots;
    return ly.norm_kernel;
}

int nslots_for(int kernel, int64_t T, int64_t d_in, int64_t d_out) {
    if (kernel == NK_MAT_TC) return nslots_skinny(d_in, d_out);
    if (kernel == NK_GHOST_TC) return nslots_gram(T);
    return nslots_cc(kernel, T, d_in, d_out);
}

namespace {

// The gradient phase of a step: G = (sum_i c_i g_i + sigma C z) / L for every
// layer, with L the step's normalizer (dp_clipped_noisy_grad) or 1 and
// sigma = 0 (dp_clipped_sum: the clipped sum alone).
dp_status clipped_grad(dp_ctx* ctx, float sigma, uint64_t seed, uint64_t step, float* const* G, float L,
                       const char* who) {
    if (ctx->phase != CLIPPED) return fail(ctx, DP_ERR_STATE, "%s needs dp_clip_factors first", who);
    if (!G) return fail(ctx, DP_ERR_INVALID_ARG, "G must not be NULL");
    for (size_t l = 0; l < ctx->layers.size(); ++l)
        if (!G[l] || !aligned16(G[l])) return fail(ctx, DP_ERR_INVALID_ARG, "G[%zu] is NULL or not 16-byte aligned", l);
    DeviceGuard g(ctx->device);
    StepScalars sc;
    sc.B = ctx->B;
    sc.C = ctx->C;
    sc.sigma = sigma;
    sc.L = L;
    sc.seed = seed;
    sc.step = step;
    // layers whose pre-scaled operand the clip kernel wrote are summed together
    // (layers with the same K in one launch); their bias sums follow them
    std::vector<GradTask> wsum, single, single_bias;
    for (size_t l = 0; l < ctx->layers.size(); ++l) {
        const Layer& ly = ctx->layers[l];
        GradTask t;
        t.A = ly.A;
        t.E = ly.E;
        t.T = ly.T;
        t.d_in = ly.d_in;
        t.d_out = ly.d_out;
        t.has_bias = ly.has_bias;
        t.dtype = ly.dtype;
        t.gstore = ly.gstore;
        t.G = G[l];
        t.coord_off = ly.coord_off;
        t.maps = ly.grad_kernel == GK_GEMM_TC ? ly.gmaps : nullptr;
        if (ly.grad_kernel == GK_WSUM) {
            wsum.push_back(t);
            continue;
        }
        cudaError_t e;
        if (ly.grad_kernel == GK_GEMM_TC && ly.prescale && ly.scaled_by_clip) {
            GradTask ts = t;
            if (ly.prescale_A) ts.A = ly.escaled;
            else ts.E = ly.escaled;
            ts.T = ctx->B * ly.T;
            single.push_back(ts);
            if (ly.has_bias) single_bias.push_back(t);
            continue;
        }
        if (ly.grad_kernel == GK_GEMM_TC && ly.prescale) {
            // c_i folded into a bf16 copy of the narrower operand, then one "record" of B*T rows with factor 1
            const int64_t K = ctx->B * ly.T;
            e = ly.prescale_A ? launch_prescale_rows(ly.A, ly.escaled, ctx->c, K, ly.T, ly.d_in, ctx->stream)
                              : launch_prescale_rows(ly.E, ly.escaled, ctx->c, K, ly.T, ly.d_out, ctx->stream);
            GradTask ts = t;
            if (ly.prescale_A) ts.A = ly.escaled;
            else ts.E = ly.escaled;
            ts.T = K;
            StepScalars s1 = sc;
            s1.B = 1;
            if (e == cudaSuccess) e = launch_clipped_sum_tc(ts, ctx->one, ctx->status, s1, nullptr, ctx->stream);
            if (e == cudaSuccess && ly.has_bias) e = launch_bias_sum(t, ctx->c, ctx->status, sc, ctx->stream);
        } else if (ly.grad_kernel == GK_GEMM_TC) {
            const FoldWork fw{ctx->fold_scratch, ctx->fold_counters, next_fold_epoch(ctx)};
            e = launch_clipped_sum_tc(t, ctx->c, ctx->status, sc, &fw, ctx->stream);
            if (e == cudaSuccess && ly.has_bias) e = launch_bias_sum(t, ctx->c, ctx->status, sc, ctx->stream);
        } else {
            e = launch_grad_gemm_cc(t, ctx->c, ctx->status, sc, ctx->stream);
        }
        if (e != cudaSuccess) return cuda_fail(ctx, e, "clipped-sum kernel launch");
    }
    {
        StepScalars s1 = sc;
        s1.B = 1;
        std::vector<bool> done(single.size(), false);
        for (size_t i = 0; i < single.size(); ++i) {
            if (done[i]) continue;
            GradTask group[kMaxSumLayersLaunch];
            int n = 0;
            for (size_t j = i; j < single.size() && n < kMaxSumLayersLaunch; ++j)
                if (!done[j] && single[j].T == single[i].T) {
                    group[n++] = single[j];
                    done[j] = true;
                }
            const cudaError_t e = launch_sum_layers_tc(group, n, ctx->status, s1, ctx->stream);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "clipped-sum kernel launch");
        }
        for (const GradTask& t : single_bias) {
            const cudaError_t e = launch_bias_sum(t, ctx->c, ctx->status, sc, ctx->stream);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "bias-sum kernel launch");
        }
    }
    if (!wsum.empty()) {
        const cudaError_t e = launch_grad_wsum(wsum.data(), (int)wsum.size(), ctx->c, ctx->status, sc, ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "weighted-sum kernel launch");
    }
    ctx->phase = IDLE;
    return DP_OK;
}

}  // namespace

extern "C" {

int dp_version(void) { return kVersion; }

int64_t dp_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int dp_kernel_launch_counts(const char** names, int64_t* counts, int cap) {
    for (int k = 0; k < KL_COUNT && k < cap; ++k) {
        if (names) names[k] = kKernelNames[k];
        if (counts) counts[k] = g_kernel_launches[k].load(std::memory_order_relaxed);
    }
    return KL_COUNT;
}

const char* dp_status_string(dp_status s) {
    switch (s) {
        case DP_OK: return "ok";
        case DP_ERR_INVALID_ARG: return "invalid argument";
        case DP_ERR_SHAPE: return "invalid shape";
        case DP_ERR_STATE: return "call out of order";
        case DP_ERR_NONFINITE: return "non-finite per-example norm";
        case DP_ERR_CUDA: return "CUDA error";
        case DP_ERR_OOM: return "out of device memory";
        case DP_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

int dp_choose_path(int64_t T, int64_t d_in, int64_t d_out) {
    if (T < 1 || d_in < 1 || d_out < 1) return -1;
    return choose(T, d_in, d_out);
}

dp_status dp_create(dp_ctx** out, int device, void* cuda_stream) {
    NvtxRange nvtx_range("dp_create");
    if (!out) return DP_ERR_INVALID_ARG;
    *out = nullptr;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
        cudaGetLastError();
        return DP_ERR_CUDA;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return DP_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return DP_ERR_UNSUPPORTED;
    dp_ctx* ctx = new (std::nothrow) dp_ctx();
    if (!ctx) return DP_ERR_OOM;
    ctx->device = device;
    ctx->stream = static_cast<cudaStream_t>(cuda_stream);
    ctx->sm_count = prop.multiProcessorCount;
    DeviceGuard g(device);
    if (cudaMalloc(reinterpret_cast<void**>(&ctx->status_words), 2 * sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        delete ctx;
        return DP_ERR_OOM;
    }
    if (cudaMemsetAsync(ctx->status_words, 0, 2 * sizeof(unsigned), ctx->stream) != cudaSuccess) {
        cudaFree(ctx->status_words);
        delete ctx;
        return DP_ERR_CUDA;
    }
    ctx->status = ctx->status_words + ctx->slot;
    // the clip factor 1 of a layer whose operand was pre-scaled
    const float one = 1.0f;
    if (cudaMalloc(reinterpret_cast<void**>(&ctx->one), sizeof(float)) != cudaSuccess ||
        cudaMemcpy(ctx->one, &one, sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(ctx->one);
        cudaFree(ctx->status_words);
        delete ctx;
        return DP_ERR_OOM;
    }
    *out = ctx;
    return DP_OK;
}

dp_status dp_destroy(dp_ctx* ctx) {
    NvtxRange nvtx_range("dp_destroy");
    if (!ctx) return DP_OK;
    DeviceGuard g(ctx->device);
    cudaStreamSynchronize(ctx->stream);
    for (Layer& ly : ctx->layers) {
        cudaFree(ly.partial);
        cudaFree(ly.gstore);
        cudaFree(ly.escaled);
    }
    cudaFree(ctx->n2);
    cudaFree(ctx->c);
    cudaFree(ctx->status_words);
    cudaFree(ctx->one);
    cudaFree(ctx->d_slots);
    cudaFree(ctx->fold_scratch);
    cudaFree(ctx->fold_counters);
    delete ctx;
    return DP_OK;
}

dp_status dp_register_layer(dp_ctx* ctx, int64_t d_in, int64_t d_out, int has_bias, dp_dtype dtype,
                            int* layer_id) {
    NvtxRange nvtx_range("dp_register_layer");
    if (!ctx || !layer_id) return fail(ctx, DP_ERR_INVALID_ARG, "NULL argument");
    if (ctx->phase != IDLE) return fail(ctx, DP_ERR_STATE, "layers are registered between steps only");
    if (d_in < 1 || d_out < 1) return fail(ctx, DP_ERR_SHAPE, "d_in and d_out must be >= 1");
    if (dtype != DP_F32 && dtype != DP_BF16) return fail(ctx, DP_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if ((int)ctx->layers.size() >= kMaxLayers) return fail(ctx, DP_ERR_UNSUPPORTED, "at most %d layers", kMaxLayers);
    const unsigned __int128 nc = (unsigned __int128)(uint64_t)d_out * (uint64_t)d_in + (has_bias ? (uint64_t)d_out : 0);
    if (nc + (uint64_t)ctx->P >= ((unsigned __int128)1 << 62)) return fail(ctx, DP_ERR_SHAPE, "too many coordinates");
    Layer ly;
    ly.d_in = d_in;
    ly.d_out = d_out;
    ly.has_bias = has_bias ? 1 : 0;
    ly.dtype = dtype == DP_F32 ? DT_F32 : DT_BF16;
    ly.coord_off = ctx->P;
    ly.ncoords = (int64_t)nc;
    ctx->P += ly.ncoords;
    ctx->layers.push_back(ly);
    *layer_id = (int)ctx->layers.size() - 1;
    return DP_OK;
}

dp_status dp_layer_info(const dp_ctx* ctx, int layer_id, int64_t* coord_offset, int64_t* ncoords) {
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (layer_id < 0 || layer_id >= (int)ctx->layers.size()) return DP_ERR_INVALID_ARG;
    if (coord_offset) *coord_offset = ctx->layers[layer_id].coord_off;
    if (ncoords) *ncoords = ctx->layers[layer_id].ncoords;
    return DP_OK;
}

int64_t dp_num_coords(const dp_ctx* ctx) { return ctx ? ctx->P : 0; }

dp_status dp_begin_step(dp_ctx* ctx, int64_t B) {
    NvtxRange nvtx_range("dp_begin_step");
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (B < 1) return fail(ctx, DP_ERR_SHAPE, "B must be >= 1");
    if (ctx->layers.empty()) return fail(ctx, DP_ERR_STATE, "no layer registered");
    DeviceGuard g(ctx->device);
    dp_status st = grow(ctx, &ctx->n2, &ctx->bcap, (size_t)B);
    if (st != DP_OK) return st;
    st = grow(ctx, &ctx->c, &ctx->ccap, (size_t)B);
    if (st != DP_OK) return st;
    // the step takes the other status word; the previous step's clip kernel
    // zeroed it, otherwise it is cleared here
    const int next = ctx->slot ^ 1;
    if (!ctx->clean[next]) {
        const cudaError_t e = cudaMemsetAsync(ctx->status_words + next, 0, sizeof(unsigned), ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemsetAsync");
    }
    ctx->clean[next] = false;
    ctx->slot = next;
    ctx->status = ctx->status_words + next;
    for (Layer& ly : ctx->layers) {
        ly.accumulated = false;
        ly.A = ly.E = nullptr;
        ly.T = 0;
    }
    ctx->B = B;
    ctx->L = (double)B;
    ctx->t1_fused = false;
    ctx->phase = OPEN;
    ctx->err.clear();
    return DP_OK;
}

dp_status dp_set_normalizer(dp_ctx* ctx, double L) {
    NvtxRange nvtx_range("dp_set_normalizer");
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (ctx->phase == IDLE) return fail(ctx, DP_ERR_STATE, "dp_set_normalizer needs an open step");
    if (!std::isfinite(L) || L <= 0.0 || !std::isfinite((float)L))
        return fail(ctx, DP_ERR_INVALID_ARG, "normalizer L must be finite and > 0");
    ctx->L = L;
    return DP_OK;
}

dp_status dp_norm_accumulate(dp_ctx* ctx, int layer_id, const void* A, const void* E, int64_t T,
                             float* sqnorm_out) {
    NvtxRange nvtx_range("dp_norm_accumulate");
    if (!ctx) return DP_ERR_INVALID_ARG;
    dp_status st = check_accumulate(ctx, layer_id, A, E, T);
    if (st != DP_OK) return st;
    if (sqnorm_out && (reinterpret_cast<uintptr_t>(sqnorm_out) & 3u))
        return fail(ctx, DP_ERR_INVALID_ARG, "sqnorm_out must be 4-byte aligned");
    DeviceGuard g(ctx->device);
    Layer plan;
    st = prepare(ctx, layer_id, A, E, T, plan);
    if (st != DP_OK) return st;
    st = launch_norm(ctx, plan);
    if (st != DP_OK) return st;
    return finish(ctx, layer_id, plan, sqnorm_out);
}

dp_status dp_norm_accumulate_batch(dp_ctx* ctx, int n, const int* layer_ids, const void* const* A,
                                   const void* const* E, const int64_t* T, float* const* sqnorm_out) {
    NvtxRange nvtx_range("dp_norm_accumulate_batch");
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (n < 0 || (n > 0 && (!layer_ids || !A || !E || !T))) return fail(ctx, DP_ERR_INVALID_ARG, "bad batch arrays");
    for (int i = 0; i < n; ++i) {
        dp_status st = check_accumulate(ctx, layer_ids[i], A[i], E[i], T[i]);
        if (st != DP_OK) return st;
        for (int j = 0; j < i; ++j)
            if (layer_ids[j] == layer_ids[i])
                return fail(ctx, DP_ERR_STATE, "layer %d appears twice in one batch", layer_ids[i]);
        if (sqnorm_out && sqnorm_out[i] && (reinterpret_cast<uintptr_t>(sqnorm_out[i]) & 3u))
            return fail(ctx, DP_ERR_INVALID_ARG, "sqnorm_out[%d] must be 4-byte aligned", i);
    }
    DeviceGuard g(ctx->device);
    std::vector<Layer> plans((size_t)n);
    for (int i = 0; i < n; ++i) {
        dp_status st = prepare(ctx, layer_ids[i], A[i], E[i], T[i], plans[i]);
        if (st != DP_OK) return st;
    }
    // every layer of the step T == 1, no per-layer outputs: the norms run inside
    // the clip call's kernel (nothing is launched here)
    bool fuse = n == (int)ctx->layers.size() && n <= kMaxFusedT1;
    for (int i = 0; i < n && fuse; ++i)
        fuse = plans[i].norm_kernel == NK_T1 && t1_groupable(make_norm_task(plans[i])) &&
               !(sqnorm_out && sqnorm_out[i]);
    if (fuse) {
        ctx->t1_tasks.assign((size_t)n, NormTask{});
        for (int i = 0; i < n; ++i) ctx->t1_tasks[(size_t)layer_ids[i]] = make_norm_task(plans[i]);
        for (int i = 0; i < n; ++i) {
            dp_status st = finish(ctx, layer_ids[i], plans[i], nullptr);
            if (st != DP_OK) return st;
        }
        ctx->t1_fused = true;
        return DP_OK;
    }
    // one grouped launch for every skinny materialized layer, one launch each for the rest
    std::vector<NormTask> skinny, t1;
    for (int i = 0; i < n; ++i) {
        const NormTask t = make_norm_task(plans[i]);
        if (plans[i].norm_kernel == NK_MAT_TC) {
            skinny.push_back(t);
        } else if (plans[i].norm_kernel == NK_T1 && t1_groupable(t)) {
            t1.push_back(t);
        } else {
            dp_status st = launch_norm(ctx, plans[i]);
            if (st != DP_OK) return st;
        }
    }
    if (!t1.empty()) {
        const cudaError_t e = launch_norm_t1_group(t1.data(), (int)t1.size(), ctx->B, ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "grouped norm kernel launch");
    }
    if (!skinny.empty()) {
        const cudaError_t e = launch_mat_skinny_tc(skinny.data(), (int)skinny.size(), ctx->B, ctx->status, ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "grouped norm kernel launch");
    }
    for (int i = 0; i < n; ++i) {
        dp_status st = finish(ctx, layer_ids[i], plans[i], sqnorm_out ? sqnorm_out[i] : nullptr);
        if (st != DP_OK) return st;
    }
    return DP_OK;
}

}  // extern "C"

namespace {

// The clip kernel's parameters besides the slot table: B, C, the next step's
// status word (zeroed by the kernel: every kernel that could write it belongs
// to an earlier, finished step) and the first kMaxPrescale pre-scaled operand
// copies, which the clip kernel writes.
ClipParams clip_params(dp_ctx* ctx, float C) {
    ClipParams p;
    p.B = ctx->B;
    p.C = C;
    p.slots = nullptr;
    p.total_slots = 0;
    p.slots_ready = 0;
    p.status_next = ctx->status_words + (ctx->slot ^ 1);
    p.nscale = 0;
    for (Layer& ly : ctx->layers) {
        ly.scaled_by_clip = ly.grad_kernel == GK_GEMM_TC && ly.prescale && p.nscale < kMaxPrescale;
        if (!ly.scaled_by_clip) continue;
        const int64_t d = ly.prescale_A ? ly.d_in : ly.d_out;
        p.scale[p.nscale++] = PrescaleJob{static_cast<const uint4*>(ly.prescale_A ? ly.A : ly.E),
                                          reinterpret_cast<uint4*>(ly.escaled), ly.T * d / 8};
    }
    return p;
}

// the deferred T == 1 norms, the clip factors and the pre-scaled copies in one launch
dp_status clip_fused_t1(dp_ctx* ctx, float C, float* c_out, float* total_sqnorm_out) {
    const ClipParams p = clip_params(ctx, C);
    T1Group grp;
    grp.n = (int)ctx->t1_tasks.size();
    grp.B = ctx->B;
    // a warp of the fused kernel keeps a pre-scaled row in registers when it
    // has one item (at most eight layers) and every such row is short enough
    grp.keep_x = grp.n <= 8 ? 1 : 0;
    int job = 0;
    for (int i = 0; i < grp.n; ++i) {
        const NormTask& t = ctx->t1_tasks[(size_t)i];
        const Layer& ly = ctx->layers[(size_t)i];
        grp.L[i].A = t.A;
        grp.L[i].E = t.E;
        grp.L[i].d_in = t.d_in;
        grp.L[i].d_out = t.d_out;
        grp.L[i].has_bias = t.has_bias;
        grp.L[i].partial = nullptr;
        grp.L[i].scale_job = ly.scaled_by_clip ? job++ : -1;
        grp.L[i].x_is_a = ly.prescale_A ? 1 : 0;
        if (ly.scaled_by_clip && (ly.prescale_A ? t.d_in : t.d_out) / 8 > 32 * kKeepUnits) grp.keep_x = 0;
    }
    const cudaError_t e =
        launch_norm_clip_t1(p, grp, ctx->n2, ctx->c, total_sqnorm_out, c_out, ctx->status, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "norm and clip kernel launch");
    ctx->clean[ctx->slot ^ 1] = true;
    ctx->C = C;
    ctx->phase = CLIPPED;
    return DP_OK;
}

}  // namespace

extern "C" {

dp_status dp_clip_factors(dp_ctx* ctx, float C, float* c_out, float* total_sqnorm_out) {
    NvtxRange nvtx_range("dp_clip_factors");
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (ctx->phase != OPEN) return fail(ctx, DP_ERR_STATE, "dp_clip_factors needs an open, unclipped step");
    if (!std::isfinite(C) || !(C > 0.0f)) return fail(ctx, DP_ERR_INVALID_ARG, "clip bound C must be finite and > 0");
    if ((reinterpret_cast<uintptr_t>(c_out) & 3u) || (reinterpret_cast<uintptr_t>(total_sqnorm_out) & 3u))
        return fail(ctx, DP_ERR_INVALID_ARG, "c_out and total_sqnorm_out must be 4-byte aligned");
    for (size_t l = 0; l < ctx->layers.size(); ++l)
        if (!ctx->layers[l].accumulated)
            return fail(ctx, DP_ERR_STATE, "layer %zu was not accumulated in this step", l);
    DeviceGuard g(ctx->device);
    if (ctx->t1_fused) return clip_fused_t1(ctx, C, c_out, total_sqnorm_out);
    std::vector<std::pair<const float*, int64_t>> key(ctx->layers.size());
    int64_t total = 0;
    for (size_t l = 0; l < ctx->layers.size(); ++l) {
        key[l] = {ctx->layers[l].partial, (int64_t)ctx->layers[l].nslots};
        total += ctx->layers[l].nslots;
    }
    const bool slots_ready = key == ctx->slots_key;
    if (!slots_ready) {
        // the flat slot table changes only when the layer set or its scratch does
        if (ctx->d_slots_cap < (size_t)total) {
            cudaError_t e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
            cudaFree(ctx->d_slots);
            ctx->d_slots = nullptr;
            ctx->d_slots_cap = 0;
            e = cudaMalloc(reinterpret_cast<void**>(&ctx->d_slots), (size_t)total * sizeof(SlotRef));
            if (e != cudaSuccess) return fail(ctx, DP_ERR_OOM, "cudaMalloc of the slot table failed");
            ctx->d_slots_cap = (size_t)total;
        }
        // an upload from pageable memory has been staged when the call returns,
        // so h_slots can be rebuilt while an earlier upload is still in flight
        ctx->h_slots.clear();
        for (const auto& k : key)
            for (int64_t j = 0; j < k.second; ++j) ctx->h_slots.push_back(SlotRef{k.first + j, k.second});
        ctx->slots_key = key;
        const cudaError_t e = cudaMemcpyAsync(ctx->d_slots, ctx->h_slots.data(), (size_t)total * sizeof(SlotRef),
                                              cudaMemcpyHostToDevice, ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "slot table upload");
    }
    ClipParams p = clip_params(ctx, C);
    p.slots = ctx->d_slots;
    p.total_slots = total;
    p.slots_ready = slots_ready ? 1 : 0;
    const cudaError_t e = launch_clip(p, ctx->n2, ctx->c, total_sqnorm_out, c_out, ctx->status, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "clip kernel launch");
    ctx->clean[ctx->slot ^ 1] = true;
    ctx->C = C;
    ctx->phase = CLIPPED;
    return DP_OK;
}


dp_status dp_clipped_noisy_grad(dp_ctx* ctx, float sigma, uint64_t seed, uint64_t step, float* const* G) {
    NvtxRange nvtx_range("dp_clipped_noisy_grad");
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (!std::isfinite(sigma) || sigma < 0.0f) return fail(ctx, DP_ERR_INVALID_ARG, "sigma must be finite and >= 0");
    return clipped_grad(ctx, sigma, seed, step, G, (float)ctx->L, "dp_clipped_noisy_grad");
}

dp_status dp_clipped_sum(dp_ctx* ctx, float* const* S) {
    NvtxRange nvtx_range("dp_clipped_sum");
    if (!ctx) return DP_ERR_INVALID_ARG;
    return clipped_grad(ctx, 0.0f, 0, 0, S, 1.0f, "dp_clipped_sum");
}

dp_status dp_noise_shard(const float* S, float* G, uint64_t k0, int64_t n, float sigma, float C, double L,
                         uint64_t seed, uint64_t step, void* stream) {
    NvtxRange nvtx_range("dp_noise_shard");
    if (n < 0) return DP_ERR_SHAPE;
    if (k0 + (uint64_t)n < k0) return DP_ERR_SHAPE;
    if (!std::isfinite(sigma) || sigma < 0.0f) return DP_ERR_INVALID_ARG;
    if (!std::isfinite(C) || !(C > 0.0f)) return DP_ERR_INVALID_ARG;
    if (!std::isfinite(L) || L <= 0.0 || !std::isfinite((float)L) || !((float)L > 0.0f)) return DP_ERR_INVALID_ARG;
    if (n == 0) return DP_OK;
    if (!S || !G || (reinterpret_cast<uintptr_t>(S) & 3u) || (reinterpret_cast<uintptr_t>(G) & 3u))
        return DP_ERR_INVALID_ARG;
    const cudaError_t e =
        launch_noise_shard(S, G, k0, n, sigma * C, (float)L, seed, step, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}

dp_status dp_step_status(dp_ctx* ctx) {
    NvtxRange nvtx_range("dp_step_status");
    if (!ctx) return DP_ERR_INVALID_ARG;
    DeviceGuard g(ctx->device);
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, ctx->status, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
    if (word & 1u) return fail(ctx, DP_ERR_NONFINITE, "a per-example gradient norm was not finite");
    if (word) return fail(ctx, DP_ERR_CUDA, "a device-side wait timed out; the step's outputs were not written");
    return DP_OK;
}

dp_status dp_check_wait_timeout(dp_ctx* ctx, uint32_t limit_ms) {
    NvtxRange nvtx_range("dp_check_wait_timeout");
    if (!ctx) return DP_ERR_INVALID_ARG;
    if (ctx->phase == IDLE) return fail(ctx, DP_ERR_STATE, "dp_check_wait_timeout needs an open step");
    if (limit_ms < 1 || limit_ms > 2000) return fail(ctx, DP_ERR_INVALID_ARG, "limit_ms must be in 1..2000");
    DeviceGuard g(ctx->device);
    const cudaError_t e = launch_wait_expiry(ctx->status, (uint64_t)limit_ms * 1000000ull, ctx->stream);
    return e == cudaSuccess ? DP_OK : cuda_fail(ctx, e, "wait check launch");
}

const char* dp_last_error(const dp_ctx* ctx) { return ctx ? ctx->err.c_str() : ""; }

dp_status dp_box_muller(const uint32_t* words, int64_t npairs, float* z_out, void* stream) {
    NvtxRange nvtx_range("dp_box_muller");
    if (npairs < 0) return DP_ERR_SHAPE;
    if (npairs == 0) return DP_OK;
    if (!words || !z_out || (reinterpret_cast<uintptr_t>(words) & 7u) || (reinterpret_cast<uintptr_t>(z_out) & 7u))
        return DP_ERR_INVALID_ARG;
    const cudaError_t e = launch_box_muller(words, npairs, z_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}

dp_status dp_philox_normals(uint64_t seed, uint64_t step, uint64_t k0, int64_t n, uint32_t* raw_out,
                            float* z_out, void* stream) {
    NvtxRange nvtx_range("dp_philox_normals");
    if (n < 0) return DP_ERR_SHAPE;
    if (n == 0) return DP_OK;
    if ((raw_out && (reinterpret_cast<uintptr_t>(raw_out) & 3u)) || (z_out && (reinterpret_cast<uintptr_t>(z_out) & 3u)))
        return DP_ERR_INVALID_ARG;
    if (k0 + (uint64_t)n < k0) return DP_ERR_SHAPE;
    const cudaError_t e = launch_philox_normals(seed, step, k0, n, raw_out, z_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DP_OK : DP_ERR_CUDA;
}

}  // extern "C"
