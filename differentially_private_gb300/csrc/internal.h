// Internal interface between the host runtime (runtime.cu) and the kernel
// translation units.  Nothing here is part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

enum { DT_F32 = 0, DT_BF16 = 1 };

// Largest number of registered layers a context accepts.
constexpr int kMaxLayers = 4096;
// Largest number of layers one grouped launch carries in its parameters.
constexpr int kMaxGroup = 64;
// Largest number of layers one skinny-materialize launch carries (each
// brings two 128-byte TMA descriptors in the kernel parameters).
constexpr int kMaxSkinnyGroup = 48;

// Norm kernels.
enum NormKernel {
    NK_T1 = 0,        // ghost, T == 1: ||a||^2 ||e||^2 (+ ||e||^2)
    NK_GHOST_CC = 1,  // ghost, CUDA-core tiled Gram
    NK_MAT_CC = 2,    // materialize, CUDA-core tiled E^T A
    NK_GHOST_TC = 3,  // ghost, tcgen05 Gram
    NK_MAT_TC = 4,    // materialize, tcgen05 skinny E^T A
};

// Gradient kernels.
enum GradKernel {
    GK_WSUM = 0,      // from stored per-example gradients
    GK_GEMM_CC = 1,   // CUDA-core reweighted E^T diag(c) A
    GK_GEMM_TC = 2,   // tcgen05 reweighted E^T diag(c) A
};

// One layer's per-example norm work for one step.
struct NormTask {
    const void* A;      // [B, T, d_in]
    const void* E;      // [B, T, d_out]
    int64_t T, d_in, d_out;
    int has_bias;
    int dtype;
    float* partial;     // [B][nslots] fp32 partial squared norms
    int nslots;
    float* gstore;      // [B][ncoords] per-example gradients, or nullptr
    const CUtensorMap* maps;  // two pre-encoded TMA descriptors (tensor-core kernels), or nullptr
};

// One layer's gradient work.
struct GradTask {
    const void* A;
    const void* E;
    int64_t T, d_in, d_out;
    int has_bias;
    int dtype;
    const float* gstore;   // stored per-example gradients (GK_WSUM)
    float* G;              // output, d_out*d_in (+ d_out)
    int64_t coord_off;     // first noise coordinate of the layer
    const CUtensorMap* maps;  // pre-encoded TMA descriptors (tc_encode_sum: three), or nullptr
};

struct StepScalars {
    int64_t B;
    float C;
    float sigma;
    float L;
    uint64_t seed;
    uint64_t step;
};

// One flat partial-norm slot of every record: record i's value is
// base[i * stride] (a layer's partials are [B][nslots], so base = the
// layer's partial array + the slot index and stride = nslots).
struct SlotRef {
    const float* base;
    int64_t stride;
};

// One operand the clip kernel copies scaled by c_i, row block by row block:
// record i's rows are units [i * units, (i + 1) * units) of 16 bytes (8 bf16)
// of src, written to the same place of dst.
struct PrescaleJob {
    const uint4* src;
    uint4* dst;
    int64_t units;
};
constexpr int kMaxPrescale = 4;

struct ClipParams {
    int64_t B;
    float C;
    const SlotRef* slots;      // device array: layers in registration order, each layer's slots in order
    int64_t total_slots;
    int slots_ready;           // the table was uploaded before an earlier step (readable before the dependency wait)
    unsigned* status_next;     // status word of the next step, zeroed by the kernel (or nullptr)
    int nscale;                // pre-scaled operand copies made by the clip kernel
    PrescaleJob scale[kMaxPrescale];
};

// Several T == 1 bf16 layers (rows of whole 16-byte vectors) in one launch,
// one warp per record.
struct T1Group {
    int n;
    int64_t B;
    struct {
        const void* A;
        const void* E;
        int64_t d_in, d_out;
        int has_bias;
        float* partial;
        int scale_job;   // fused norm + clip kernel: index of the layer's pre-scale job, or -1
        int x_is_a;      // that job's operand is A (else E)
    } L[kMaxGroup];
    int keep_x;          // fused kernel: every pre-scaled row fits kKeepUnits vectors per lane
};
// 16-byte vectors per lane of a pre-scaled row that the fused kernel keeps in registers
constexpr int kKeepUnits = 4;
// at most this many T == 1 layers take the fused norm + clip kernel (a lane per layer)
constexpr int kMaxFusedT1 = 32;

// one-thread kernel whose bounded wait on a barrier nobody completes gives up
// after limit_ns and sets the timeout bit of *status (waitcheck.cu)
cudaError_t launch_wait_expiry(unsigned* status, uint64_t limit_ns, cudaStream_t s);

// ---- host helpers shared by the tensor-core launchers (runtime.cu)
// cuTensorMapEncodeTiled, fetched once through the runtime (the library does
// not link libcuda directly); nullptr when the driver does not provide it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
// The kernel's dynamic shared-memory limit raised to `bytes` on the current
// device (once per device and kernel; safe from several host threads).
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// ---- every kernel launch of the library is counted here, per kernel
// (dp_kernel_launches, dp_kernel_launch_counts)
enum KernelId {
    KL_NORM_T1, KL_NORM_T1_GROUP, KL_NORM_GHOST_CC, KL_NORM_MAT_CC, KL_LAYER_SQNORM, KL_LAYER_SQNORM_STATUS,
    KL_GHOST_GRAM_TC, KL_MAT_SKINNY_TC, KL_CLIP, KL_NORM_CLIP_T1, KL_GRAD_WSUM, KL_GRAD_GEMM_SMALL, KL_GRAD_GEMM_CC, KL_BIAS_SUM,
    KL_PRESCALE_ROWS, KL_CLIPPED_SUM_FOLD_PAIR_TC, KL_CLIPPED_SUM_TC, KL_SUM_LAYERS_PAIR_TC, KL_NOISE_SHARD,
    KL_BOX_MULLER, KL_PHILOX_NORMALS, KL_PACK_GROUPS, KL_INT8_QUANTIZE_WEIGHT, KL_INT8_ROWSCAN,
    KL_INT8_GEMM, KL_INT8_CODES, KL_INT8_GEMM_TC, KL_WAIT_EXPIRES, KL_COUNT
};
void count_launch(KernelId k);

// ---- NVTX range over the body of a public entry point (header-only NVTX 3:
// a no-op unless a profiler is attached)
struct NvtxRange {
    explicit NvtxRange(const char* name);
    ~NvtxRange();
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---- slot counts (depend on the shapes only, never on B)
int nslots_for(int kernel, int64_t T, int64_t d_in, int64_t d_out);
// norm kernel the runtime picks for these shapes (NormKernel), and its slot count
int plan_norm_kernel(int dtype, int64_t T, int64_t d_in, int64_t d_out, int has_bias, int* nslots);
int nslots_cc(int kernel, int64_t T, int64_t d_in, int64_t d_out);

// ---- launchers; each returns the cudaGetLastError() of its launches
cudaError_t launch_norm_t1(const NormTask& t, int64_t B, cudaStream_t s);
// several bf16 T == 1 layers with 16-byte rows in one launch (same result per record as launch_norm_t1)
bool t1_groupable(const NormTask& t);
cudaError_t launch_norm_t1_group(const NormTask* tasks, int n, int64_t B, cudaStream_t s);
cudaError_t launch_norm_ghost_cc(const NormTask& t, int64_t B, cudaStream_t s);
cudaError_t launch_norm_mat_cc(const NormTask& t, int64_t B, cudaStream_t s);
cudaError_t launch_layer_sqnorm(const float* partial, int nslots, int64_t B, float* out, cudaStream_t s);
// the same, but every output is NaN when *status is not zero (read after the producers ran)
cudaError_t launch_layer_sqnorm_checked(const float* partial, int nslots, int64_t B, float* out,
                                        const unsigned* status, cudaStream_t s);
cudaError_t launch_clip(const ClipParams& p, float* n2, float* c, float* n2_user, float* c_user,
                        unsigned* status, cudaStream_t s);
// every layer of the step T == 1: the layers' norms, the clip factors and the
// pre-scaled copies in one launch, instead of the norm kernel and the clip kernel
cudaError_t launch_norm_clip_t1(const ClipParams& p, const T1Group& g, float* n2, float* c, float* n2_user,
                                float* c_user, unsigned* status, cudaStream_t s);
cudaError_t launch_grad_wsum(const GradTask* tasks, int n, const float* c, const unsigned* status,
                             const StepScalars& sc, cudaStream_t s);
cudaError_t launch_grad_gemm_cc(const GradTask& t, const float* c, const unsigned* status,
                                const StepScalars& sc, cudaStream_t s);
// G[j] = (S[j] + scale z_{k0+j}) / L over a contiguous range of global coordinates
cudaError_t launch_noise_shard(const float* S, float* G, uint64_t k0, int64_t n, float scale, float L,
                               uint64_t seed, uint64_t step, cudaStream_t s);
cudaError_t launch_box_muller(const uint32_t* words, int64_t npairs, float* z, cudaStream_t s);
cudaError_t launch_philox_normals(uint64_t seed, uint64_t step, uint64_t k0, int64_t n,
                                  uint32_t* raw, float* z, cudaStream_t s);
cudaError_t launch_bias_sum(const GradTask& t, const float* c, const unsigned* status,
                            const StepScalars& sc, cudaStream_t s);
// E2 = c[row / T] * E row by row (bf16, d % 8 == 0, 16-byte aligned)
cudaError_t launch_prescale_rows(const void* E, void* E2, const float* c, int64_t K, int64_t T, int64_t d,
                                 cudaStream_t s);

// ---- tcgen05 kernels (tc_gemm.cu)
// Scratch of the tensor-core clipped sum for the tiles of a partial last wave
// that are split into record ranges over the grid.
struct FoldWork {
    float* scratch;                  // fold_scratch_floats(sms) floats
    unsigned long long* counters;    // sms entries; zero when allocated, never reset
    unsigned epoch;                  // different for every launch (never 0)
};
size_t fold_scratch_floats(int sms);
int device_sm_count();
bool tc_sum_supported(int dtype, int64_t d_in, int64_t d_out, int has_bias);
bool tc_skinny_supported(int dtype, int64_t d_in, int64_t d_out, int has_bias);
int nslots_skinny(int64_t d_in, int64_t d_out);
// B > 1 (T % 64 == 0): the per-record fold on CTA pairs, the tiles of a
// partial last wave cut into record ranges when work != nullptr; B == 1: one
// record of T rows with factor c[0], one CTA per tile
cudaError_t launch_clipped_sum_tc(const GradTask& t, const float* c, unsigned* status,
                                  const StepScalars& sc, const FoldWork* work, cudaStream_t s);
// Single-record sums of up to kMaxSumLayersLaunch layers sharing K = T rows
// (tasks[i].T = K; factor 1: their clip factors are in the pre-scaled
// operand) in one persistent launch, whole tiles strided over the CTAs.
constexpr int kMaxSumLayersLaunch = 4;
cudaError_t launch_sum_layers_tc(const GradTask* tasks, int n, unsigned* status, const StepScalars& sc,
                                 cudaStream_t s);
cudaError_t launch_mat_skinny_tc(const NormTask* tasks, int n, int64_t B, unsigned* status, cudaStream_t s);
// TMA descriptors of a layer, encoded once per (pointers, T, B) and cached by the runtime
bool tc_encode_skinny(const NormTask& t, int64_t B, CUtensorMap* maps2);
// maps3: E, A in 256-column tiles, A in 128-column halves (CTA pairs)
bool tc_encode_sum(const GradTask& t, int64_t B, CUtensorMap* maps3);
bool tc_encode_gram(const NormTask& t, int64_t B, CUtensorMap* maps2);

// ---- tcgen05 ghost Gram (tc_gram.cu)
bool tc_gram_supported(int dtype, int64_t T, int64_t d_in, int64_t d_out);
int nslots_gram(int64_t T);
cudaError_t launch_ghost_gram_tc(const NormTask& t, int64_t B, unsigned* status, cudaStream_t s);
