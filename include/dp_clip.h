/*
 * dp_clip.h -- C ABI of the GB300 (sm_103a) DP-SGD private-gradient library.
 *
 * One DP-SGD step over the trainable linear layers of a model, for a batch of
 * B records, as the pages describe it:
 *   per-example gradient norms -> clip factors -> clipped sum -> Gaussian
 *   noise N(0, sigma^2 C^2 I) added once -> divide by the normalizer L.
 * ("Privacy-Preserving Machine Learning", section "Differentially private
 * stochastic gradient descent", phases 2-5; "Differential Privacy: DP-SGD,
 * Privacy Budgets, and LLMs", "Step 1: Per-example gradient clipping" and
 * "Step 2: Gaussian noise addition"; "Differential Privacy in Fine-Tuning
 * (DP-SGD)", "Per-Sample Gradient Clipping" and "Calibrated Gaussian Noise
 * Addition"; "Sensitivity Inflation from Cross-Record Precision Routing in
 * Private Quantized Fine-Tuning", section 2, Eq. 2 and Eq. 3.)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - A linear layer y = x W^T (+ b) has W in R^{d_out x d_in}.  For record i
 *   the caller supplies its activations A_i [T, d_in] and output errors
 *   E_i = dLoss/dy [T, d_out]; the per-example weight gradient is
 *   g_i = E_i^T A_i [d_out, d_in] and the bias gradient sum_t E_i[t, :].
 * - A and E are row-major, contiguous [B, T, d_in] / [B, T, d_out] device
 *   arrays of the layer's dtype, 16-byte aligned.  They are BORROWED: the
 *   caller keeps them alive and unmodified from dp_norm_accumulate until the
 *   work of dp_clipped_noisy_grad has completed on the context's stream
 *   (the clipped sum may re-read them).
 * - Gradient layout: per layer, the weight gradient [d_out][d_in] row-major
 *   (the layout of W), then the bias [d_out].  Layers are concatenated in
 *   registration order; noise coordinate k = layer offset + row * d_in + col
 *   (weights) or layer offset + d_out * d_in + row (bias).
 * - Every call is asynchronous on the context's CUDA stream except
 *   dp_step_status.  Argument errors are detected on the host before any
 *   launch and leave the context unchanged.  One context is driven by one
 *   host thread.
 * - Device buffers owned by the library (norm partials, clip factors, stored
 *   per-example gradients, a status word) belong to the context and are
 *   released by dp_destroy.  The library never frees caller memory.
 */
#ifndef DP_CLIP_H
#define DP_CLIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dp_ctx dp_ctx;

typedef enum dp_status {
    DP_OK = 0,
    DP_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, non-finite or out-of-range scalar  */
    DP_ERR_SHAPE = 2,        /* a size is zero/negative where forbidden, or overflows        */
    DP_ERR_STATE = 3,        /* call out of order (see each entry point)                     */
    DP_ERR_NONFINITE = 4,    /* a per-example norm was NaN/Inf; gradients were not written   */
    DP_ERR_CUDA = 5,         /* a CUDA runtime call failed; dp_last_error has the message    */
    DP_ERR_OOM = 6,          /* device allocation of context scratch failed                   */
    DP_ERR_UNSUPPORTED = 7   /* valid request this build cannot serve (e.g. wrong GPU arch)  */
} dp_status;

typedef enum dp_dtype { DP_F32 = 0, DP_BF16 = 1 } dp_dtype;

/* Norm path of a layer, from dp_choose_path. */
enum { DP_PATH_GHOST = 0, DP_PATH_MATERIALIZE = 1 };

/* Library version, major * 10000 + minor * 100 + patch. */
int dp_version(void);

/*
 * dp_kernel_launches -- number of CUDA kernels this library has launched in
 * the process so far (all contexts, all devices).  Host-side counter, for
 * instrumentation; it never synchronizes.
 */
int64_t dp_kernel_launches(void);

/*
 * dp_kernel_launch_counts -- the same counter split by kernel: for each
 * kernel kind k < min(cap, K), names[k] receives its kernel's name (a static
 * string owned by the library) and counts[k] the number of its launches so
 * far; either array may be NULL.  Returns K, the number of kernel kinds.
 * Host-side counters, for the release record of a run; never synchronizes.
 */
int dp_kernel_launch_counts(const char** names, int64_t* counts, int cap);

/* Static description of a status code (never NULL). */
const char* dp_status_string(dp_status s);

/*
 * dp_create -- make a context bound to CUDA device `device` and the caller's
 * stream `cuda_stream` (a cudaStream_t; NULL means the legacy default stream).
 * The stream is borrowed, not destroyed.  Fails with DP_ERR_UNSUPPORTED when
 * the device is not compute capability 10.3 (the library carries sm_103a code
 * only) and DP_ERR_CUDA when the device cannot be used.  *out receives the
 * context, or NULL on failure.
 */
dp_status dp_create(dp_ctx** out, int device, void* cuda_stream);

/* dp_destroy -- synchronize the stream, free all context scratch, free ctx.  NULL is a no-op. */
dp_status dp_destroy(dp_ctx* ctx);

/*
 * dp_register_layer -- declare one trainable linear layer W in R^{d_out x d_in}
 * (with a bias of d_out entries when has_bias != 0) whose A and E arrays have
 * element type `dtype`.  Layers are numbered 0, 1, ... in call order, which is
 * also their order in the flattened gradient.  Allowed only while no step is
 * open (before dp_begin_step, or after dp_clipped_noisy_grad): DP_ERR_STATE
 * otherwise.  d_in, d_out >= 1 (DP_ERR_SHAPE).
 */
dp_status dp_register_layer(dp_ctx* ctx, int64_t d_in, int64_t d_out, int has_bias,
                            dp_dtype dtype, int* layer_id);

/* dp_layer_info -- first noise coordinate and coordinate count of a layer (either may be NULL). */
dp_status dp_layer_info(const dp_ctx* ctx, int layer_id, int64_t* coord_offset, int64_t* ncoords);

/* dp_num_coords -- total coordinate count P over all registered layers (0 for NULL ctx). */
int64_t dp_num_coords(const dp_ctx* ctx);

/*
 * dp_choose_path -- the ghost / materialize decision for one layer:
 * DP_PATH_GHOST when T*T < d_in*d_out (exact integer comparison, no overflow),
 * else DP_PATH_MATERIALIZE (equality materializes).  Ghost clipping gets each
 * record's norm without forming its full gradient ("Privacy-Preserving Machine
 * Learning", phase 2; "Differential Privacy: DP-SGD, Privacy Budgets, and LLMs",
 * section on computational cost); the rule itself is this library's contract.
 * Returns -1 when an argument is < 1.
 */
int dp_choose_path(int64_t T, int64_t d_in, int64_t d_out);

/*
 * dp_begin_step -- open a step for a batch of B >= 1 records.  Clears the
 * per-step record of which layers were accumulated, resets the device status
 * word and sets the normalizer L to B.  Grows context scratch when B grew
 * (this synchronizes the stream; it happens only when B or a layer's work
 * exceeds every earlier step).  Calling it while a step is open abandons
 * that step: nothing of it is released.  DP_ERR_STATE when no layer is
 * registered.
 */
dp_status dp_begin_step(dp_ctx* ctx, int64_t B);

/*
 * dp_set_normalizer -- use a fixed public normalizer L (finite, > 0) instead of
 * B for this step ("Privacy-Preserving Machine Learning", phase 5 divides by a
 * fixed public L; "Differential Privacy: DP-SGD, Privacy Budgets, and LLMs",
 * Step 2, divides by the batch size B, the default).  Needs an open step.
 */
dp_status dp_set_normalizer(dp_ctx* ctx, double L);

/*
 * dp_norm_accumulate -- per-example squared gradient norms of one layer.
 * A: [B, T, d_in], E: [B, T, d_out] (device, layer dtype, 16-byte aligned,
 * borrowed; see above).  The path is dp_choose_path(T, d_in, d_out):
 *   ghost:        n2_i = <A_i A_i^T, E_i E_i^T> (+ 1^T E_i E_i^T 1 for a bias),
 *                 for T = 1 the closed form ||a_i||^2 ||e_i||^2 (+ ||e_i||^2);
 *   materialize:  n2_i = ||E_i^T A_i||_F^2 (+ ||sum_t E_i[t]||^2), and the
 *                 per-example gradients are kept in context memory for the sum.
 * If sqnorm_out is not NULL it receives this layer's n2 (device float [B], 4-byte
 * aligned: DP_ERR_INVALID_ARG otherwise).
 * The per-record result depends only on that record's rows and the shapes:
 * it is bitwise identical whatever B or the other records are (record
 * isolation: "Sensitivity Inflation ...", Proposition 2).
 * Errors: DP_ERR_STATE without an open step, after dp_clip_factors, or when
 * the layer was already accumulated in this step (the noise must cover each
 * gradient exactly once: "Differential Privacy: DP-SGD, Privacy Budgets, and
 * LLMs", implementation failures); DP_ERR_SHAPE for T < 1;
 * DP_ERR_INVALID_ARG for a bad id or pointer.
 */
dp_status dp_norm_accumulate(dp_ctx* ctx, int layer_id, const void* A, const void* E,
                             int64_t T, float* sqnorm_out);

/*
 * dp_norm_accumulate_batch -- the same for n layers at once, with one grouped
 * launch per kernel kind instead of one launch per layer.  Arrays are host
 * arrays of length n; sqnorm_out may be NULL (or hold NULL entries).  All
 * arguments are validated before anything is launched.
 * When the call holds every registered layer, every one of them takes the
 * T = 1 closed form in bf16 with rows of whole 16-byte vectors, there are at
 * most 32 of them and no sqnorm_out entry is given, nothing is launched here:
 * dp_clip_factors computes these norms, the clip factors and the pre-scaled
 * operands in one kernel, with bitwise the results of the separate launches.
 * A and E are borrowed until dp_clipped_noisy_grad in either case.
 */
dp_status dp_norm_accumulate_batch(dp_ctx* ctx, int n, const int* layer_ids,
                                   const void* const* A, const void* const* E,
                                   const int64_t* T, float* const* sqnorm_out);

/*
 * dp_clip_factors -- total squared norm n2_i = sum over layers (registration
 * order) and clip factor c_i = min(1, C / sqrt(n2_i)), with c_i = 1 for a zero
 * gradient ("Privacy-Preserving Machine Learning", phase 3; "Differential
 * Privacy in Fine-Tuning (DP-SGD)", g / max(1, ||g|| / C)).  c_i is C / n_i
 * rounded toward zero, so that c_i * n_i <= C in float arithmetic.
 * C must be finite and > 0 (DP_ERR_INVALID_ARG).  Every registered layer must
 * have been accumulated in this step (DP_ERR_STATE otherwise: a layer left out
 * would be released without noise).  c_out / total_sqnorm_out, if not NULL,
 * receive c and n2 (device float [B], 4-byte aligned: DP_ERR_INVALID_ARG
 * otherwise).  A non-finite n2_i sets the device
 * status word; dp_clipped_noisy_grad then writes nothing and dp_step_status
 * reports DP_ERR_NONFINITE.
 */
dp_status dp_clip_factors(dp_ctx* ctx, float C, float* c_out, float* total_sqnorm_out);

/*
 * dp_clipped_noisy_grad -- for every registered layer write
 *   G = ( sum_i c_i g_i + sigma * C * z ) / L          (float32)
 * into G[layer] (device, 16-byte aligned, d_out*d_in (+ d_out) floats in the
 * layout above).  z_k is the standard normal of coordinate k drawn from
 * Philox4x32-10 (Salmon et al., SC'11) with key = (seed lo, seed hi), counter
 * = (j lo, j hi, step lo, step hi), j = k / 4, and Box-Muller on the word
 * pairs (x0,x1) -> z[4j], z[4j+1], (x2,x3) -> z[4j+2], z[4j+3], with
 * u1 = ((x >> 8) + 1) 2^-24, u2 = (x >> 8) 2^-24, r = sqrt(-2 ln u1),
 * z = (r cos 2 pi u2, r sin 2 pi u2).  Noise is added once per call, to every
 * coordinate ("Privacy-Preserving Machine Learning", phase 4; "Differential
 * Privacy: DP-SGD, Privacy Budgets, and LLMs", implementation failures).
 * sigma must be finite and >= 0.  DP_ERR_STATE unless dp_clip_factors ran in
 * this step.  Closes the step.  G is written only when no non-finite norm
 * was seen.
 */
dp_status dp_clipped_noisy_grad(dp_ctx* ctx, float sigma, uint64_t seed, uint64_t step,
                                float* const* G);

/*
 * dp_clipped_sum -- the gradient phase without noise and without the
 * normalizer: S = sum_i c_i g_i (+ the bias sum) for every registered layer,
 * written to S[layer] in the layout of dp_clipped_noisy_grad (device,
 * 16-byte aligned).  It is the partial sum one rank contributes when the
 * records of a batch are split over several GPUs: the ranks add their
 * partial sums, and the noise is then drawn once on the total by
 * dp_noise_shard, keyed by the global coordinate, so each coordinate gets
 * exactly one draw whatever the number of ranks ("Privacy-Preserving Machine
 * Learning", phases 4-5: noise added once to the clipped sum, then the
 * division; "Sensitivity Inflation ...", section 4.1, Proposition 2: every
 * record's clipped contribution depends on that record only, so the sum over
 * ranks is the batch's sum).  Same state rules and errors as
 * dp_clipped_noisy_grad, which it replaces in a step: it closes the step.
 */
dp_status dp_clipped_sum(dp_ctx* ctx, float* const* S);

/*
 * dp_noise_shard -- noise and normalizer on a contiguous range of global
 * coordinates: G[j] = (S[j] + sigma * C * z_{k0 + j}) / L for 0 <= j < n,
 * with z the coordinate's standard normal of the (seed, step) stream exactly
 * as dp_clipped_noisy_grad draws it, evaluated in float (sigma * C rounded to
 * float first, L rounded to float).  S and G: device float [n], 4-byte
 * aligned (16-byte alignment with k0 % 4 == 0 takes vector loads), G may
 * equal S; caller-owned.  sigma finite and >= 0, C finite and > 0, L finite
 * and > 0 (DP_ERR_INVALID_ARG otherwise); n >= 0 and k0 + n must not wrap
 * (DP_ERR_SHAPE).  Launches on `stream` (NULL = legacy default);
 * DP_ERR_CUDA for a launch failure.
 */
dp_status dp_noise_shard(const float* S, float* G, uint64_t k0, int64_t n, float sigma, float C, double L,
                         uint64_t seed, uint64_t step, void* stream);

/*
 * dp_step_status -- synchronize the context's stream and return the deferred
 * device-side result of the step: DP_OK, DP_ERR_NONFINITE, or DP_ERR_CUDA for
 * an asynchronous CUDA error or a device-side wait that gave up (a kernel
 * waits at most 2 s for its own copies and MMAs; the step's G is then not
 * written).
 */
dp_status dp_step_status(dp_ctx* ctx);

/* dp_last_error -- message of the most recent failure on this context ("" if none; never NULL). */
const char* dp_last_error(const dp_ctx* ctx);

/*
 * dp_pack_groups -- lay out records grouped by user for user-level clipping
 * ("Privacy-Preserving Machine Learning", section "Differentially private
 * stochastic gradient descent", the user-level construction: records are
 * grouped, a vector is built per user and that vector is clipped).  A user's
 * vector is the sum of its records' gradients, sum_i E_i^T A_i = E_u^T A_u
 * with A_u, E_u the user's records stacked along T, so a user of k records is
 * one record of length k*T for every other call of this library.
 *
 * src: device [B, T, d] row-major (dtype DP_F32 or DP_BF16), the records of
 * user u being src records group_starts[u] .. group_starts[u+1]-1;
 * group_starts: device int64 [U+1], non-decreasing, group_starts[U] <= B;
 * dst: device [U, kmax, T, d] (= [U, kmax*T, d]), written in full: slot s of
 * user u is record group_starts[u] + s when that is below group_starts[u+1],
 * else zeros (a zero record adds nothing to a norm or a sum).  kmax must be at
 * least the largest group; records beyond it are dropped.  Source indices
 * outside [0, B) read as zeros.  Launches on `stream` (NULL = legacy default);
 * src, dst and group_starts are caller-owned.  DP_ERR_INVALID_ARG for NULL
 * pointers or an unknown dtype, DP_ERR_SHAPE for negative sizes or T, d < 1,
 * DP_ERR_CUDA for a launch failure.
 */
dp_status dp_pack_groups(const void* src, void* dst, int64_t B, int64_t T, int64_t d, int dtype,
                         const int64_t* group_starts, int64_t U, int64_t kmax, void* stream);

/*
 * Record-owned LLM.int8 forward of a frozen layer ("Sensitivity Inflation
 * from Cross-Record Precision Routing in Private Quantized Fine-Tuning",
 * section 4.2, Eq. 6 and Algorithm 1; Appendix A).  A producer of the
 * activations a private adapter sees, kept record-isolated: a row's output
 * depends only on its own record's rows.
 *
 * dp_int8_quantize_weight -- W: device half [N, K] row-major (caller-owned).
 * Writes Wq (device int8 [N, K]) = rint(127 W / sW_n), sW (device float [N])
 * = max_j |W_nj|, What (device half [N, K]) = half(Wq sW_n / 127); a zero row
 * gives zeros.  DP_ERR_INVALID_ARG for NULL pointers, DP_ERR_SHAPE for N or
 * K < 1.
 *
 * dp_int8_workspace_bytes -- bytes of the device workspace dp_int8_forward
 * needs for n rows of K columns in records of rows_per_record rows and N
 * outputs; -1 for invalid sizes (n not a multiple of rows_per_record, n, K,
 * N or rows < 1).
 *
 * dp_int8_forward -- A: device half [n, K] row-major (any 2-byte alignment;
 * rows that are whole 16-byte vectors on 16-byte boundaries are read as
 * such), rows r*rows_per_record .. (r+1)*rows_per_record-1 owned by record r.  With O_r the columns where
 * some row of record r has |A| >= tau (tau > 0), U their union, s_i the
 * largest |A_ij| below tau in row i, and O = O_r of the row's record
 * (record_owned != 0) or U (record_owned == 0, batched LLM.int8):
 *   Q_ij = rint((127 A_ij) / s_i) for j not in O (0 when s_i = 0), else 0;
 *   Y_in = half( ((float(sum_j Q_ij Wq_nj) * s_i) * sW_n) / 16129
 *                + sum over j in O ascending of fma(A_ij, What_nj, .) )
 * written to Y (device half [n, N]).  The integer sum is exact: for K up to
 * 4096 on the bf16 tensor cores (the int8 codes are exact in bf16, and each
 * chunk of 1024 products stays below 2^24 in the fp32 accumulator; the
 * chunks are added in int32), beyond on the CUDA cores; K below 133,000.
 * workspace: device, 256-byte aligned, dp_int8_workspace_bytes bytes,
 * overwritten.  Launches on `stream`.  A wait of the tensor-core kernel that
 * gives up (2 s bound) leaves NaN in the affected outputs.  DP_ERR_INVALID_ARG
 * for NULL pointers, tau <= 0 or a misaligned workspace; DP_ERR_SHAPE for
 * invalid sizes; DP_ERR_CUDA for a launch failure.
 */
dp_status dp_int8_quantize_weight(const void* W, int64_t N, int64_t K, int8_t* Wq, float* sW, void* What,
                                  void* stream);
int64_t dp_int8_workspace_bytes(int64_t n, int64_t K, int64_t N, int64_t rows_per_record);
dp_status dp_int8_forward(const void* A, int64_t n, int64_t K, int64_t rows_per_record, const int8_t* Wq,
                          const float* sW, const void* What, int64_t N, float tau, int record_owned, void* Y,
                          void* workspace, void* stream);

/*
 * dp_philox_normals -- the noise generator on its own, for testing: for
 * coordinates k0 .. k0+n-1 of the (seed, step) stream write z (device float
 * [n], if z_out != NULL) and the raw Philox words of blocks k0/4 ..
 * (k0+n-1)/4 (device uint32 [4 * nblocks], if raw_out != NULL).  Launches on
 * `stream` (cudaStream_t, NULL = legacy default).  n >= 0.
 */
dp_status dp_philox_normals(uint64_t seed, uint64_t step, uint64_t k0, int64_t n,
                            uint32_t* raw_out, float* z_out, void* stream);

/*
 * dp_box_muller -- the Box-Muller map of the noise on its own, for testing:
 * for i < npairs, (z_out[2i], z_out[2i+1]) = (r cos 2 pi u2, r sin 2 pi u2)
 * with u1, u2 and r from words[2i], words[2i+1] exactly as in
 * dp_clipped_noisy_grad.  words: device uint32 [2 * npairs], z_out: device
 * float [2 * npairs], both 8-byte aligned (DP_ERR_INVALID_ARG otherwise).
 * Launches on `stream`.  npairs >= 0 (DP_ERR_SHAPE otherwise).
 */
dp_status dp_box_muller(const uint32_t* words, int64_t npairs, float* z_out, void* stream);

/*
 * dp_check_wait_timeout -- test hook for the failure path of the device-side
 * waits.  Every wait of the tensor-core kernels on their own copies and MMAs
 * is bounded; one that gives up sets the timeout bit of the step's status
 * word, the gradient kernels then write nothing, and dp_step_status reports
 * DP_ERR_CUDA.  This call enqueues, on the context's stream, a one-thread
 * kernel whose wait on a barrier that nothing completes gives up after
 * limit_ms milliseconds (1..2000, DP_ERR_INVALID_ARG otherwise) and takes
 * that path.  Needs an open step (DP_ERR_STATE otherwise); the next step is
 * not affected.
 */
dp_status dp_check_wait_timeout(dp_ctx* ctx, uint32_t limit_ms);

/*
 * dp_layer_sqnorms_static -- per-example squared gradient norms of ONE layer
 * without allocating anything.  The pages have no counterpart of this entry
 * point: it exists for callers that cannot call cudaMalloc -- a process that
 * reserved all device memory for its own pool at start-up, a program whose
 * device memory is owned by another framework's allocator, or a
 * latency-bound loop that cannot afford the device-wide synchronization
 * cudaMalloc / cudaFree may perform.
 *
 * It computes what dp_norm_accumulate writes to sqnorm_out (same kernels,
 * same shape rule, no context): sqnorm_out[i] = ||E_i^T A_i||_F^2
 * (+ ||sum_t E_i[t]||^2 when has_bias).  A [B, T, d_in], E [B, T, d_out]
 * (device, dtype, 16-byte aligned), sqnorm_out device float [B]; work is
 * enqueued on `stream` (cudaStream_t, NULL = legacy default) of the CURRENT
 * device.  The kernels' partial sums go to a fixed file-scope device array
 * of 2^20 floats (4 MiB) that every GPU loading the library keeps until the
 * process exits; a request needing more than 2^20 partial slots
 * (B times the slots per record, which depend on T, d_in and d_out) fails
 * with DP_ERR_SHAPE before anything is launched.  The first call on a
 * device resolves the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  The address is kept per
 * device and resolved again when the device's current context changes (a
 * cudaDeviceReset loads the library's device code anew).  All calls share
 * the one array and it keeps the last call's contents: calls whose work
 * overlaps on the GPU (other streams, other host threads) race and give
 * wrong results; serialize them.  The tensor-core norm kernels wait at most
 * 2 s for their own copies and MMAs; when such a wait gives up, every
 * sqnorm_out[i] of that call is NaN (the call itself has returned DP_OK
 * before the kernels ran), and the next call starts clean.  Returns
 * DP_ERR_INVALID_ARG / DP_ERR_SHAPE for bad arguments, DP_ERR_CUDA when a
 * CUDA call or launch fails.  No cudaMalloc, cudaFree or allocating library
 * routine is called.
 */
dp_status dp_layer_sqnorms_static(const void* A, const void* E, int64_t B, int64_t T, int64_t d_in,
                                  int64_t d_out, int has_bias, dp_dtype dtype, float* sqnorm_out,
                                  void* stream);

/*
 * dp_static_check_wait_timeout -- test hook for the NaN report above:
 * enqueues on `stream`, on the current device, a one-thread kernel whose
 * wait on a barrier that nothing completes gives up after limit_ms
 * milliseconds (1..2000, DP_ERR_INVALID_ARG otherwise) and records the
 * timeout exactly as a norm kernel's wait would.  The next
 * dp_layer_sqnorms_static call on the same stream then writes NaN norms; the
 * one after it is clean.  Allocates nothing.  DP_ERR_CUDA for a launch
 * failure.
 */
dp_status dp_static_check_wait_timeout(uint32_t limit_ms, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DP_CLIP_H */
