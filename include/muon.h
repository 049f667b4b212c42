/*
 * libmuon — the Muon optimizer step on one NVIDIA GB300 GPU (sm_103a).
 *
 * One call, muon_step(), updates every registered 2-D weight matrix:
 *
 *   1. momentum      M <- beta*M + G ; U = G + beta*M (Nesterov) or U = M
 *   2. normalise     X0 = U / (||U||_F + 1e-7), oriented short side first
 *                    (a matrix with rows > cols is processed as U^T)
 *   3. orthogonalise ns_steps quintic Newton-Schulz iterations, three
 *                    products each: A = X X^T, B = b A + c A A, X <- a X + B X
 *   4. update        W <- W - lr * max(1, rows/cols)^0.5 * O, O = X (or X^T)
 *
 * Sources: "Advancing Emerging Optimizers for Accelerated LLM Training"
 * (NVIDIA developer blog, 22 Apr 2026, and its summaries).  Section
 * "Distributed Newton-Schulz": the optimizer needs each layer's whole
 * momentum-buffer matrix; section "Duplicated mode": the iteration runs
 * "usually five" times per update and the weights are then updated with the
 * orthogonalised momentum; section "Distributed mode": three matrix products
 * per iteration; section "SYRK and fused all-reduce": the first two products
 * are symmetric rank-k updates that compute only the upper-triangle tiles
 * (diagonal tiles in full) and write the full, mirrored matrix; section
 * "Blockwise mode": each locally held block is orthogonalised and updated on
 * its own, with no communication; section "Load balancing": matrices differ
 * in cost, so work is balanced by estimated cost rather than round-robin.
 * The momentum form, the normalisation, the orientation rule and the shape
 * scale are not written out on the pages; the library takes the plain
 * readings listed above.
 *
 * Conventions for every entry point
 *   - Return value: MUON_OK (0) or a negative MUON_ERR_* code.  The text of
 *     the last error of a handle is available from muon_last_error().
 *   - All argument checks run before any GPU work is queued, so a call that
 *     returns an error has changed no memory.
 *   - Pointers named "device" are CUDA device addresses on the handle's
 *     device; nothing is copied from or to the host unless stated.
 *   - GPU work is queued on the handle's stream and runs asynchronously;
 *     errors raised on the GPU surface at muon_sync().
 *   - Results are deterministic: the same inputs give bit-identical outputs
 *     from run to run, and a matrix gives the same bits whether it is stepped
 *     alone or together with others.
 *   - A handle is not thread-safe; use one handle per host thread.
 */
#ifndef LIBMUON_MUON_H
#define LIBMUON_MUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

/* error codes */
#define MUON_OK                    0
#define MUON_ERR_INVALID_ARG      -1  /* null pointer, bad size, bad enum   */
#define MUON_ERR_UNSUPPORTED      -2  /* shape or dtype the library rejects */
#define MUON_ERR_NO_WORKSPACE     -3  /* no workspace, or too small         */
#define MUON_ERR_CUDA             -4  /* a CUDA runtime/driver call failed  */
#define MUON_ERR_TIMEOUT          -5  /* a bounded wait on the GPU ran out  */
#define MUON_ERR_STATE            -6  /* call out of order (e.g. no params) */

/* element types */
#define MUON_F32   0
#define MUON_BF16  1

/* orthogonalisation modes */
#define MUON_FULL       0   /* each registered matrix as a whole            */
#define MUON_BLOCKWISE  1   /* nb equal column blocks, each on its own      */
/* Distributed mode ("Advancing Emerging Optimizers for Accelerated LLM
 * Training", section "Distributed mode"): the iteration as a tensor-parallel
 * group of nb ranks runs it, each rank holding an equal contiguous slice of
 * the iterate's long side n.  The first product of every iteration is the
 * sum of the slices' partial products (the all-reduce), added in fp32 in
 * slice order 0, 1, ..., nb-1; the other two products are as in full mode.
 * One GPU computes all slices.  nb must divide every n with n / nb a
 * multiple of 64 (MUON_ERR_UNSUPPORTED otherwise); nb = 1 is full mode. */
#define MUON_DISTRIBUTED 2

typedef struct muon_ctx* muon_handle;

/* One 2-D parameter.  w, g and m are device pointers to row-major matrices
 * of rows x cols elements with leading dimensions ld_w, ld_g, ld_m (in
 * elements, >= cols).  w is updated in place (w_dtype: MUON_BF16 or
 * MUON_F32), g is read only (g_dtype: MUON_BF16 or MUON_F32), m is the fp32
 * momentum buffer, updated in place.  The caller owns all three and keeps
 * them valid while they are registered.  1 <= rows, cols <= 1048576 and
 * min(rows, cols) <= 32768 (the m x m intermediates stay addressable). */
typedef struct {
    void*       w;
    const void* g;
    float*      m;
    int64_t     rows, cols;
    int64_t     ld_w, ld_g, ld_m;
    int32_t     w_dtype, g_dtype;
} muon_param;

/* Creates a handle bound to CUDA device `device` and stream `cuda_stream`
 * (a cudaStream_t; NULL = the legacy default stream).  Allocates no device
 * memory.  *out receives the handle.  device = MUON_HOST_ONLY gives a handle
 * that makes no CUDA call at all: it registers parameters (pointers are not
 * dereferenced) and answers muon_workspace_size / muon_get_plan_info, while
 * muon_step and muon_sync return MUON_ERR_STATE. */
#define MUON_HOST_ONLY (-1)
MUON_API int muon_create(muon_handle* out, int device, void* cuda_stream);

/* Replaces the stream that later calls queue their work on. */
MUON_API int muon_set_stream(muon_handle h, void* cuda_stream);

/* Registers n >= 1 parameters (copied; the array may be freed afterwards),
 * replacing any previous set.  Invalidates the current plan. */
MUON_API int muon_register_params(muon_handle h, int n, const muon_param* params);

/* Workspace the step needs for `mode` / `nb` with the registered set.
 * *min_bytes: enough to run the step one group of matrices at a time
 * (the largest single matrix or block plus the plan's tables);
 * *full_bytes: enough to run every matrix in a single group.  Any size in
 * between works; larger sizes give fewer, larger groups.  In blockwise mode
 * nb must divide every registered cols, in distributed mode every long side
 * (see MUON_DISTRIBUTED); MUON_ERR_UNSUPPORTED otherwise. */
MUON_API int muon_workspace_size(muon_handle h, int mode, int nb, size_t* min_bytes,
                        size_t* full_bytes);

/* Hands the library a caller-owned device buffer of `bytes` bytes (start
 * aligned to 1024 bytes) to hold the plan's tables and all intermediate
 * matrices.  The library never allocates device memory itself.  The buffer
 * must stay valid until replaced or the handle is destroyed. */
MUON_API int muon_set_workspace(muon_handle h, void* dptr, size_t bytes);

/* One Muon step over all registered parameters.
 *   lr, beta, nesterov   learning rate, momentum factor, Nesterov on/off
 *   ns_steps             Newton-Schulz iterations (1..64; 5 is usual)
 *   a, b, c              coefficients of a X + (b A + c A A) X
 *   mode, nb             MUON_FULL (nb ignored), MUON_BLOCKWISE with nb
 *                        column blocks (nb >= 1 dividing every cols), or
 *                        MUON_DISTRIBUTED with nb tensor-parallel slices
 * The first step after registering params, changing the workspace, the mode
 * or nb builds the plan and uploads its tables (host work plus one copy);
 * later steps only queue kernels.  Returns once the work is queued.
 * A step carries no device state from earlier steps beyond W and M, so a
 * step queued while the handle's stream is being captured into a CUDA graph
 * replays correctly; the plan must exist before the capture (run one step
 * outside it first: MUON_ERR_STATE otherwise), and stage profiling must be
 * off during the capture. */
MUON_API int muon_step(muon_handle h, float lr, float beta, int nesterov, int ns_steps,
              float a, float b, float c, int mode, int nb);

/* The same step with the gradients taken from, and the updated weights
 * returned to, host memory.  n must equal the number of registered
 * parameters.  g_host[i] holds parameter i's gradient (rows x cols, row-major,
 * leading dimension cols, element type g_dtype); it is copied into the
 * registered device g before the step.  After the step the updated weight
 * (element type w_dtype) is copied to w_host[i] (rows x cols, leading
 * dimension cols); a NULL w_host[i] skips that copy.  Everything is queued on
 * the handle's stream and the call returns once it is queued: host buffers
 * must stay valid, and unchanged, until muon_sync returns, and should be
 * pinned (page-locked) for the copies to run asynchronously.  The caller
 * owns them.  Errors as muon_step; a failed copy is MUON_ERR_CUDA.
 * The copies overlap the compute: the step runs in groups of whole matrices
 * (about 1/16 of the registered elements each, at least 32 M elements), a
 * group's gradients are copied in on a second stream while earlier groups
 * compute, and its weights go out on a third stream once its update is
 * done; the handle's stream waits for all of them.  The first call builds
 * that grouping (later muon_step calls reuse it; results are the same bits
 * with any grouping). */
MUON_API int muon_step_host(muon_handle h, int n, const void* const* g_host,
                            void* const* w_host, float lr, float beta, int nesterov,
                            int ns_steps, float a, float b, float c, int mode, int nb);

/* Waits for the handle's stream and reports any error raised on the GPU
 * (MUON_ERR_TIMEOUT when a bounded wait ran out, MUON_ERR_CUDA otherwise). */
MUON_API int muon_sync(muon_handle h);

/* Releases the handle (no device memory is owned, none is freed). */
MUON_API int muon_destroy(muon_handle h);

/* Text of the handle's last error ("" if none).  Valid until the next call
 * on the handle.  h may be NULL (returns the last create error). */
MUON_API const char* muon_last_error(muon_handle h);

/* ---- measurement and validation helpers ------------------------------- */

/* Stage timing.  When on, muon_step records CUDA events around each kind of
 * launch on the handle's stream; muon_stage_times() (after muon_sync) fills
 * up to `n` totals in milliseconds for the last step, in the order
 * momentum, norm, normalise, syrk1, syrk2, gemm, update, chain (one launch
 * with every product of the step but the last X update), and the number
 * of launches of each kind into `launches` (may be NULL).  Returns the
 * number of stages written. */
#define MUON_N_STAGES 8
MUON_API int muon_set_profiling(muon_handle h, int on);
MUON_API int muon_stage_times(muon_handle h, float* ms, int* launches, int n);

/* Number of kernel launches the last muon_step queued. */
MUON_API int muon_last_launch_count(muon_handle h);

/* Optional exports written by the update stage of every later step, for
 * parameter i (0 <= i < n): w_f32[i] receives the updated weight in fp32
 * before it is stored in the weight's dtype, o_bf16[i] the orthogonalised
 * update O in bf16; both rows x cols row-major with leading dimension cols,
 * in the weight's orientation.  Entries (or whole arrays) may be NULL.
 * n = 0 turns exports off.  Changing exports rebuilds the plan. */
MUON_API int muon_debug_set_exports(muon_handle h, int n, float* const* w_f32,
                           void* const* o_bf16);

/* Failure-path check of the kernels' bounded waits: launches one block that
 * waits on a barrier nothing arrives at, with a limit of `limit_ms`
 * (1..10000) milliseconds, and reads the device error word `err_word` (a
 * caller-owned device int).  Returns MUON_ERR_TIMEOUT when the wait ran out
 * and reported it as the tensor-core kernels do (the expected outcome); the
 * CUDA context stays usable.  Makes no other change. */
MUON_API int muon_debug_wait_timeout(muon_handle h, int* err_word, int limit_ms);

/* Validation of the chained launch (see muon_get_plan_info: groups of few
 * large matrices run every product of a step in one launch whose tiles wait
 * on per-tile counters; the launch's last CTA zeroes them as it leaves).
 * skew_rounds > 0 makes the second products of later chained launches wait
 * for that many counter rounds more than will ever be completed, so their
 * bounded waits run out and muon_sync reports MUON_ERR_TIMEOUT (a timeout
 * test without a fault; 0 = off).  Applies to later steps of this handle;
 * MUON_ERR_INVALID_ARG for values out of range. */
MUON_API int muon_debug_set_chain_test(muon_handle h, int skew_rounds);

/* Host-only check of the chained launch's schedule for `mode`/`nb`: for every
 * group of the registered matrices (ignoring the size bounds that decide
 * whether a group chains), builds the per-pair tile lists and checks that
 * every tile appears once, that each pair's list is in stage order (first
 * products, second products, X updates: the order that keeps every wait on
 * tiles of earlier stages) and that the pair offsets and last-iteration ends
 * are consistent.  No CUDA call; works on MUON_HOST_ONLY handles.  Returns
 * MUON_OK, or MUON_ERR_STATE with the violated property in
 * muon_last_error. */
MUON_API int muon_debug_check_chain_schedule(muon_handle h, int mode, int nb);

/* Plan statistics for `mode`/`nb`: number of units (matrices or blocks),
 * groups, and tiles of the symmetric-product and GEMM stages. */
typedef struct {
    int64_t units, groups, syrk_tiles, gemm_tiles, ew_tiles;
    /* per Newton-Schulz iteration, all units: useful = upper-triangle
     * symmetric products + the GEMM; executed = what the tiles compute */
    int64_t useful_flops, executed_flops;
    /* groups whose products run as one chained launch per step (every
     * product but the last X update; groups of few large matrices) */
    int64_t chained_groups;
} muon_plan_info;
MUON_API int muon_get_plan_info(muon_handle h, int mode, int nb, muon_plan_info* out);

/* ---- distributed mode across ranks ------------------------------------- */

/* "Advancing Emerging Optimizers for Accelerated LLM Training", section
 * "Distributed mode": the iterate X (m x n, short side first) of one matrix
 * is split along n over the P ranks of a tensor-parallel group, one GPU
 * each.  A rank holds its slice of W, G and M and runs the step in phases;
 * between the phases the caller sums across the group (an all-reduce, e.g.
 * torch.distributed over NCCL).  Per iteration the only exchange is the sum
 * of the partial products X_r X_r^T (the all-reduce after the first matrix
 * product), plus one sum of squares for the norm before the first:
 *
 *   muon_dist_momentum(h, ...)        momentum on the slice; the slice's
 *                                     sum of squares of U -> sumsq
 *   [sum sumsq over the group]
 *   for s = 0 .. ns_steps - 1:
 *     muon_dist_gram(h, ...)          the partial X_r X_r^T -> A (fp32)
 *     [sum A over the group]
 *     muon_dist_update(h, ...)        B' = b A + c A A + a I from the sum,
 *                                     X_r <- B' X_r; on the last iteration
 *                                     W_r <- W_r - lr * scale * O_r
 *
 * The handle must hold exactly one registered parameter, the rank's slice,
 * and must have been configured with muon_dist_configure first; the phases
 * use its workspace (muon_workspace_size with MUON_FULL).  Phases are queued
 * on the handle's stream in the order above; errors as for muon_step, and
 * MUON_ERR_STATE for a phase out of order.  The weight update of the last
 * iteration is folded into the X update as in muon_step. */

/* The slice's place in the whole matrix: transposed = 1 if the whole weight
 * is tall (rows > cols; its iterate is W^T, and the slice is a block of W's
 * rows), 0 otherwise (the slice is a block of W's columns); shape_scale =
 * the whole matrix's max(1, rows / cols) ** 0.5.  The slice's short side must
 * then be the whole matrix's short side: its iterate is m x n_r with
 * m = cols (transposed) or rows.  Invalidates the plan. */
MUON_API int muon_dist_configure(muon_handle h, int transposed, float shape_scale);

/* M <- beta M + G and U on the slice; the iterate slice X_r = bf16(U), not
 * yet normalised.  *sumsq (device memory, one double) receives the slice's
 * sum of U^2, taken per 64 x 64 tile and then over the tiles in a fixed
 * order, so that the sum of all slices' values is ||U||_F^2. */
MUON_API int muon_dist_momentum(muon_handle h, float beta, int nesterov, double* sumsq);

/* Iteration s's partial product A_r = X_r X_r^T of the slice, unscaled fp32,
 * into the m x m row-major device buffer a (leading dimension lda >= m),
 * for the 256 x 256 tiles (ti, tj) with ti <= tj and band_begin <= ti <
 * band_end (256-row blocks; band_end = -1: to the last).  Nothing else of a
 * is written: the caller zeroes it once, so that the tiles below the
 * diagonal stay zero, and may sum the bands as each is queued (the
 * "SYRK and fused all-reduce" exchange of finished upper tiles). */
MUON_API int muon_dist_gram(muon_handle h, float* a, int64_t lda, int band_begin,
                            int band_end);

/* The rest of iteration s from the group's sum of the partial products in
 * a (fp32, upper tiles as written by muon_dist_gram): A = bf16(sum * scale)
 * with scale = 1 / (||U||_F + eps)^2 when first (sumsq_total: device double,
 * the group's sum of the momentum phase's values; ignored otherwise), then
 * B' = b A + c A A + a I and X_r <- B' X_r (times 1 / (||U||_F + eps) when
 * first).  When last, the update O_r = X_r (transposed back) is applied:
 * W_r <- W_r - lr * shape_scale * O_r. */
MUON_API int muon_dist_update(muon_handle h, const float* a, int64_t lda, int first, int last,
                              const double* sumsq_total, float lr, float ca, float cb, float cc);

/* ---- step without a workspace ------------------------------------------ */

/* One Muon step (full mode) on ONE matrix without any workspace: the plan
 * tables and every intermediate (partial sums, the two iterates X, and A, B)
 * live in a fixed 32 MiB array inside the library.  This is for callers who
 * cannot call cudaMalloc or hand over a buffer: a plugin whose host owns all
 * device memory through a pool it does not expose, a process whose caching
 * allocator has already reserved the GPU, or a hot loop that cannot afford
 * cudaMalloc's implicit device synchronisation.  The paper has no
 * counterpart of this entry point; it is a convenience of this library.
 *
 *   param          one matrix as for muon_register_params (device pointers;
 *                  W and M updated in place, G read only)
 *   lr ... c       as for muon_step
 *   cuda_stream    stream for the work (NULL = legacy default stream); the
 *                  CUDA device is the caller's current device
 *   err, err_len   optional buffer that receives a message on error
 *
 * Limits and behaviour:
 *   - The matrix must fit the fixed array: roughly 4 bytes per element of
 *     the matrix plus 4 bytes per element of its m x m square (m = short
 *     side), plus small tables, at most 33554432 bytes in total (a 1024 x
 *     4096 matrix fits, a 2048 x 2048 does not).  Larger matrices are
 *     rejected with MUON_ERR_UNSUPPORTED and a message before any GPU work.
 *   - The array exists once per device that loads this code and is held
 *     until the process exits.  The first call on a device is its set-up:
 *     it resolves the array's address (cudaGetSymbolAddress) with that
 *     device current, so make that first call before any stream capture.
 *     The address is resolved again only if the device's context has been
 *     replaced since (for example after cudaDeviceReset).
 *   - Every call reuses the same array and overwrites what the previous
 *     call left there; calls whose GPU work overlaps (different streams or
 *     threads) race and give wrong results.  Queue them on one stream.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  The work is
 *     queued asynchronously; a bounded GPU wait that runs out makes the
 *     kernels return early, which this entry point cannot report (use the
 *     handle-based muon_step and muon_sync where that report matters). */
MUON_API int muon_step_noalloc(const muon_param* param, float lr, float beta,
                               int nesterov, int ns_steps, float a, float b,
                               float c, void* cuda_stream, char* err,
                               size_t err_len);

#ifdef __cplusplus
}
#endif
#endif /* LIBMUON_MUON_H */
