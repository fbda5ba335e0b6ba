/*
 * gbnorm.h -- C ABI of the fused row-wise RMSNorm / LayerNorm library for
 * GB300 (sm_103a): forward and backward over [M, N] row-major tensors.
 *
 * What is computed (per row i of M, over its N contiguous elements):
 *
 *   RMSNorm ("SOTA normalization performance with torch.compile", section
 *   "How Did Torch.compile Catch Quack?"; "Fused RMSNorm", section
 *   "What it is": a square, a mean, an add of eps, a reciprocal square root,
 *   a multiply and another multiply):
 *       rstd_i = 1 / sqrt((1/N) sum_j x_ij^2 + eps)
 *       y_ij   = (x_ij * rstd_i) * gamma_j
 *
 *   LayerNorm (same page and section: subtract the mean, divide by the
 *   standard deviation, scale by gamma, add beta; biased variance):
 *       mean_i = (1/N) sum_j x_ij
 *       rstd_i = 1 / sqrt((1/N) sum_j (x_ij - mean_i)^2 + eps)
 *       y_ij   = ((x_ij - mean_i) * rstd_i) * gamma_j + beta_j
 *
 *   Backward (the outputs dX, dW and dB that the torch.compile page's
 *   backward paragraph names; the formulas are the analytic gradients):
 *       xhat_ij = (x_ij - mean_i) * rstd_i         (mean_i = 0 for RMSNorm)
 *       g_ij    = dy_ij * gamma_j
 *       RMSNorm:   dx_ij = rstd_i * (g_ij - xhat_ij * (1/N) sum_k g_ik xhat_ik)
 *       LayerNorm: dx_ij = rstd_i * (g_ij - (1/N) sum_k g_ik
 *                                         - xhat_ij * (1/N) sum_k g_ik xhat_ik)
 *       dgamma_j = sum_i dy_ij * xhat_ij,     dbeta_j = sum_i dy_ij
 *   dgamma/dbeta are reduced in two stages without atomics, as the "Fused
 *   RMSNorm" page's "What didn't work" and "Next" sections describe: per-block
 *   partial rows into a caller-provided workspace, then a second kernel that
 *   sums the workspace column by column in a fixed order (deterministic).
 *
 * Conventions shared by every entry point:
 *   - Layout: x, y, dy, dx are [M, N] row-major and contiguous (row stride N
 *     elements).  gamma and beta are [N].  mean and rstd are [M] float32.
 *     dgamma and dbeta are [N] float32.  All are DEVICE pointers on the
 *     current CUDA device.
 *   - dtype selects the element type of x, y, dy, dx, gamma and beta; all of
 *     them share it.  Arithmetic is float32 throughout; each output element
 *     is rounded once to dtype, round-to-nearest-even.
 *   - Ownership: the caller allocates and owns every buffer.  The library
 *     never allocates device memory, never frees, and never synchronises.
 *     All work is enqueued on `stream` (NULL = the legacy default stream)
 *     and completes asynchronously.
 *   - Optional parameters: gamma may be NULL in every entry point (gamma_j =
 *     1: RMSNorm or LayerNorm without a scale), beta may be NULL in
 *     layernorm_fwd (beta_j = 0: no bias), and dgamma / dbeta may be NULL in
 *     the backward (that column sum is not produced).  The kernels use the
 *     constants in place of the missing row; nothing is read for it.
 *   - Alignment: with 16-byte-aligned pointers and N * sizeof(dtype) a
 *     multiple of 16, rows move as 128-bit vectors; anything else takes a
 *     correct element-wise path.
 *   - Aliasing: y may equal x exactly (in place) and dx may equal dy exactly;
 *     any other overlap between an output and an input is rejected.
 *   - Shapes: M >= 0 (M == 0 launches nothing in the forward and writes zero
 *     dgamma/dbeta in the backward), 1 <= N <= GBNORM_MAX_N.
 *   - Errors: every function returns a gbnorm_status_t.  Arguments are
 *     checked before anything is enqueued; a rejected call enqueues nothing.
 *     GBNORM_ERR_CUDA reports a failed launch (cudaGetLastError right after
 *     it).  No C++ exception crosses this interface.
 *   - Thread safety: all entry points may be called concurrently from several
 *     host threads; the only shared state is a per-device cache of device
 *     attributes and occupancy filled once.
 */
#ifndef GBNORM_H
#define GBNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA headers. */
typedef struct CUstream_st *gbnorm_stream_t;

typedef enum {
    GBNORM_F32 = 0,
    GBNORM_F16 = 1,
    GBNORM_BF16 = 2
} gbnorm_dtype_t;

typedef enum {
    GBNORM_OK = 0,
    GBNORM_ERR_INVALID_ARG = 1, /* required pointer null, bad shape or dtype, overlapping buffers, bad eps */
    GBNORM_ERR_UNSUPPORTED = 2, /* a valid request this build cannot serve (e.g. no sm_103a device) */
    GBNORM_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than norm_bwd_workspace_size */
    GBNORM_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} gbnorm_status_t;

/* Largest row length N accepted by every entry point. */
#define GBNORM_MAX_N ((int64_t)1 << 24)

/*
 * RMSNorm forward.
 *   x      [M, N] dtype, read only.
 *   gamma  [N] dtype, read only; may be NULL (gamma = 1).
 *   y      [M, N] dtype, written (may equal x).
 *   rstd   [M] float32, written; may be NULL (nothing stored, e.g. inference).
 *   eps    added to the mean square under the root; finite and >= 0.
 */
int rmsnorm_fwd(const void *x, const void *gamma, void *y, float *rstd, int64_t M, int64_t N,
                int dtype, float eps, gbnorm_stream_t stream);

/*
 * LayerNorm forward.
 *   x, gamma, y, rstd as for rmsnorm_fwd; beta [N] dtype, read only, may be
 *   NULL (beta = 0).
 *   mean   [M] float32, written; may be NULL.  rstd may be NULL.
 *   eps    added to the biased variance under the root; finite and >= 0.
 */
int layernorm_fwd(const void *x, const void *gamma, const void *beta, void *y, float *mean,
                  float *rstd, int64_t M, int64_t N, int dtype, float eps,
                  gbnorm_stream_t stream);

/*
 * Bytes of device workspace the backward of this shape needs on the current
 * device (the per-block partial rows of dgamma, and of dbeta for LayerNorm).
 * Returns 0 if the arguments are invalid or no CUDA device is usable.
 */
size_t norm_bwd_workspace_size(int is_layernorm, int64_t M, int64_t N, int dtype);

/*
 * RMSNorm backward.
 *   dy, x  [M, N] dtype, read only.   gamma [N] dtype, read only, may be
 *          NULL (gamma = 1).
 *   rstd   [M] float32 as saved by rmsnorm_fwd, read only.
 *   dx     [M, N] dtype, written (may equal dy).
 *   dgamma [N] float32, written (overwritten, not accumulated); may be NULL
 *          (not produced).
 *   workspace / workspace_bytes: device scratch of at least
 *          norm_bwd_workspace_size(0, M, N, dtype) bytes, 16-byte aligned;
 *          its contents on entry are ignored and on exit are unspecified.
 *          It must not be used by another call that may run concurrently.
 */
int rmsnorm_bwd(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx,
                float *dgamma, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                int dtype, gbnorm_stream_t stream);

/*
 * LayerNorm backward.
 *   as rmsnorm_bwd, plus mean [M] float32 as saved by layernorm_fwd (read
 *   only) and dbeta [N] float32 (written; may be NULL).  Workspace of at least
 *   norm_bwd_workspace_size(1, M, N, dtype) bytes.
 */
int layernorm_bwd(const void *dy, const void *x, const void *gamma, const float *mean,
                  const float *rstd, void *dx, float *dgamma, float *dbeta, void *workspace,
                  size_t workspace_bytes, int64_t M, int64_t N, int dtype,
                  gbnorm_stream_t stream);

/*
 * General form: strided rows, a storage type per tensor, and a residual add
 * fused in front of the norm.
 *
 * Rows with a stride other than N and optional gamma / beta are the path's
 * first ranked extension, parameters and outputs in their own types (for
 * example bf16 rows with fp32 gamma, or fp32 rows with a bf16 y) the second,
 * and the fused residual add the third; the "Fused RMSNorm" page's "How it
 * works" section (16-bit storage, fp32 arithmetic) and the "SOTA
 * normalization performance with torch.compile" page's paragraphs on fusing a
 * norm with its neighbouring operations describe the motivation.  What is
 * computed is the definition at the top of this file, with:
 *
 *   h_ij = rnd_x(x_ij + r_ij)  when a residual r is given (else h = x): the
 *          sum in fp32, rounded once to x_dtype -- what an unfused h = x + r
 *          followed by the norm computes; h is normalised and, if `h` is
 *          given, stored.
 *   y    = the forward of h, rounded once to y_dtype.
 *   dx   = the input gradient of the norm at h, plus dres (the gradient that
 *          reaches h from the residual stream), rounded once to x_dtype; it is
 *          the gradient of both x and r.
 *
 * Arguments:
 *   is_layernorm  0 RMSNorm, 1 LayerNorm.
 *   M, N          rows and row length (M >= 0, 1 <= N <= GBNORM_MAX_N).
 *   x, ldx, x_dtype           [M] rows of N elements, row i at x + i * ldx
 *                             elements (ldx >= N); read only.
 *   residual, ldr             rows of x_dtype, or NULL (no residual add).
 *   h, ldh                    rows of x_dtype written with the residual sum,
 *                             or NULL (not stored); must be NULL without a
 *                             residual.
 *   gamma, beta, param_dtype  [N] each, or NULL (1 / 0); beta LayerNorm only.
 *   y, ldy, y_dtype           output rows.
 *   mean, rstd                [M] float32, written; may be NULL (mean is
 *                             LayerNorm only).
 *   dy, lddy, y_dtype         [M] rows: gradient of y, read only.
 *   x, ldx, x_dtype (bwd)     the rows that were normalised (h when the
 *                             forward added a residual), read only.
 *   dres, lddres              rows of x_dtype added into dx, or NULL.
 *   dx, lddx                  rows of x_dtype, written.
 *   dgamma, dbeta             [N] float32, written; may be NULL.
 *   workspace                 at least norm_bwd_ex_workspace_size(is_layernorm,
 *                             M, N) bytes, 16-byte aligned, not shared with a
 *                             concurrent call.
 *
 * An output may be exactly one of the inputs (same address, row stride and
 * element size: in place, e.g. h over r, or dx over dres or dy); any other
 * overlap of the spans [p, p + ((M - 1) * ld + N) * size) is rejected, and dx
 * may not be x.  With every row 16-byte aligned (base and stride), N a
 * multiple of 8 and 16-byte-aligned gamma / beta, rows move as 16-byte
 * vectors: for rows up to 16384 elements they are staged through a
 * shared-memory ring by bulk asynchronous copies (in the backward only when
 * rstd, and mean for LayerNorm, are 16-byte aligned too), else read straight
 * into registers; anything else takes a correct element-wise path.  Status
 * codes, ownership, streams and threading as above.
 */
int norm_fwd_ex(int is_layernorm, int64_t M, int64_t N, float eps, const void *x, int64_t ldx, int x_dtype,
                const void *residual, int64_t ldr, void *h, int64_t ldh, const void *gamma, const void *beta,
                int param_dtype, void *y, int64_t ldy, int y_dtype, float *mean, float *rstd,
                gbnorm_stream_t stream);
size_t norm_bwd_ex_workspace_size(int is_layernorm, int64_t M, int64_t N);
int norm_bwd_ex(int is_layernorm, int64_t M, int64_t N, const void *dy, int64_t lddy, int y_dtype,
                const void *x, int64_t ldx, int x_dtype, const void *dres, int64_t lddres, const void *gamma,
                int param_dtype, const float *mean, const float *rstd, void *dx, int64_t lddx, float *dgamma,
                float *dbeta, void *workspace, size_t workspace_bytes, gbnorm_stream_t stream);

/*
 * RMSNorm backward without a caller-provided workspace.
 *
 * No counterpart on the pages: this entry point exists for callers that cannot
 * allocate device memory at the point where they run the backward -- for
 * example code inside a framework's allocator or memory-pool callback (which
 * must not re-enter the allocator), a plugin whose enqueue function runs
 * under a fixed memory budget, or a runtime that forbids cudaMalloc on its
 * hot path because it synchronises the device.  It allocates nothing: it calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 * Arguments, layout and results are those of rmsnorm_bwd minus the workspace.
 * The dgamma partial rows go to a fixed scratch array of
 * GBNORM_NOALLOC_SCRATCH_BYTES inside the library, one per device, reserved
 * when the library's device code is loaded on that device and held until the
 * process exits.  A shape whose partial rows need more than that
 * (norm_bwd_workspace_size(0, M, N, dtype) > GBNORM_NOALLOC_SCRATCH_BYTES) is
 * refused with GBNORM_ERR_WORKSPACE before anything is enqueued.
 *
 * All calls on a device share that one scratch array, which keeps the last
 * call's contents (the kernels overwrite every entry they read, so nothing
 * needs clearing).  Two calls whose work overlaps on the GPU -- on different
 * streams, or from different host threads -- race on it and give wrong
 * dgamma; serialise them.
 *
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.
 */
#define GBNORM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *gamma, const float *rstd,
                        void *dx, float *dgamma, int64_t M, int64_t N, int dtype,
                        gbnorm_stream_t stream);

/* Static, human-readable text for a status code. */
const char *gbnorm_status_string(int status);

/*
 * Dispatch introspection and tuning (not needed for normal use).
 *
 * gbnorm_variant_name writes into buf (NUL-terminated, at most len bytes) the
 * name of the kernel variant that a call with these arguments would launch on
 * the current device, and returns GBNORM_OK; `aligned` says whether every
 * pointer of the call would be 16-byte aligned.  dir is 0 for the forward, 1
 * for the backward.
 *
 * gbnorm_force_variant makes every later call of (is_layernorm, dir, dtype)
 * in this process launch the named variant whenever it can serve the shape
 * (otherwise dispatch proceeds as usual); name NULL or "" removes the
 * override.  Returns GBNORM_ERR_INVALID_ARG for an unknown name.  Meant for
 * tests and tuning sweeps; not to be changed while another host thread is
 * calling the library.
 */
int gbnorm_variant_name(int is_layernorm, int dir, int64_t M, int64_t N, int dtype, int aligned,
                        char *buf, size_t len);
int gbnorm_force_variant(int is_layernorm, int dir, int dtype, const char *name);

/*
 * Number of kernel variants built for (is_layernorm, dir, dtype), and the
 * name of the index-th one (NULL if out of range).  For tests and tuning.
 */
int gbnorm_variant_count(int is_layernorm, int dir, int dtype);
const char *gbnorm_variant_at(int is_layernorm, int dir, int dtype, int index);

/*
 * The general form's kernels (norm_fwd_ex / norm_bwd_ex), for tests and
 * tuning.  gbnorm_ex_variant_count gives how many there are for
 * (is_layernorm, dir), the last being the element-wise kernel "exe";
 * gbnorm_ex_variant_at the index-th name (static string; NULL if out of
 * range).  gbnorm_ex_force_variant makes every later general-form call of
 * (is_layernorm, dir) in this process launch the named kernel whenever it can
 * serve the call (otherwise the usual choice is made); NULL or "" removes the
 * override; GBNORM_ERR_INVALID_ARG for an unknown name.  Not to be changed
 * while another host thread is calling the library.
 * gbnorm_ex_last_variant writes into buf (NUL-terminated, at most len bytes)
 * the name of the kernel that the calling thread's last norm_fwd_ex (dir 0)
 * or norm_bwd_ex (dir 1) launched, "" if that call launched none (M = 0 or
 * an error before the launch) or there was no such call.
 */
int gbnorm_ex_variant_count(int is_layernorm, int dir);
const char *gbnorm_ex_variant_at(int is_layernorm, int dir, int index);
int gbnorm_ex_force_variant(int is_layernorm, int dir, const char *name);
int gbnorm_ex_last_variant(int dir, char *buf, size_t len);

/*
 * Caps the persistent grid of every later launch at max_ctas CTAs (0 removes
 * the cap; negative values are rejected).  Results do not change, only how
 * many rows each CTA walks through; the backward workspace size follows the
 * cap.  For tests and tuning; not to be changed while another host thread is
 * calling the library.
 */
int gbnorm_set_grid_limit(int max_ctas);

/*
 * Device fault word of the current device.  The kernels that stage rows
 * through shared memory wait on hardware barriers; every such wait gives up
 * after about two seconds, sets this word to nonzero and lets the kernel run
 * to its end (its outputs are then meaningless) instead of hanging the GPU.
 * Writes the word into *value and, if reset is nonzero, clears it.  This call
 * synchronises with the device (it is a diagnostic, not for the hot path).
 */
int gbnorm_read_fault(int reset, int *value);

#ifdef __cplusplus
}
#endif

#endif /* GBNORM_H */
