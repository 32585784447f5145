/*
 * mt_norm.h -- C ABI of the GB300 (sm_103a) row-wise normalization library.
 *
 * Three training operations, each a forward and a backward entry point:
 *   RMSNorm                       mt_rmsnorm_forward / mt_rmsnorm_backward
 *   LayerNorm                     mt_layernorm_forward / mt_layernorm_backward
 *   fused residual-add + RMSNorm  mt_add_rmsnorm_forward / mt_add_rmsnorm_backward
 * with explicit storage types (mt_norm_forward_ex / mt_norm_backward_ex), and on the same
 * row skeleton a row softmax / log-softmax (mt_softmax_*), a per-row cross-entropy
 * (mt_cross_entropy_*) and, for decode, normalization fused into the GEMV that consumes
 * it (mt_fused_rmsnorm_gemv / mt_fused_layernorm_gemv).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.   Activations (X, R, S, Y, dY, dS, dX) are dense row-major [N, D] arrays of
 *           IEEE binary16 (fp16), row i starting at element i*D. gamma and beta are [D]
 *           fp16. mean and rstd are [N] fp32. dgamma and dbeta are [D] fp32.
 * Memory.   Every pointer is a device pointer on the CUDA device current on the calling
 *           thread. The caller owns every buffer; the library keeps no pointer after the
 *           call returns. Any alignment is accepted (16-byte aligned rows with D a
 *           multiple of 8 take the vectorised path).
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *           asynchronous: work is enqueued on `stream` and the function returns.
 * Outputs.  Outputs are overwritten, never accumulated into. Outputs may not overlap any
 *           input or any other output (no in-place operation).
 * Saved state. The forward's saved tensors (X or S, mean, rstd) must not be modified
 *           between a forward and the backward that consumes them.
 * Arithmetic. All arithmetic is fp32; fp16 results are rounded to nearest even.
 *           dgamma/dbeta are reduced in a fixed order without atomics, so every output
 *           is bitwise identical from run to run on the same device and shape.
 * Bounds.   0 <= N <= 2^31 - 1 and 1 <= D <= MT_MAX_COLS. eps must be finite and > 0.
 * Empty batch. N = 0 is a no-op that returns MT_OK: nothing is read, the activation
 *           and per-row pointers may be NULL, and a backward only sets dgamma (and
 *           dbeta) to 0, the empty sum over rows, with no workspace.
 * Errors.   Arguments are validated before any CUDA call is made:
 *             MT_ERR_INVALID_ARG  a required pointer is NULL, N < 0, D < 1, eps not
 *                                 finite or not > 0, or an output overlaps an input or
 *                                 another output;
 *             MT_ERR_UNSUPPORTED  D > MT_MAX_COLS, N > 2^31 - 1, or a caller-supplied
 *                                 workspace smaller than the size query returns;
 *             MT_ERR_CUDA         a CUDA call or kernel launch failed;
 *                                 mt_last_cuda_error() returns its cudaError_t value.
 *           Non-finite input values are not repaired: a NaN or Inf propagates to its
 *           row's outputs and to the dgamma/dbeta columns it touches.
 *
 * Sources (page title, section):
 *   [meTile] "Kernel coverage and training scope", "Exact native normalization contract".
 *   [tc]     "Training kernels" (tensorcore docs), "RMSnorm -- Llama-style" and
 *            "LayerNorm -- standard": the C signatures, buffer dtypes and saved statistics.
 */
#ifndef MT_NORM_H
#define MT_NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes; the [tc] API returns a status code the same way. */
typedef enum mt_status {
    MT_OK = 0,
    MT_ERR_INVALID_ARG = 1,
    MT_ERR_UNSUPPORTED = 2,
    MT_ERR_CUDA = 3
} mt_status_t;

/* Operation selector for the workspace-size query and the explicit-dtype entry points. */
typedef enum mt_norm_op {
    MT_OP_RMSNORM = 0,
    MT_OP_LAYERNORM = 1,
    MT_OP_ADD_RMSNORM = 2
} mt_norm_op_t;

/* ABI-identical to cudaStream_t, so this header needs no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st *mt_stream_t;

/* Widest supported row of the normalizations. [meTile] bounds rows to 1..8192 columns;
 * this library extends the bound to 131072. Rows up to 16384 columns run on one CTA.
 * Wider rows: the forward of an aligned row (D % 8 == 0, 16-byte row bases) reads the
 * row twice on one CTA (a reduction pass, then the apply); the backward, and the
 * forward of other rows, split the row across a thread-block cluster of 2, 4 or 8 CTAs
 * (one slice of at most 16384 columns each) that add their row sums through
 * distributed shared memory in a fixed order. Results stay bitwise reproducible. */
#define MT_MAX_COLS 131072

/* Widest row of the softmax / log-softmax: [meTile] training_losses bounds last-axis
 * softmax to 1..262144 columns. Rows up to 16384 columns stay in registers (one read,
 * one write); wider rows run two passes over the row on one CTA (a running maximum and
 * sum of exponentials, then the outputs; the second read mostly hits L2). */
#define MT_MAX_SOFTMAX_COLS 262144

/* ---------------------------------------------------------------- RMSNorm ---
 * [tc] "RMSnorm -- Llama-style", Math; [meTile] contract (zero-offset weight):
 *   rstd_i = 1 / sqrt(mean_j(X_ij^2) + eps),   Y_ij = X_ij * rstd_i * gamma_j.
 * In:  X [N,D] fp16, gamma [D] fp16, eps.
 * Out: Y [N,D] fp16, rstd [N] fp32 (saved for the backward).                     */
mt_status_t mt_rmsnorm_forward(const void *X, const void *gamma, void *Y, float *rstd,
                               int64_t N, int64_t D, float eps, mt_stream_t stream);

/* Backward of mt_rmsnorm_forward at the saved rstd (no eps argument: [tc]
 * signature). With xhat = X*rstd, g = dY*gamma, c_i = mean_j(g_ij*xhat_ij):
 *   dX_ij = rstd_i * (g_ij - xhat_ij*c_i),   dgamma_j = sum_i dY_ij*xhat_ij.
 * In:  X, dY [N,D] fp16, gamma [D] fp16, rstd [N] fp32.
 * Out: dX [N,D] fp16, dgamma [D] fp32.
 * Scratch: a stream-ordered allocation (cudaMallocAsync on `stream`) of
 * mt_norm_backward_workspace_size() bytes, freed on `stream` before returning.   */
mt_status_t mt_rmsnorm_backward(const void *X, const void *gamma, const void *dY,
                                const float *rstd, void *dX, float *dgamma,
                                int64_t N, int64_t D, mt_stream_t stream);

/* As mt_rmsnorm_backward, with caller-owned scratch: `workspace` is a device buffer of
 * at least mt_norm_backward_workspace_size(MT_OP_RMSNORM, N, D, device) bytes, used
 * only for the duration of the enqueued work. No allocation is made.               */
mt_status_t mt_rmsnorm_backward_ws(const void *X, const void *gamma, const void *dY,
                                   const float *rstd, void *dX, float *dgamma,
                                   int64_t N, int64_t D, void *workspace,
                                   size_t workspace_bytes, mt_stream_t stream);

/* -------------------------------------------------------------- LayerNorm ---
 * [meTile] contract: centre each row by its mean, population variance of the
 * centred values, then weight and bias; [tc] "LayerNorm -- standard": mean and
 * rstd saved for backward.
 *   mean_i = mean_j X_ij,  rstd_i = 1/sqrt(mean_j (X_ij - mean_i)^2 + eps),
 *   Y_ij = (X_ij - mean_i) * rstd_i * gamma_j + beta_j.
 * In:  X [N,D] fp16, gamma, beta [D] fp16, eps.
 * Out: Y [N,D] fp16, mean [N] fp32, rstd [N] fp32.                               */
mt_status_t mt_layernorm_forward(const void *X, const void *gamma, const void *beta,
                                 void *Y, float *mean, float *rstd,
                                 int64_t N, int64_t D, float eps, mt_stream_t stream);

/* Backward of mt_layernorm_forward at the saved mean and rstd. With
 * xhat = (X - mean)*rstd, g = dY*gamma, a_i = mean_j g_ij, c_i = mean_j g_ij*xhat_ij:
 *   dX_ij = rstd_i * (g_ij - a_i - xhat_ij*c_i),
 *   dgamma_j = sum_i dY_ij*xhat_ij,   dbeta_j = sum_i dY_ij.
 * [tc]'s printed signature has no parameter gradients; [meTile] returns both, and
 * so does this entry point.
 * In:  X, dY [N,D] fp16, gamma [D] fp16, mean, rstd [N] fp32.
 * Out: dX [N,D] fp16, dgamma, dbeta [D] fp32. Scratch as mt_rmsnorm_backward.      */
mt_status_t mt_layernorm_backward(const void *X, const void *gamma, const void *dY,
                                  const float *mean, const float *rstd, void *dX,
                                  float *dgamma, float *dbeta,
                                  int64_t N, int64_t D, mt_stream_t stream);

mt_status_t mt_layernorm_backward_ws(const void *X, const void *gamma, const void *dY,
                                     const float *mean, const float *rstd, void *dX,
                                     float *dgamma, float *dbeta, int64_t N, int64_t D,
                                     void *workspace, size_t workspace_bytes,
                                     mt_stream_t stream);

/* ------------------------------------------------- fused residual add + RMSNorm ---
 * [meTile] contract: the sum is formed in fp32 and the UNROUNDED sum is normalised;
 * the residual sum is also returned, rounded to fp16.
 *   s_ij = X_ij + R_ij (fp32),  S_ij = fp16(s_ij),
 *   rstd_i = 1/sqrt(mean_j s_ij^2 + eps),  Y_ij = s_ij * rstd_i * gamma_j.
 * In:  X, R [N,D] fp16, gamma [D] fp16, eps.
 * Out: S [N,D] fp16 (the residual stream), Y [N,D] fp16, rstd [N] fp32.            */
mt_status_t mt_add_rmsnorm_forward(const void *X, const void *R, const void *gamma,
                                   void *S, void *Y, float *rstd,
                                   int64_t N, int64_t D, float eps, mt_stream_t stream);

/* Backward of mt_add_rmsnorm_forward. [meTile] contract: takes both output
 * cotangents; the residual-output cotangent dS is added to both input gradients,
 * and a NULL dS means zero. With xhat = S*rstd (S the saved fp16 residual sum),
 * g = dY*gamma, c_i = mean_j g_ij*xhat_ij:
 *   dX_ij = rstd_i * (g_ij - xhat_ij*c_i) + dS_ij,   dgamma_j = sum_i dY_ij*xhat_ij.
 * dX is both d(source) and d(residual): the two are equal, so one buffer is written.
 * In:  S, dY [N,D] fp16, dS [N,D] fp16 or NULL, gamma [D] fp16, rstd [N] fp32.
 * Out: dX [N,D] fp16, dgamma [D] fp32. Scratch as mt_rmsnorm_backward.              */
mt_status_t mt_add_rmsnorm_backward(const void *S, const void *gamma, const void *dY,
                                    const void *dS, const float *rstd, void *dX,
                                    float *dgamma, int64_t N, int64_t D,
                                    mt_stream_t stream);

mt_status_t mt_add_rmsnorm_backward_ws(const void *S, const void *gamma, const void *dY,
                                       const void *dS, const float *rstd, void *dX,
                                       float *dgamma, int64_t N, int64_t D,
                                       void *workspace, size_t workspace_bytes,
                                       mt_stream_t stream);

/* -------------------------------------------------------- explicit storage types ---
 * [meTile] contract: storage is FP16 or FP32, with weight, bias and cotangents each in
 * either type independently; statistics, accumulation and parameter gradients are FP32.
 * This library adds bf16 as a third storage type. The entry points above are the fp16
 * case of these two.
 *
 * x_dtype  X, R, S, Y (forward) and X or S, dX (backward): the activations. The
 *          forward output and the residual sum use the source type, as [meTile]
 *          states; dX also uses it, as the fp16 entry points do.
 * w_dtype  gamma, beta.
 * g_dtype  dY, dS: the cotangents.
 * mean, rstd, dgamma, dbeta are fp32 in every combination. Any combination of the three
 * types is accepted; fp16/bf16 activations with parameters and cotangents of the same
 * type or fp32, and all-fp32, take the vectorised kernels (D % 8 == 0 and 16-byte-aligned
 * bases), everything else the scalar kernels. Results are rounded to nearest even.
 *
 * op selects which pointers are used: MT_OP_RMSNORM uses X, gamma, Y, rstd (forward)
 * and X, gamma, dY, rstd, dX, dgamma (backward); MT_OP_LAYERNORM adds beta and mean
 * (forward) and mean and dbeta (backward); MT_OP_ADD_RMSNORM adds R and S (forward)
 * and takes the saved S as X and the optional dS (backward). Pointers an op does not
 * use are ignored. Errors as for the fp16 entry points, plus MT_ERR_INVALID_ARG for an
 * unknown op or dtype code.
 * Backward workspace: NULL allocates stream-ordered scratch as mt_rmsnorm_backward
 * does; otherwise it is a caller buffer of workspace_bytes >=
 * mt_norm_backward_workspace_size(op, N, D, device), which covers every dtype.       */
typedef enum mt_dtype {
    MT_DTYPE_F16 = 0,
    MT_DTYPE_BF16 = 1,
    MT_DTYPE_F32 = 2
} mt_dtype_t;

mt_status_t mt_norm_forward_ex(mt_norm_op_t op, mt_dtype_t x_dtype, mt_dtype_t w_dtype,
                               const void *X, const void *R, const void *gamma,
                               const void *beta, void *S, void *Y, float *mean, float *rstd,
                               int64_t N, int64_t D, float eps, mt_stream_t stream);

mt_status_t mt_norm_backward_ex(mt_norm_op_t op, mt_dtype_t x_dtype, mt_dtype_t w_dtype,
                                mt_dtype_t g_dtype, const void *X, const void *gamma,
                                const void *dY, const void *dS, const float *mean,
                                const float *rstd, void *dX, float *dgamma, float *dbeta,
                                int64_t N, int64_t D, void *workspace, size_t workspace_bytes,
                                mt_stream_t stream);

/* ------------------------------------------------------------ row softmax ---
 * [tc] "Softmax -- standalone, row-wise": numerically stable softmax of each row
 * (subtract the row maximum, exponentiate, sum, divide); [meTile] reduction checklist:
 * softmax and log-softmax with input gradients.
 *   softmax:      Y_ij = exp(X_ij - m_i) / sum_k exp(X_ik - m_i),  m_i = max_k X_ik
 *   log-softmax:  Y_ij = X_ij - m_i - log(sum_k exp(X_ik - m_i))
 *   backward from the forward output Y and dY:
 *     softmax:      dX_ij = Y_ij * (dY_ij - sum_k dY_ik * Y_ik)
 *     log-softmax:  dX_ij = dY_ij - exp(Y_ij) * sum_k dY_ik
 * X, Y, dY, dX are [N, D] of type `dtype`; log_softmax != 0 selects log-softmax.
 * Bounds: 1 <= D <= MT_MAX_SOFTMAX_COLS, 0 <= N <= 2^31 - 1 (N = 0: a no-op, pointers
 * may be NULL). Errors: MT_ERR_INVALID_ARG for a NULL pointer, N < 0, D < 1, an unknown
 * dtype or an output overlapping an input; MT_ERR_UNSUPPORTED for D or N past the bound.
 * Arithmetic fp32; results rounded to `dtype`, nearest even.                       */
mt_status_t mt_softmax_forward(mt_dtype_t dtype, const void *X, void *Y, int64_t N, int64_t D,
                               int log_softmax, mt_stream_t stream);
mt_status_t mt_softmax_backward(mt_dtype_t dtype, const void *Y, const void *dY, void *dX,
                                int64_t N, int64_t D, int log_softmax, mt_stream_t stream);

/* ---------------------------------------------------------- cross-entropy ---
 * [meTile] loss checklist and training_losses notes: per-row cross-entropy of logits
 * with integer class targets; rows whose target equals ignore_index are skipped;
 * the row losses are returned as they are, summed, or averaged (over the rows not
 * skipped; 0 when there is none); label smoothing spreads its mass evenly over the
 * classes; a z-loss penalises the squared log-sum-exp; the log-denominators are kept
 * for the backward. ["Metal subgroup LayerNorm and cross-entropy report", "Structural
 * repair exercised by cross-entropy"]: loss = log(total) + peak - selected.
 *   lse_i  = log(sum_j exp(X_ij))                 (computed from the row maximum)
 *   q_ij   = (1 - label_smoothing) [j == t_i] + label_smoothing / D
 *   loss_i = lse_i - (1 - label_smoothing) X_i,t_i - (label_smoothing / D) sum_j X_ij
 *            + z_loss * lse_i^2,      0 when t_i == ignore_index
 *   backward: dX_ij = g_i * ((1 + 2 z_loss lse_i) exp(X_ij - lse_i) - q_ij),
 *            g_i = dloss_i (NONE), dloss (SUM), dloss / n_valid (MEAN), 0 if ignored.
 * logits X / dX: [N, D] of type `dtype`; targets: [N] int64 (device); loss_rows, lse:
 * [N] fp32 (lse is saved for the backward and written for every row); loss_out and
 * n_valid: one fp32 each, written for SUM/MEAN (may be NULL for NONE). n_valid is the
 * number of rows not skipped, counted exactly and rounded to fp32 (exact up to 2^24
 * rows); MEAN divides the fp32 sum by the exact count. The backward's dloss is [N] for
 * NONE and one value otherwise, and n_valid (MEAN) is the forward's.
 * A target outside [0, D) that is not ignore_index gives a NaN loss for its row.
 * Bounds: 1 <= D <= MT_MAX_CE_COLS, 0 <= N <= 2^31 - 1; 0 <= label_smoothing <= 1,
 * z_loss >= 0 (both finite), else MT_ERR_INVALID_ARG. N = 0: the forward writes only
 * loss_out = 0 and n_valid = 0 (SUM/MEAN), the backward nothing; the [N] pointers may
 * be NULL. The sum over rows runs in a fixed order, so every result is bitwise
 * identical run to run.                                                             */
#define MT_MAX_CE_COLS 262144

typedef enum mt_reduction {
    MT_REDUCTION_NONE = 0,
    MT_REDUCTION_SUM = 1,
    MT_REDUCTION_MEAN = 2
} mt_reduction_t;

mt_status_t mt_cross_entropy_forward(mt_dtype_t dtype, const void *logits,
                                     const int64_t *targets, int64_t N, int64_t D,
                                     int64_t ignore_index, float label_smoothing, float z_loss,
                                     mt_reduction_t reduction, float *loss_rows, float *lse,
                                     float *loss_out, float *n_valid, mt_stream_t stream);
mt_status_t mt_cross_entropy_backward(mt_dtype_t dtype, const void *logits,
                                      const int64_t *targets, const float *lse, int64_t N,
                                      int64_t D, int64_t ignore_index, float label_smoothing,
                                      float z_loss, mt_reduction_t reduction,
                                      const float *dloss, const float *n_valid, void *dlogits,
                                      mt_stream_t stream);

/* ------------------------------------------ fused normalization + GEMV (decode) ---
 * [tc] "Fused Norm + GEMV":  Y = Norm(X, gamma[, beta]) @ W  for the small batches of a
 * decode step, with Norm the RMSNorm (eps inside the square root, zero-offset weight) or
 * LayerNorm (centred population variance) forward above. The normalized rows are
 * applied in registers during the accumulation and never stored, so there is no
 * x_norm round trip; the statistics are not returned (inference only, as on the page).
 *   X:     [M, K] fp16 (row-major)          gamma, beta: [K] fp16
 *   W:     [K, N] fp16 (row-major; row k holds the weights of input feature k)
 *   Y:     [M, N] fp16 (row-major)          Y_mn = sum_k Norm(x_m)_k * W_kn
 * Arithmetic fp32 (statistics, normalized values, products, sums); Y rounded to fp16,
 * nearest even. The sums over k run in a fixed order, so Y is bitwise identical run to
 * run on the same device and shape. Any alignment (N % 8 == 0 with a 16-byte aligned W
 * takes 16-byte loads).
 * Bounds: 0 <= M <= MT_MAX_GEMV_ROWS, 1 <= K <= MT_MAX_GEMV_K, 0 <= N <= 2^31 - 1; M = 0
 * or N = 0 is a no-op (pointers may be NULL). Errors: MT_ERR_INVALID_ARG for a NULL
 * pointer, a negative size, K < 1, eps not finite or not > 0, or Y overlapping an
 * input; MT_ERR_UNSUPPORTED past the bounds.                                       */
#define MT_MAX_GEMV_ROWS 8
#define MT_MAX_GEMV_K 32768

mt_status_t mt_fused_rmsnorm_gemv(const void *X, const void *gamma, const void *W, void *Y,
                                  int64_t M, int64_t N, int64_t K, float eps,
                                  mt_stream_t stream);
mt_status_t mt_fused_layernorm_gemv(const void *X, const void *gamma, const void *beta,
                                    const void *W, void *Y, int64_t M, int64_t N, int64_t K,
                                    float eps, mt_stream_t stream);

/* ----------------------------------------------- backward without allocation ---
 * No counterpart on the pages: this entry point exists for callers that cannot
 * allocate device memory. mt_rmsnorm_backward allocates its scratch and
 * mt_rmsnorm_backward_ws needs the caller to provide it; a caller whose device memory
 * is owned by a framework pool that must not be bypassed, or that runs in a loop where
 * an allocator call is not allowed, can do neither.
 *
 * Same arguments, outputs and results as mt_rmsnorm_backward. The scratch comes from
 * one fixed array of MT_NOALLOC_SCRATCH_BYTES compiled into the library, which every
 * GPU that loads the library holds until the process exits; no allocation or free is
 * made. The first call on each device looks up the array's device address (with that
 * device current) and caches it, so make that first call before any stream capture.
 * All calls share the array and leave their partials in it; nothing has to be cleared
 * between calls, but calls that overlap on the GPU race on it and must not be made.
 * A shape whose dgamma partials (one fp32 row of D per persistent CTA, or per cluster
 * of a split row) exceed MT_NOALLOC_SCRATCH_BYTES returns MT_ERR_UNSUPPORTED and
 * launches nothing; on a 152-SM GB300 every shape up to MT_MAX_COLS columns fits (the
 * largest need is about 10 MB: rows of 16383 columns on the scalar kernel, one partial row
 * per SM, and split rows of up to 131072 columns, one per cluster).
 * A device reset (cudaDeviceReset) unloads the library's device code, so the cached
 * address no longer names the array: after a reset of a device, this entry point must not
 * be called on it again in the same process.                                         */
#define MT_NOALLOC_SCRATCH_BYTES (16u << 20)

mt_status_t mt_rmsnorm_backward_noalloc(const void *X, const void *gamma, const void *dY,
                                        const float *rstd, void *dX, float *dgamma,
                                        int64_t N, int64_t D, mt_stream_t stream);

/* ------------------------------------------------------------------ utilities --- */

/* Scratch bytes a backward of `op` at [N, D] needs on CUDA device `device`, whatever
 * its storage types: the fixed-order dgamma (and dbeta) partials, one fp32 row of D per
 * persistent CTA (per cluster of a split row); 0 for N = 0.
 * Writes the size to *bytes. Errors: MT_ERR_INVALID_ARG / MT_ERR_UNSUPPORTED as the
 * backward would return them, MT_ERR_INVALID_ARG for a NULL `bytes` or an unknown
 * op, MT_ERR_CUDA if the device cannot be queried.                                */
mt_status_t mt_norm_backward_workspace_size(mt_norm_op_t op, int64_t N, int64_t D,
                                            int device, size_t *bytes);

/* cudaError_t value of the most recent MT_ERR_CUDA on the calling thread (0 if none). */
int mt_last_cuda_error(void);

/* The backward of a row split across a thread-block cluster (aligned rows wider than one
 * CTA's slice) exchanges its CTAs' row sums through distributed shared memory, each CTA
 * waiting on its own mbarrier for its peers' sums. Every such wait is bounded: one that
 * has not completed after 200 ms of device time gives up, the kernel ORs an error bit
 * into a status word of the device, skips the rows' remaining work and runs to its end,
 * so that no wait can hang the GPU; the call's outputs are then incomplete.
 * mt_device_wait_errors copies the word of CUDA device `device` to *flags (0: no wait has
 * ever given up; MT_WAIT_ERR_CLUSTER: a split row's exchange did) and, when `clear` is
 * non-zero, resets it. It synchronizes with the device (blocking copies). Errors:
 * MT_ERR_INVALID_ARG for a NULL `flags` or a negative device, MT_ERR_CUDA if a CUDA call
 * fails.                                                                            */
#define MT_WAIT_ERR_CLUSTER 1u
mt_status_t mt_device_wait_errors(int device, unsigned *flags, int clear);

/* Static, human-readable name of a status code. */
const char *mt_status_string(mt_status_t status);

/* Library version, major*10000 + minor*100 + patch. */
int mt_norm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MT_NORM_H */
