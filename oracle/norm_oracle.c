/*
 * norm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded fp64 CPU oracle for row-wise normalization:
 * RMSNorm, LayerNorm and fused residual-add + RMSNorm, forward and backward.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it. It shares no code, header or constant with the CUDA library, and the
 * CUDA library never loads it.
 *
 * Every input arrives as fp64 (the fp16 storage values widened exactly by the
 * caller); every output is fp64, unrounded. Rounding to the fp16 storage type
 * is left to the caller. Arrays are row-major [N, D]; parameter vectors are [D];
 * per-row statistics are [N]. There is no blocking, fusion or reordering: each
 * function is the textbook definition written out, row by row, left to right.
 *
 * Sources (page title, section):
 *   [meTile]  "Kernel coverage and training scope", section "Exact native
 *             normalization contract": the three forward formulas, population
 *             variance of the centred row, the fused op normalising the unrounded
 *             FP32 sum, the residual-output cotangent added to both input
 *             gradients, the backward being the exact derivative of the
 *             forward formula, taken at the saved fp32 statistics.
 *   [tc]      "Training kernels" (tensorcore docs), sections "RMSnorm -- Llama-style"
 *             (Math: rms(x) = sqrt(mean(x^2) + eps), y = x / rms * gamma) and
 *             "LayerNorm -- standard" (the mean and rstd kept
 *             for backward).
 *   The backward expressions below are the derivative of those forward formulas;
 *   the test suite pins them against central finite differences.
 *
 * Parity pins: every function here is pinned by tests in tests/test_oracle_pins.py
 * (finite differences, closed forms, invariants, a worked example from [meTile],
 * and a textbook library routine in fp64).
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (no FMA contraction,
 * so x86-64 and aarch64 hosts give the same bits).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* ------------------------------------------------------------------------- */
/* RMSNorm forward. [tc] "RMSnorm -- Llama-style", Math; [meTile] contract:
 *   ms_i   = (1/D) sum_j x_ij^2
 *   rstd_i = 1 / sqrt(ms_i + eps)
 *   y_ij   = x_ij * rstd_i * gamma_j          (zero-offset weight)            */
void oracle_rmsnorm_forward(const double *X, const double *gamma,
                            double *Y, double *rstd,
                            int64_t N, int64_t D, double eps)
{
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        double sum_sq = 0.0;
        for (int64_t j = 0; j < D; ++j)
            sum_sq += x[j] * x[j];
        double ms = sum_sq / (double)D;
        double r = 1.0 / sqrt(ms + eps);
        rstd[i] = r;
        for (int64_t j = 0; j < D; ++j)
            Y[i * D + j] = x[j] * r * gamma[j];
    }
}

/* RMSNorm backward: derivative of the forward above for the loss
 * L = sum_ij dY_ij * y_ij, at the saved rstd ([meTile] contract: the backward is the
 * exact derivative of the forward formula at the saved statistics).
 *   xhat_ij = x_ij * rstd_i,   g_ij = dY_ij * gamma_j
 *   c_i     = (1/D) sum_j g_ij * xhat_ij
 *   dX_ij   = rstd_i * (g_ij - xhat_ij * c_i)
 *   dgamma_j = sum_i dY_ij * xhat_ij            (rows in ascending order)
 * dgamma_abs_j = sum_i |dY_ij * xhat_ij| is the scale of the dgamma tolerance. */
void oracle_rmsnorm_backward(const double *X, const double *gamma,
                             const double *dY, const double *rstd,
                             double *dX, double *dgamma, double *dgamma_abs,
                             int64_t N, int64_t D)
{
    for (int64_t j = 0; j < D; ++j) {
        dgamma[j] = 0.0;
        dgamma_abs[j] = 0.0;
    }
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        const double *dy = dY + i * D;
        double r = rstd[i];
        double sum_gx = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = x[j] * r;
            double g = dy[j] * gamma[j];
            sum_gx += g * xhat;
        }
        double c = sum_gx / (double)D;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = x[j] * r;
            double g = dy[j] * gamma[j];
            dX[i * D + j] = r * (g - xhat * c);
            double term = dy[j] * xhat;
            dgamma[j] += term;
            dgamma_abs[j] += fabs(term);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* LayerNorm forward. [meTile] contract: centre the row by its mean, take the
 * population variance of the centred values, then apply weight and bias.
 * [tc] "LayerNorm -- standard": mean and rstd are saved for backward.
 *   mean_i = (1/D) sum_j x_ij
 *   var_i  = (1/D) sum_j (x_ij - mean_i)^2
 *   rstd_i = 1 / sqrt(var_i + eps)
 *   y_ij   = (x_ij - mean_i) * rstd_i * gamma_j + beta_j                       */
void oracle_layernorm_forward(const double *X, const double *gamma,
                              const double *beta, double *Y,
                              double *mean, double *rstd,
                              int64_t N, int64_t D, double eps)
{
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        double sum = 0.0;
        for (int64_t j = 0; j < D; ++j)
            sum += x[j];
        double mu = sum / (double)D;
        double sum_sq = 0.0;
        for (int64_t j = 0; j < D; ++j)
            sum_sq += (x[j] - mu) * (x[j] - mu);
        double var = sum_sq / (double)D;
        double r = 1.0 / sqrt(var + eps);
        mean[i] = mu;
        rstd[i] = r;
        for (int64_t j = 0; j < D; ++j)
            Y[i * D + j] = (x[j] - mu) * r * gamma[j] + beta[j];
    }
}

/* LayerNorm backward: derivative of the forward above for L = sum dY * y, at
 * the saved mean and rstd.
 *   xhat_ij = (x_ij - mean_i) * rstd_i,   g_ij = dY_ij * gamma_j
 *   a_i = (1/D) sum_j g_ij,   c_i = (1/D) sum_j g_ij * xhat_ij
 *   dX_ij = rstd_i * (g_ij - a_i - xhat_ij * c_i)
 *   dgamma_j = sum_i dY_ij * xhat_ij,   dbeta_j = sum_i dY_ij
 * The *_abs outputs are the per-column sums of absolute terms.                 */
void oracle_layernorm_backward(const double *X, const double *gamma,
                               const double *dY, const double *mean,
                               const double *rstd,
                               double *dX, double *dgamma, double *dbeta,
                               double *dgamma_abs, double *dbeta_abs,
                               int64_t N, int64_t D)
{
    for (int64_t j = 0; j < D; ++j) {
        dgamma[j] = 0.0;
        dbeta[j] = 0.0;
        dgamma_abs[j] = 0.0;
        dbeta_abs[j] = 0.0;
    }
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        const double *dy = dY + i * D;
        double mu = mean[i];
        double r = rstd[i];
        double sum_g = 0.0;
        double sum_gx = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = (x[j] - mu) * r;
            double g = dy[j] * gamma[j];
            sum_g += g;
            sum_gx += g * xhat;
        }
        double a = sum_g / (double)D;
        double c = sum_gx / (double)D;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = (x[j] - mu) * r;
            double g = dy[j] * gamma[j];
            dX[i * D + j] = r * (g - a - xhat * c);
            double term = dy[j] * xhat;
            dgamma[j] += term;
            dgamma_abs[j] += fabs(term);
            dbeta[j] += dy[j];
            dbeta_abs[j] += fabs(dy[j]);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Fused residual-add + RMSNorm forward. [meTile] contract: the sum is formed
 * at full precision and the UNROUNDED sum is normalised; the residual sum is
 * also returned (the caller rounds it to the storage dtype).
 *   s_ij  = x_ij + res_ij          (exact in fp64 for fp16 operands)
 *   rstd_i, y_ij as RMSNorm forward of s.
 * S receives the exact sum s.                                                  */
void oracle_add_rmsnorm_forward(const double *X, const double *R,
                                const double *gamma, double *S, double *Y,
                                double *rstd, int64_t N, int64_t D, double eps)
{
    for (int64_t i = 0; i < N * D; ++i)
        S[i] = X[i] + R[i];
    oracle_rmsnorm_forward(S, gamma, Y, rstd, N, D, eps);
}

/* Fused residual-add + RMSNorm backward. [meTile] contract: takes both output
 * cotangents; the residual-output cotangent dS (NULL means zero) is added to
 * both input gradients, so d(source) = d(residual) = dX.
 *   dX_ij = rstd_i * (g_ij - xhat_ij * c_i) + dS_ij,   xhat_ij = S_ij * rstd_i
 * S is the saved residual sum the caller passes in (the rounded storage value,
 * or the exact sum for the exact-s reading).                                  */
void oracle_add_rmsnorm_backward(const double *S, const double *gamma,
                                 const double *dY, const double *dS,
                                 const double *rstd,
                                 double *dX, double *dgamma, double *dgamma_abs,
                                 int64_t N, int64_t D)
{
    oracle_rmsnorm_backward(S, gamma, dY, rstd, dX, dgamma, dgamma_abs, N, D);
    if (dS != NULL) {
        for (int64_t i = 0; i < N * D; ++i)
            dX[i] += dS[i];
    }
}

/* ========================================================================= */
/* Row softmax and per-row cross-entropy (the next row-reduction family).
 *
 * Sources (page title, section):
 *   [tc]      "Training kernels", section "Softmax -- standalone, row-wise":
 *             numerically stable row softmax, subtract the row maximum,
 *             exponentiate, sum, divide; backward from the output Y and dY.
 *   [meTile]  "Kernel coverage and training scope", "Reduction and attention
 *             parity checklist" (softmax and log-softmax with input gradients)
 *             and "Loss parity checklist" / the native training_losses notes
 *             (cross-entropy row loss and logit gradients: an index whose rows
 *             are skipped, losses per row, summed or averaged over the rows
 *             kept, label smoothing spread evenly over the classes, a penalty
 *             on the squared log-sum-exp; maxima and log-denominators kept
 *             for the backward).
 *   [report]  "Metal subgroup LayerNorm and cross-entropy report", section
 *             "Structural repair exercised by cross-entropy": peak = max,
 *             total = sum exp(logit - peak), loss = log(total) + peak - selected.
 * The reductions over rows (sum, mean) are left to the caller.              */

/* Softmax forward. [tc] Softmax; [meTile] softmax / log-softmax:
 *   m_i = max_j x_ij,   s_i = sum_j exp(x_ij - m_i)
 *   softmax:      y_ij = exp(x_ij - m_i) / s_i
 *   log-softmax:  y_ij = x_ij - m_i - log(s_i)                                 */
void oracle_softmax_forward(const double *X, double *Y, int64_t N, int64_t D,
                            int log_softmax)
{
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        double m = x[0];
        for (int64_t j = 1; j < D; ++j)
            if (x[j] > m) m = x[j];
        double s = 0.0;
        for (int64_t j = 0; j < D; ++j)
            s += exp(x[j] - m);
        for (int64_t j = 0; j < D; ++j)
            Y[i * D + j] = log_softmax ? (x[j] - m - log(s)) : (exp(x[j] - m) / s);
    }
}

/* Softmax backward from the forward output, for L = sum_ij dY_ij * y_ij:
 *   softmax:      dX_ij = y_ij * (dY_ij - sum_k dY_ik * y_ik)
 *   log-softmax:  dX_ij = dY_ij - exp(y_ij) * sum_k dY_ik                       */
void oracle_softmax_backward(const double *Y, const double *dY, double *dX,
                             int64_t N, int64_t D, int log_softmax)
{
    for (int64_t i = 0; i < N; ++i) {
        const double *y = Y + i * D;
        const double *dy = dY + i * D;
        double dot = 0.0;
        for (int64_t j = 0; j < D; ++j)
            dot += log_softmax ? dy[j] : dy[j] * y[j];
        for (int64_t j = 0; j < D; ++j)
            dX[i * D + j] = log_softmax ? (dy[j] - exp(y[j]) * dot) : (y[j] * (dy[j] - dot));
    }
}

/* Cross-entropy forward per row. [meTile] losses; [report] formula. Target
 * distribution with uniform label smoothing eps over the D classes:
 *   q_ij = (1 - eps) * [j == t_i] + eps / D
 *   lse_i  = m_i + log(sum_j exp(x_ij - m_i))            (saved for backward)
 *   loss_i = sum_j q_ij * (lse_i - x_ij) + z * lse_i^2
 *          = lse_i - (1 - eps) * x_i,t_i - (eps / D) * sum_j x_ij + z * lse_i^2
 * A row whose target equals ignore_index has loss 0 (lse still written). A
 * target outside [0, D) that is not ignore_index gives a NaN loss.            */
void oracle_cross_entropy_forward(const double *X, const int64_t *T, int64_t N,
                                  int64_t D, int64_t ignore_index, double eps,
                                  double z, double *loss, double *lse)
{
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        double m = x[0];
        for (int64_t j = 1; j < D; ++j)
            if (x[j] > m) m = x[j];
        double s = 0.0, sum_x = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            s += exp(x[j] - m);
            sum_x += x[j];
        }
        double l = m + log(s);
        lse[i] = l;
        int64_t t = T[i];
        if (t == ignore_index) {
            loss[i] = 0.0;
        } else if (t < 0 || t >= D) {
            loss[i] = NAN;
        } else {
            loss[i] = l - (1.0 - eps) * x[t] - (eps / (double)D) * sum_x + z * l * l;
        }
    }
}

/* Cross-entropy backward: derivative of loss_i above, times the row's upstream
 * gradient g_i (the caller forms g from the reduction: none -> dloss_i,
 * sum -> dloss, mean -> dloss / number of valid rows), at the saved lse:
 *   p_ij   = exp(x_ij - lse_i)
 *   dX_ij  = g_i * ((1 + 2 z lse_i) * p_ij - q_ij)
 * Ignored rows get 0.                                                          */
void oracle_cross_entropy_backward(const double *X, const int64_t *T,
                                   const double *lse, const double *g,
                                   int64_t N, int64_t D, int64_t ignore_index,
                                   double eps, double z, double *dX)
{
    for (int64_t i = 0; i < N; ++i) {
        const double *x = X + i * D;
        int64_t t = T[i];
        for (int64_t j = 0; j < D; ++j) {
            if (t == ignore_index) {
                dX[i * D + j] = 0.0;
                continue;
            }
            double p = exp(x[j] - lse[i]);
            double q = (1.0 - eps) * (j == t ? 1.0 : 0.0) + eps / (double)D;
            dX[i * D + j] = g[i] * ((1.0 + 2.0 * z * lse[i]) * p - q);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Fused normalization + GEMV. [tc] "Fused Norm + GEMV": Y = Norm(X, gamma[, beta]) @ W
 * with X [M, K], W [K, N] (row k of W holds the weights of input feature k), Y [M, N];
 * Norm is the RMSNorm forward (op 0) or the LayerNorm forward (op 1) above. The
 * normalized row is used unrounded: the fused kernels apply it in registers during
 * the accumulation and never store it.
 *   xn_m  = Norm(x_m)                         (the forward above, one row)
 *   Y_mn  = sum_k xn_mk * W_kn                (k ascending)
 *   Y_abs_mn = sum_k |xn_mk * W_kn|           (the scale of the sum's rounding)
 * xn: caller-provided scratch of K doubles.                                     */
void oracle_norm_gemv(int op, const double *X, const double *gamma, const double *beta,
                      const double *W, double *Y, double *Y_abs, double *xn,
                      int64_t M, int64_t N, int64_t K, double eps)
{
    for (int64_t m = 0; m < M; ++m) {
        double mean, rstd;
        if (op == 0)
            oracle_rmsnorm_forward(X + m * K, gamma, xn, &rstd, 1, K, eps);
        else
            oracle_layernorm_forward(X + m * K, gamma, beta, xn, &mean, &rstd, 1, K, eps);
        double *y = Y + m * N, *ya = Y_abs + m * N;
        for (int64_t n = 0; n < N; ++n) {
            y[n] = 0.0;
            ya[n] = 0.0;
        }
        for (int64_t k = 0; k < K; ++k) {
            const double *w = W + k * N;
            for (int64_t n = 0; n < N; ++n) {
                double t = xn[k] * w[n];
                y[n] += t;
                ya[n] += fabs(t);
            }
        }
    }
}
