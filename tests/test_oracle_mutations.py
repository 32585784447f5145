"""Plant plausible mistakes in copies of the oracle (CPU only) and check that a pin fails.

Each mutation is a one-token slip of the kind the pins are meant to catch: a dropped
term, a flipped sign, a wrong index, a transposed operand, a misplaced eps, the sample
instead of the population variance. The committed oracle is never modified; each
mutant is compiled from a patched copy in a temporary directory. The cross-entropy
reductions written in Python (the mean over the rows not ignored, and its gradient) are
mutated by replacing the function for the duration of one test.
"""
import pytest

import oracle
from oracle_pins import ALL_PINS

MUTATIONS = {
    "rms_eps_outside_sqrt": ("double r = 1.0 / sqrt(ms + eps);", "double r = 1.0 / (sqrt(ms) + eps);"),
    "rms_gamma_index": ("Y[i * D + j] = x[j] * r * gamma[j];", "Y[i * D + j] = x[j] * r * gamma[D - 1 - j];"),
    "rms_bwd_sign": ("dX[i * D + j] = r * (g - xhat * c);", "dX[i * D + j] = r * (g + xhat * c);"),
    "rms_bwd_dropped_c": ("dX[i * D + j] = r * (g - xhat * c);", "dX[i * D + j] = r * g;"),
    "rms_bwd_missing_r": ("dX[i * D + j] = r * (g - xhat * c);", "dX[i * D + j] = (g - xhat * c);"),
    "rms_dgamma_uses_g": ("double term = dy[j] * xhat;\n            dgamma[j] += term;\n            dgamma_abs[j] += fabs(term);\n        }\n    }\n}",
                          "double term = g * xhat;\n            dgamma[j] += term;\n            dgamma_abs[j] += fabs(term);\n        }\n    }\n}"),
    "ln_sample_variance": ("double var = sum_sq / (double)D;", "double var = sum_sq / (double)(D - 1);"),
    "ln_uncentred_variance": ("sum_sq += (x[j] - mu) * (x[j] - mu);", "sum_sq += x[j] * x[j];"),
    "ln_bias_dropped": ("Y[i * D + j] = (x[j] - mu) * r * gamma[j] + beta[j];", "Y[i * D + j] = (x[j] - mu) * r * gamma[j];"),
    "ln_bwd_dropped_mean_g": ("dX[i * D + j] = r * (g - a - xhat * c);", "dX[i * D + j] = r * (g - xhat * c);"),
    "ln_dbeta_uses_g": ("dbeta[j] += dy[j];", "dbeta[j] += g;"),
    "ln_dgamma_transposed": ("double term = dy[j] * xhat;\n            dgamma[j] += term;\n            dgamma_abs[j] += fabs(term);\n            dbeta",
                             "double term = dy[j] * ((x[D - 1 - j] - mu) * r);\n            dgamma[j] += term;\n            dgamma_abs[j] += fabs(term);\n            dbeta"),
    "add_residual_dropped": ("S[i] = X[i] + R[i];", "S[i] = X[i];"),
    "add_ds_subtracted": ("dX[i] += dS[i];", "dX[i] -= dS[i];"),
    "add_ds_ignored": ("dX[i] += dS[i];", "dX[i] += 0.0 * dS[i];"),
    "softmax_sum_without_max": ("        for (int64_t j = 0; j < D; ++j)\n            s += exp(x[j] - m);",
                                "        for (int64_t j = 0; j < D; ++j)\n            s += exp(x[j]);"),
    "softmax_bwd_sign": ("(y[j] * (dy[j] - dot))", "(y[j] * (dy[j] + dot))"),
    "logsoftmax_bwd_missing_exp": ("(dy[j] - exp(y[j]) * dot)", "(dy[j] - y[j] * dot)"),
    "logsoftmax_missing_log": ("(x[j] - m - log(s))", "(x[j] - m - s)"),
    "ce_smoothing_dropped": ("- (eps / (double)D) * sum_x", "- 0.0 * sum_x"),
    "ce_target_index": ("l - (1.0 - eps) * x[t]", "l - (1.0 - eps) * x[(t + 1) % D]"),
    "ce_zloss_factor": ("(1.0 + 2.0 * z * lse[i])", "(1.0 + z * lse[i])"),
    "ce_grad_sign": ("* p - q);", "* p + q);"),
    "ce_ignored_row_not_zeroed": ("                dX[i * D + j] = 0.0;\n                continue;",
                                  "                ;"),
    "gemv_column_reversed": ("double t = xn[k] * w[n];", "double t = xn[k] * w[N - 1 - n];"),
    "gemv_first_feature_dropped": ("for (int64_t k = 0; k < K; ++k) {\n            const double *w",
                                   "for (int64_t k = 1; k < K; ++k) {\n            const double *w"),
    "gemv_layernorm_as_rmsnorm": ("        if (op == 0)\n            oracle_rmsnorm_forward",
                                  "        if (op >= 0)\n            oracle_rmsnorm_forward"),
    "gemv_abs_terms_signed": ("ya[n] += fabs(t);", "ya[n] += t;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.load_library(oracle.compile_oracle(str(mutated), str(tmp_path / "libmutant.so")))
    failures = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {str(e).splitlines()[0]}")
    assert failures, f"no pin caught mutation {name}"


# Slips in the Python-level reductions of the cross-entropy oracle, planted by replacing the
# function for the duration of the test.
def _mean_over_all_rows(orig):
    def reduce(loss, T, ignore_index, reduction):
        val, n_valid = orig(loss, T, ignore_index, reduction)
        if reduction == "mean":
            return float(sum(loss)) / len(loss), n_valid
        return val, n_valid
    return "cross_entropy_reduce", reduce


def _mean_grad_without_count(orig):
    def row_grad(dloss, N, n_valid, reduction):
        return orig(dloss, N, n_valid, "sum" if reduction == "mean" else reduction)
    return "cross_entropy_row_grad", row_grad


PY_MUTATIONS = {
    "ce_mean_over_all_rows": (_mean_over_all_rows, "cross_entropy_reduce"),
    "ce_mean_grad_without_count": (_mean_grad_without_count, "cross_entropy_row_grad"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_python_mutation_is_caught(monkeypatch, name):
    make, attr = PY_MUTATIONS[name]
    target, fn = make(getattr(oracle, attr))
    monkeypatch.setattr(oracle, target, fn)
    lib = oracle.load_library()
    failures = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {str(e).splitlines()[0]}")
    assert failures, f"no pin caught mutation {name}"
