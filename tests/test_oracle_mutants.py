"""The pins must reject a wrong oracle.

Each case plants one plausible mistake (a dropped term, a wrong sign, an
off-by-one index, a transposed operand, a wrong variance divisor ...) in a
copy of the oracle's C source, compiles that copy, swaps it in and runs every
pin: at least one pin has to fail.  Everything happens on the CPU; the real
oracle is restored afterwards.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "rowops_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("softmax_sum_without_max", "            s += exp(xi[k] - m);\n        for (int64_t j = 0; j < cols; ++j)\n            yi[j] = exp(xi[j] - m) / s;",
     "            s += exp(xi[k]);\n        for (int64_t j = 0; j < cols; ++j)\n            yi[j] = exp(xi[j] - m) / s;"),
    ("softmax_exp_sign", "            yi[j] = exp(xi[j] - m) / s;", "            yi[j] = exp(m - xi[j]) / s;"),
    ("softmax_bwd_sign", "            dxi[j] = yi[j] * (dyi[j] - c);", "            dxi[j] = yi[j] * (dyi[j] + c);"),
    ("softmax_bwd_operand", "            c += yi[k] * dyi[k];", "            c += yi[k] * yi[k];"),
    ("attn_diagonal_off_by_one", "        const int64_t n = q + 1 < cols ? q + 1 : cols; /* keys 0..q survive the mask */",
     "        const int64_t n = q < cols ? q : cols;"),
    ("attn_scale_dropped_in_output", "            pi[j] = exp(scale * si[j] - m) / sum;", "            pi[j] = exp(si[j] - m) / sum;"),
    ("attn_bwd_scale_dropped", "            dsi[j] = scale * pi[j] * (dpi[j] - c);", "            dsi[j] = pi[j] * (dpi[j] - c);"),
    ("attn_query_index", "        const int64_t q = (row0 + r) % seq_len;      /* query position */",
     "        const int64_t q = r % seq_len;"),
    ("lse_max_not_added", "        out[i] = m + log(s);", "        out[i] = log(s);"),
    ("ce_loss_sign", "        row_loss[i] = valid ? lse - xi[t] : NAN;", "        row_loss[i] = valid ? lse + xi[t] : NAN;"),
    ("ce_loss_index", "        row_loss[i] = valid ? lse - xi[t] : NAN;", "        row_loss[i] = valid ? lse - xi[i % cols] : NAN;"),
    ("ce_onehot_sign", "(exp(xi[j] - m) / s - ((valid && j == t) ? 1.0 : 0.0))", "(exp(xi[j] - m) / s + ((valid && j == t) ? 1.0 : 0.0))"),
    ("ce_grad_scale_dropped", "            gi[j] = grad_scale * (exp", "            gi[j] = (exp"),
    ("mean_divisor", "    return s / (double)n;", "    return s / (double)(n + 1);"),
    ("ln_unbiased_variance", "        v /= (double)cols;", "        v /= (double)(cols - 1);"),
    ("ln_eps_outside_sqrt", "        const double r = 1.0 / sqrt(v + eps);", "        const double r = 1.0 / (sqrt(v) + eps);"),
    ("ln_beta_dropped", "            oi[j] = gamma[j] * hi[j] + beta[j];", "            oi[j] = gamma[j] * hi[j];"),
    ("ln_bwd_sign", "            dxi[j] = inv_std[i] * (gi[j] * gamma[j] - a - hi[j] * b);",
     "            dxi[j] = inv_std[i] * (gi[j] * gamma[j] - a + hi[j] * b);"),
    ("ln_bwd_gamma_dropped_in_b", "            b += gi[k] * gamma[k] * hi[k];", "            b += gi[k] * hi[k];"),
    ("ln_bwd_mean_term_dropped", "(gi[j] * gamma[j] - a - hi[j] * b)", "(gi[j] * gamma[j] - hi[j] * b)"),
    ("ln_dgamma_operand", "            dgamma[j] += g[i * cols + j] * xhat[i * cols + j];", "            dgamma[j] += g[i * cols + j];"),
    ("ln_dbeta_transposed", "            dbeta[j] += g[i * cols + j];", "            dbeta[j] += g[j * cols + i % cols];"),
    ("masked_max_over_all", "            if (mi[j] != 0) {\n                m = fmax(m, xi[j]);", "            if (1) {\n                m = fmax(m, xi[j]);"),
    ("masked_blocked_in_sum", "            if (mi[k] != 0)\n                s += exp(xi[k] - m);", "            s += exp(xi[k] - m);"),
    ("masked_empty_row_nan", "                ++allowed;\n            }\n        if (allowed == 0) {\n            for (int64_t j = 0; j < cols; ++j)\n                yi[j] = 0.0;\n            continue;\n        }\n        double s = 0.0;\n        for (int64_t k = 0; k < cols; ++k)\n            if (mi[k] != 0)\n",
     "                ++allowed;\n            }\n        if (allowed == 0) {\n            for (int64_t j = 0; j < cols; ++j)\n                yi[j] = NAN;\n            continue;\n        }\n        double s = 0.0;\n        for (int64_t k = 0; k < cols; ++k)\n            if (mi[k] != 0)\n"),
    ("masked_blocked_negative_zero", "            yi[j] = mi[j] != 0 ? exp(xi[j] - m) / s : 0.0;",
     "            yi[j] = mi[j] != 0 ? exp(xi[j] - m) / s : -0.0;"),
    ("kept_tie_direction", "if (larger || (neither && j < i))", "if (larger || (neither && j > i))"),
    ("kept_ties_ignored", "if (larger || (neither && j < i))", "if (larger)"),
    ("kept_count_bound", "            kr[i] = beaten_by < k ? 1 : 0;", "            kr[i] = beaten_by <= k ? 1 : 0;"),
    ("top_k_tie_direction", "    return ia < ib; /* equal rank: lower column first */", "    return ia > ib;"),
    ("top_k_nan_below", "        a_above = na && !nb;\n        b_above = nb && !na;", "        a_above = nb && !na;\n        b_above = na && !nb;"),
    ("top_k_largest_flag_ignored", "        return largest ? a_above : b_above;", "        return a_above;"),
    ("top_k_index_column", "            indices[r * k + t] = (double)best;", "            indices[r * k + t] = (double)t;"),
    ("rms_eps_outside_sqrt", "        const double rms = sqrt(ss / (double)cols + eps);", "        const double rms = sqrt(ss / (double)cols) + eps;"),
    ("rms_mean_missing", "        const double rms = sqrt(ss / (double)cols + eps);", "        const double rms = sqrt(ss + eps);"),
    ("rms_bwd_r_squared", "            dx[i * cols + j] = (gi[j] * gamma[j] - xi[j] * s / (r * r)) / r;", "            dx[i * cols + j] = (gi[j] * gamma[j] - xi[j] * s / r) / r;"),
    ("rms_bwd_sign", "            dx[i * cols + j] = (gi[j] * gamma[j] - xi[j] * s / (r * r)) / r;", "            dx[i * cols + j] = (gi[j] * gamma[j] + xi[j] * s / (r * r)) / r;"),
    ("rms_terms_gamma", "            gamma_terms[i * cols + j] = gi[j] * xi[j] / r;", "            gamma_terms[i * cols + j] = gi[j] * gamma[j] * xi[j] / r;"),
    ("colsum_beta_dropped", "        out[j] = (beta == 0.0 ? 0.0 : beta * out[j]) + s;", "        out[j] = s;"),
    ("colsum_beta_reads_out", "        out[j] = (beta == 0.0 ? 0.0 : beta * out[j]) + s;", "        out[j] = beta * out[j] + s;"),
    ("lrp_sign", "            r_in[i * cols + j] = xi[j] * (ri[j] - yi[j] * s);", "            r_in[i * cols + j] = xi[j] * (ri[j] + yi[j] * s);"),
    ("lrp_y_dropped", "            r_in[i * cols + j] = xi[j] * (ri[j] - yi[j] * s);", "            r_in[i * cols + j] = xi[j] * (ri[j] - s);"),
    ("fmask_nonzero_test", "            if (mi[j] != 0.0) {\n                m = fmax(m, xi[j]);", "            if (mi[j] > 0.0) {\n                m = fmax(m, xi[j]);"),
    ("argmax_last_max", "                if (xr[i] > xr[j])\n                    exceeded = 1;", "                if (xr[i] >= xr[j] && i != j)\n                    exceeded = 1;"),
    ("softce_wsum_dropped", "            grad[i * cols + j] = grad_scale * (exp(xi[j] - m) / s * wsum - wi[j]);", "            grad[i * cols + j] = grad_scale * (exp(xi[j] - m) / s - wi[j]);"),
    ("softce_loss_sign", "            loss += wi[j] * (lse - xi[j]);", "            loss += wi[j] * (xi[j] - lse);"),
    ("teacher_swapped", "            grad[i * cols + j] = grad_scale * (exp(si[j] - ms) / ss - exp(ti[j] - mt) / st);", "            grad[i * cols + j] = grad_scale * (exp(ti[j] - mt) / st - exp(si[j] - ms) / ss);"),
    ("teacher_loss_student_weights", "            loss += exp(ti[j] - mt) / st * (lse - si[j]);", "            loss += exp(si[j] - ms) / ss * (lse - si[j]);"),
    ("kept_larger_or_equal", "                const int larger = xr[j] > xr[i];", "                const int larger = xr[j] >= xr[i];"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, source, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    c = tmp_path / "mutant.c"
    c.write_text(source.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(c), "-lm"])
    prev = oracle.swap_library(oracle.bind(str(so)))
    failed = []
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError, FloatingPointError, IndexError):
                failed.append(pin.__name__)
    finally:
        oracle.swap_library(prev)
    assert failed, f"no pin caught the planted mistake {name}"
