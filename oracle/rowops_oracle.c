/*
 * rowops_oracle.c - the CPU oracle for the row-wise normalise-and-reduce ops.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what each row op computes.  Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline leg load it; the CUDA library never links,
 * includes or calls it, and it shares no code with the CUDA path.
 *
 * Conventions
 *   - Every value is a C double.  Inputs arrive as doubles (callers widen the
 *     fp32 arrays exactly), so the arithmetic below is the definition evaluated
 *     in double precision.
 *   - Matrices are row-major (rows x cols) with row stride cols.
 *   - Every loop walks a row in increasing column index and every column sum
 *     walks rows in increasing row index; nothing is blocked, fused or reordered.
 *   - exp, log and sqrt are the host C library's double routines.
 *
 * Sources (documentation pages of four compute back ends; each function names
 * the member it follows):
 *   [P1] pulsatrix HIPBackend class reference
 *   [P2] MicroGPT CuBLASBackend API page
 *   [P3] TorchLean NN.Runtime.Autograd.Engine.LibTorch.Kernels (CUDA buffer
 *        kernels FFI)
 *   [P4] oxicuda-backend ComputeBackend trait
 *
 * Parity pins: every function here is pinned by tests that do not reuse its own
 * formula (closed forms, invariants, finite differences, brute force and
 * textbook library routines); no function lacks a pin.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* Largest entry of a row; -inf for an empty row.  fmax ignores a NaN operand. */
static double row_max(const double *x, int64_t n)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        m = fmax(m, x[j]);
    return m;
}

/*
 * [P1] softmax_rows(): row-wise softmax of a (rows x cols) matrix, with the row
 * maximum subtracted before exponentiation; [P2] softmax_rows(x); [P4]
 * softmax(input, output, shape, axis) along the last axis.
 *   m = max_j x_j,  y_j = exp(x_j - m) / sum_k exp(x_k - m).
 * cols == 0 leaves nothing to write ([P3]'s stable softmax accepts empty
 * tensors).
 */
void oracle_softmax_rows(const double *x, double *y, int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols;
        double *yi = y + i * cols;
        if (cols == 0)
            continue;
        const double m = row_max(xi, cols);
        double s = 0.0;
        for (int64_t k = 0; k < cols; ++k)
            s += exp(xi[k] - m);
        for (int64_t j = 0; j < cols; ++j)
            yi[j] = exp(xi[j] - m) / s;
    }
}

/*
 * [P1] softmax_rows_backward(): gradient from the softmax output y,
 *   dx_j = y_j * (dy_j - sum_k y_k * dy_k);
 * [P2] softmax_backward(s, ds) is the same map.
 */
void oracle_softmax_rows_backward(const double *y, const double *dy, double *dx,
                                  int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *yi = y + i * cols, *dyi = dy + i * cols;
        double *dxi = dx + i * cols;
        double c = 0.0;
        for (int64_t k = 0; k < cols; ++k)
            c += yi[k] * dyi[k];
        for (int64_t j = 0; j < cols; ++j)
            dxi[j] = yi[j] * (dyi[j] - c);
    }
}

/*
 * [P2] fused_attn_softmax(scores, scale): scaling, causal masking and softmax in one op, whose
 * default implementation is the composition of the separate ops; rows are the
 * stacked (batch * heads * seq_len, seq_len) score matrix of
 * causal_mask_batched(scores, seq_len), so row r holds query position
 * i = r mod seq_len, and the causal mask removes the keys j > i.
 *   z_j = scale * s_j            (every j)
 *   p_j = exp(z_j - max_{k<=i} z_k) / sum_{k<=i} exp(z_k - max)   for j <= i
 *   p_j = 0                                                       for j > i
 * row0 is the global index of the first row passed, so callers can hand the
 * oracle any contiguous block of rows.
 */
void oracle_attn_softmax_forward(const double *s, double *p, int64_t rows, int64_t cols,
                                 int64_t seq_len, int64_t row0, double scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *si = s + r * cols;
        double *pi = p + r * cols;
        const int64_t q = (row0 + r) % seq_len;      /* query position */
        const int64_t n = q + 1 < cols ? q + 1 : cols; /* keys 0..q survive the mask */
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j)
            m = fmax(m, scale * si[j]);
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j)
            sum += exp(scale * si[j] - m);
        for (int64_t j = 0; j < n; ++j)
            pi[j] = exp(scale * si[j] - m) / sum;
        for (int64_t j = n; j < cols; ++j)
            pi[j] = 0.0;
    }
}

/*
 * [P2] fused_attn_softmax_backward(s, ds, scale): the vector-Jacobian product of
 * the map above with respect to the raw scores, from its output p (the same
 * output-based form as [P1] softmax_rows_backward), times the chain-rule
 * factor scale:
 *   c = sum_{k<=i} p_k dp_k,  ds_j = scale * p_j * (dp_j - c)  (j <= i),
 *   ds_j = 0  (j > i).
 */
void oracle_attn_softmax_backward(const double *p, const double *dp, double *ds,
                                  int64_t rows, int64_t cols, int64_t seq_len,
                                  int64_t row0, double scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *pi = p + r * cols, *dpi = dp + r * cols;
        double *dsi = ds + r * cols;
        const int64_t q = (row0 + r) % seq_len;
        const int64_t n = q + 1 < cols ? q + 1 : cols;
        double c = 0.0;
        for (int64_t k = 0; k < n; ++k)
            c += pi[k] * dpi[k];
        for (int64_t j = 0; j < n; ++j)
            dsi[j] = scale * pi[j] * (dpi[j] - c);
        for (int64_t j = n; j < cols; ++j)
            dsi[j] = 0.0;
    }
}

/*
 * [P1] logsumexp_rows(): out_i = log sum_j exp(x_ij), evaluated with the row
 * maximum subtracted: m + log sum_j exp(x_ij - m).  An empty row is the log of
 * an empty sum, -inf; a row whose maximum is +-inf has that maximum as its value
 * (the limit of the definition; the subtraction would give inf - inf).
 */
void oracle_logsumexp_rows(const double *x, double *out, int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols;
        const double m = row_max(xi, cols);
        if (isinf(m)) {
            out[i] = m;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += exp(xi[j] - m);
        out[i] = m + log(s);
    }
}

/*
 * [P2] fused_softmax_ce_grad(logits, targets): softmax + cross-entropy loss +
 * logits gradient for integer targets.  Per row i with target t = targets[i]:
 *   lse_i  = m + log sum_j exp(x_ij - m)
 *   loss_i = lse_i - x_it
 *   g_ij   = grad_scale * (exp(x_ij - m) / sum_k exp(x_ik - m) - [j == t])
 * grad_scale is the factor of the gradient of whatever the caller reduces the
 * row losses to (1/rows for the mean loss).  A target outside [0, cols) has no
 * defined loss: its row_loss is NaN and its gradient row carries no one-hot term.
 */
void oracle_softmax_cross_entropy(const double *x, const int32_t *targets, double *grad,
                                  double *row_loss, int64_t rows, int64_t cols,
                                  double grad_scale)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols;
        double *gi = grad + i * cols;
        const double m = row_max(xi, cols);
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += exp(xi[j] - m);
        const double lse = m + log(s);
        const int64_t t = targets[i];
        const int valid = t >= 0 && t < cols;
        row_loss[i] = valid ? lse - xi[t] : NAN;
        for (int64_t j = 0; j < cols; ++j)
            gi[j] = grad_scale * (exp(xi[j] - m) / s - ((valid && j == t) ? 1.0 : 0.0));
    }
}

/* The mean loss returned by [P2] fused_softmax_ce_grad: (1/n) sum_i v_i, summed
 * in increasing i. */
double oracle_mean(const double *v, int64_t n)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        s += v[i];
    return s / (double)n;
}

/*
 * [P1] layer_norm_forward(): per row, xhat = (x - mean) / sqrt(var + eps),
 * out = gamma * xhat + beta; [P3] layer normalisation over the columns returning
 * (output, normalized, invStd); [P2] layer_norm_forward(x, gamma, beta).
 *   mu = (1/C) sum_j x_j,  v = (1/C) sum_j (x_j - mu)^2  (population variance),
 *   r  = 1 / sqrt(v + eps), xhat_j = (x_j - mu) * r, out_j = gamma_j xhat_j + beta_j.
 * The cached per-row statistic is r, the inverse standard deviation ([P3]
 * invStd, [P2] std_inv).
 */
void oracle_layernorm_forward(const double *x, const double *gamma, const double *beta,
                              double *out, double *xhat, double *inv_std,
                              int64_t rows, int64_t cols, double eps)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols;
        double *oi = out + i * cols, *hi = xhat + i * cols;
        double mu = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            mu += xi[j];
        mu /= (double)cols;
        double v = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            v += (xi[j] - mu) * (xi[j] - mu);
        v /= (double)cols;
        const double r = 1.0 / sqrt(v + eps);
        inv_std[i] = r;
        for (int64_t j = 0; j < cols; ++j) {
            hi[j] = (xi[j] - mu) * r;
            oi[j] = gamma[j] * hi[j] + beta[j];
        }
    }
}

/*
 * [P3] layer-normalisation VJP, dX part; [P1] layer_norm_backward() (input
 * gradient from the cached xhat and the per-row statistic); [P2]
 * layer_norm_backward(grad, norm, std_inv, gamma).
 * With g' = g * gamma, the derivative of the forward above with respect to x is
 *   dx_j = r * (g'_j - (1/C) sum_k g'_k - xhat_j * (1/C) sum_k g'_k xhat_k),
 * which follows from xhat = (x - mu) r and d r / d x_k = -r^3 (x_k - mu) / C.
 */
void oracle_layernorm_backward_input(const double *g, const double *gamma,
                                     const double *xhat, const double *inv_std,
                                     double *dx, int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *gi = g + i * cols, *hi = xhat + i * cols;
        double *dxi = dx + i * cols;
        double a = 0.0, b = 0.0;
        for (int64_t k = 0; k < cols; ++k) {
            a += gi[k] * gamma[k];
            b += gi[k] * gamma[k] * hi[k];
        }
        a /= (double)cols;
        b /= (double)cols;
        for (int64_t j = 0; j < cols; ++j)
            dxi[j] = inv_std[i] * (gi[j] * gamma[j] - a - hi[j] * b);
    }
}

/*
 * [P3] layer-normalisation VJP, dGamma and dBeta parts; the column reduction is
 * [P1] column_sums() with beta = 0 (rows summed in increasing i):
 *   dgamma_j = sum_i g_ij * xhat_ij,  dbeta_j = sum_i g_ij.
 * Both outputs are overwritten.
 */
void oracle_layernorm_backward_params(const double *g, const double *xhat,
                                      double *dgamma, double *dbeta,
                                      int64_t rows, int64_t cols)
{
    for (int64_t j = 0; j < cols; ++j) {
        dgamma[j] = 0.0;
        dbeta[j] = 0.0;
    }
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            dgamma[j] += g[i * cols + j] * xhat[i * cols + j];
            dbeta[j] += g[i * cols + j];
        }
}

/*
 * [P3] stable row-wise hard-masked softmax: the maximum and the denominator use
 * only entries whose mask value is nonzero; blocked entries are exactly zero; a
 * row with no allowed entry is all zeros.
 *   A = {j : mask_j != 0},  y_j = exp(x_j - max_A x) / sum_{k in A} exp(x_k - max_A x)
 *   for j in A, y_j = 0 otherwise.
 */
void oracle_masked_softmax(const double *x, const uint8_t *mask, double *y,
                           int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols;
        const uint8_t *mi = mask + i * cols;
        double *yi = y + i * cols;
        int64_t allowed = 0;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j)
            if (mi[j] != 0) {
                m = fmax(m, xi[j]);
                ++allowed;
            }
        if (allowed == 0) {
            for (int64_t j = 0; j < cols; ++j)
                yi[j] = 0.0;
            continue;
        }
        double s = 0.0;
        for (int64_t k = 0; k < cols; ++k)
            if (mi[k] != 0)
                s += exp(xi[k] - m);
        for (int64_t j = 0; j < cols; ++j)
            yi[j] = mi[j] != 0 ? exp(xi[j] - m) / s : 0.0;
    }
}

/*
 * [P3] top-k kept mask (Spec.MoE.kept): entry i of a row is kept (1) when fewer
 * than k entries of the row beat it, else 0; entry j beats entry i when it is
 * larger, or when neither is larger and j < i.  Compare and count, literally,
 * O(cols^2) per row.  With double inputs widened from fp32 the comparisons are
 * the fp32 comparisons (-0 equals +0; a NaN is larger than nothing and nothing
 * is larger than it).
 */
void oracle_topk_kept(const double *x, uint8_t *kept, int64_t rows, int64_t cols, int64_t k)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        uint8_t *kr = kept + r * cols;
        for (int64_t i = 0; i < cols; ++i) {
            int64_t beaten_by = 0;
            for (int64_t j = 0; j < cols; ++j) {
                const int larger = xr[j] > xr[i];
                const int neither = !(xr[j] > xr[i]) && !(xr[i] > xr[j]);
                if (larger || (neither && j < i))
                    ++beaten_by;
            }
            kr[i] = beaten_by < k ? 1 : 0;
        }
    }
}

/*
 * [P1] top_k_rows(in, values, indices, rows, cols, k, largest): per row, the k
 * largest (largest != 0) or smallest values in rank order, and their column
 * indices as whole-number floats.  Order: NaN ranks above every number (so it
 * comes first when selecting the largest and last when selecting the
 * smallest); equal values (all NaNs among themselves, and -0 with +0) keep the
 * lower column first.  Selection: k passes, each taking the best entry not yet
 * taken.
 */
static int ranks_before(double a, int64_t ia, double b, int64_t ib, int largest)
{
    const int na = isnan(a), nb = isnan(b);
    int a_above, b_above; /* in the value order, NaN above every number */
    if (na || nb) {
        a_above = na && !nb;
        b_above = nb && !na;
    } else {
        a_above = a > b;
        b_above = b > a;
    }
    if (a_above || b_above)
        return largest ? a_above : b_above;
    return ia < ib; /* equal rank: lower column first */
}

void oracle_top_k_rows(const double *x, double *values, double *indices, int64_t rows,
                       int64_t cols, int64_t k, int largest, unsigned char *taken)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        for (int64_t j = 0; j < cols; ++j)
            taken[j] = 0;
        for (int64_t t = 0; t < k; ++t) {
            int64_t best = -1;
            for (int64_t j = 0; j < cols; ++j)
                if (!taken[j] && (best < 0 || ranks_before(xr[j], j, xr[best], best, largest)))
                    best = j;
            taken[best] = 1;
            values[r * k + t] = xr[best];
            indices[r * k + t] = (double)best;
        }
    }
}

/*
 * [P1] rms_norm_forward(in, gamma, out, row_rms, rows, cols, eps):
 *   rms_i = sqrt((1/C) sum_j x_ij^2 + eps),  out_ij = gamma_j * x_ij / rms_i.
 * The cached per-row statistic is rms_i itself ([P1] row_rms).
 */
void oracle_rms_norm_forward(const double *x, const double *gamma, double *out, double *row_rms,
                             int64_t rows, int64_t cols, double eps)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols;
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            ss += xi[j] * xi[j];
        const double rms = sqrt(ss / (double)cols + eps);
        row_rms[i] = rms;
        for (int64_t j = 0; j < cols; ++j)
            out[i * cols + j] = gamma[j] * xi[j] / rms;
    }
}

/*
 * [P1] rms_norm_backward(grad_out, gamma, in, row_rms, grad_in, gamma_terms, ...):
 * input gradient of the forward above, plus the per-row contributions to gamma's
 * gradient, gamma_terms_ij = g_ij * x_ij / rms_i ([P1]: column_sums reduces them).
 * With g' = g * gamma, y_j = gamma_j x_j / r and d r / d x_k = x_k / (C r):
 *   dx_k = (1/r) * (g'_k - x_k * ((1/C) sum_j g'_j x_j) / r^2).
 */
void oracle_rms_norm_backward(const double *g, const double *gamma, const double *x,
                              const double *row_rms, double *dx, double *gamma_terms,
                              int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *gi = g + i * cols, *xi = x + i * cols;
        const double r = row_rms[i];
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += gi[j] * gamma[j] * xi[j];
        s /= (double)cols;
        for (int64_t j = 0; j < cols; ++j) {
            dx[i * cols + j] = (gi[j] * gamma[j] - xi[j] * s / (r * r)) / r;
            gamma_terms[i * cols + j] = gi[j] * xi[j] / r;
        }
    }
}

/*
 * [P1] column_sums(in, out, rows, cols, beta): out_j = beta * out_j + sum_i in_ij,
 * rows summed in increasing i.  beta == 0 does not read out (a NaN there does not
 * survive).
 */
void oracle_column_sums(const double *in, double *out, int64_t rows, int64_t cols, double beta)
{
    for (int64_t j = 0; j < cols; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < rows; ++i)
            s += in[i * cols + j];
        out[j] = (beta == 0.0 ? 0.0 : beta * out[j]) + s;
    }
}

/*
 * [P1] lrp_softmax_rows(x, y, r, r_in, rows, cols): the SoftmaxModule relevance
 * rule per row, r_in_j = x_j * (r_j - y_j * sum_k r_k).
 */
void oracle_lrp_softmax_rows(const double *x, const double *y, const double *r, double *r_in,
                             int64_t rows, int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols, *yi = y + i * cols, *ri = r + i * cols;
        double s = 0.0;
        for (int64_t k = 0; k < cols; ++k)
            s += ri[k];
        for (int64_t j = 0; j < cols; ++j)
            r_in[i * cols + j] = xi[j] * (ri[j] - yi[j] * s);
    }
}

/*
 * [P3] hard-masked softmax with a floating-point mask: an entry is allowed when
 * its mask value is not zero (mask != 0.0; -0.0 blocks, NaN allows); otherwise
 * as oracle_masked_softmax.
 */
void oracle_masked_softmax_fmask(const double *x, const double *mask, double *y, int64_t rows,
                                 int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols, *mi = mask + i * cols;
        double *yi = y + i * cols;
        int64_t allowed = 0;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j)
            if (mi[j] != 0.0) {
                m = fmax(m, xi[j]);
                ++allowed;
            }
        if (allowed == 0) {
            for (int64_t j = 0; j < cols; ++j)
                yi[j] = 0.0;
            continue;
        }
        double s = 0.0;
        for (int64_t k = 0; k < cols; ++k)
            if (mi[k] != 0.0)
                s += exp(xi[k] - m);
        for (int64_t j = 0; j < cols; ++j)
            yi[j] = mi[j] != 0.0 ? exp(xi[j] - m) / s : 0.0;
    }
}

/*
 * [P3] first-max one-hot: 1 at the first maximal coordinate of each nonempty row,
 * 0 elsewhere.  A coordinate is maximal when no entry of the row is larger than it
 * (x_i > x_j holds for no i); the first maximal coordinate is the lowest such j.
 * Without NaN this is the first index of the maximum; a NaN is never exceeded, so
 * it is maximal too.
 */
void oracle_argmax_onehot(const double *x, double *out, int64_t rows, int64_t cols)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        int64_t first = -1;
        for (int64_t j = 0; j < cols && first < 0; ++j) {
            int exceeded = 0;
            for (int64_t i = 0; i < cols; ++i)
                if (xr[i] > xr[j])
                    exceeded = 1;
            if (!exceeded)
                first = j;
        }
        for (int64_t j = 0; j < cols; ++j)
            out[r * cols + j] = j == first ? 1.0 : 0.0;
    }
}

/*
 * [P3] mean weighted-logits cross-entropy, read as cross-entropy against a
 * weight (soft-target) row: every term is weighted, and its log-probability is
 * taken from the original logits as x_j - lse, so a term whose probability
 * underflows still has a finite log-probability.
 *   lse_i = m + log sum_j exp(x_ij - m),  loss_i = sum_j w_ij * (lse_i - x_ij),
 *   g_ij = grad_scale * (p_ij * sum_k w_ik - w_ij),  p = softmax(x_i).
 * With a one-hot w this is oracle_softmax_cross_entropy.
 */
void oracle_soft_ce(const double *x, const double *w, double *grad, double *row_loss,
                    int64_t rows, int64_t cols, double grad_scale)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * cols, *wi = w + i * cols;
        const double m = row_max(xi, cols);
        double s = 0.0, wsum = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            s += exp(xi[j] - m);
            wsum += wi[j];
        }
        const double lse = m + log(s);
        double loss = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            loss += wi[j] * (lse - xi[j]);
        row_loss[i] = loss;
        for (int64_t j = 0; j < cols; ++j)
            grad[i * cols + j] = grad_scale * (exp(xi[j] - m) / s * wsum - wi[j]);
    }
}

/*
 * [P3] fixed-teacher mean cross-entropy and its student gradient: the teacher
 * distribution q = softmax(t) is a constant, and with p = softmax(s)
 *   loss_i = -sum_j q_ij log p_ij = sum_j q_ij (lse(s_i) - s_ij),
 *   g_ij = grad_scale * (p_ij - q_ij)        (gradient with respect to s).
 */
void oracle_teacher_ce(const double *s, const double *t, double *grad, double *row_loss,
                       int64_t rows, int64_t cols, double grad_scale)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *si = s + i * cols, *ti = t + i * cols;
        const double ms = row_max(si, cols), mt = row_max(ti, cols);
        double ss = 0.0, st = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            ss += exp(si[j] - ms);
            st += exp(ti[j] - mt);
        }
        const double lse = ms + log(ss);
        double loss = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            loss += exp(ti[j] - mt) / st * (lse - si[j]);
        row_loss[i] = loss;
        for (int64_t j = 0; j < cols; ++j)
            grad[i * cols + j] = grad_scale * (exp(si[j] - ms) / ss - exp(ti[j] - mt) / st);
    }
}
