/*
 * rowops.h - C ABI of librowops, the GB300 (sm_103a) row-wise
 * normalise-and-reduce ops of a transformer training step.
 *
 * Every op works on row-major fp32 matrices of `rows` x `cols` with row stride
 * `cols` and launches hand-written CUDA kernels on the caller's stream.
 *
 * Common contract (applies to every entry point below):
 *   - Pointers are DEVICE pointers on the current CUDA device.  The caller owns
 *     every buffer (inputs, outputs and workspace); the library never allocates
 *     device memory and keeps no per-call state, so calls are reentrant.
 *   - Calls are asynchronous: they validate the arguments on the host, queue
 *     the kernel(s) on `stream` and return.  No call synchronises the device.
 *   - A NULL `stream` is the legacy default stream.
 *   - Return value: ROWOPS_OK, or the first error found.  Nothing is launched
 *     when an error is returned, except ROWOPS_ERR_CUDA, which reports a failed
 *     launch (the CUDA runtime's error after the launch).
 *   - rows == 0 is a successful no-op for every op (after the scalar
 *     parameters are checked), except rowops_column_sums, which still scales
 *     its output by beta.  Negative sizes, cols >= 2^31, and matrices of
 *     more than 2^60 elements are ROWOPS_ERR_SHAPE.
 *   - A pointer may be NULL only when the buffer it names is empty.
 *   - Buffers must not overlap unless the entry point says so
 *     (ROWOPS_ERR_ALIAS); overlap is checked by address range.
 *   - Every pointer must be aligned to its element type (4 bytes for float
 *     and int32_t, 8 for double, any for uint8_t); a pointer that is not is
 *     ROWOPS_ERR_ALIGN.  Beyond that any alignment is accepted: 16-byte
 *     aligned buffers with cols % 4 == 0 take the 128-bit vector path; others
 *     take scalar paths with the same results up to fp32 rounding order.
 *   - Reductions use a fixed order: repeated calls on the same inputs give
 *     bit-identical outputs.
 *
 * The definitions follow four API-documentation pages:
 *   [P1] pulsatrix HIPBackend class reference
 *   [P2] MicroGPT CuBLASBackend API page
 *   [P3] TorchLean NN.Runtime.Autograd.Engine.LibTorch.Kernels (CUDA buffer kernels FFI)
 *   [P4] oxicuda-backend ComputeBackend trait
 */
#ifndef ROWOPS_H
#define ROWOPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ROWOPS_OK = 0,
    ROWOPS_ERR_NULL = 1,      /* a required pointer is NULL */
    ROWOPS_ERR_SHAPE = 2,     /* bad size, k, seq_len, scale, eps or grad_scale */
    ROWOPS_ERR_ALIAS = 3,     /* buffers overlap where the op forbids it */
    ROWOPS_ERR_WORKSPACE = 4, /* workspace missing, misaligned or too small */
    ROWOPS_ERR_CUDA = 5,      /* the CUDA runtime reported an error at launch */
    ROWOPS_ERR_ALIGN = 6      /* a pointer is not aligned to its element type */
} rowops_status;

/* Same object as cudaStream_t. */
typedef struct CUstream_st *rowops_stream;

/* Human-readable name of a status code (static string, never NULL). */
const char *rowops_status_string(int status);

/* Number of kernels this library has queued since it was loaded (all devices,
 * all threads).  Diagnostic counter for benchmarks. */
uint64_t rowops_kernel_launches(void);

/* Number of times a pipelined kernel of this library gave up a bounded wait on
 * the current device since the library was loaded (0 in correct operation; a
 * kernel that gives up leaves its outputs incomplete).  Synchronous: copies a
 * counter from the device; returns 0xffffffff if the copy fails. */
uint32_t rowops_pipeline_timeouts(void);

/*
 * Row softmax, max-subtracted.  [P1] softmax_rows(in, out, rows, cols); [P2]
 * softmax_rows(x); [P4] softmax(..., axis) on the last axis.
 *   y_ij = exp(x_ij - m_i) / sum_k exp(x_ik - m_i),  m_i = max_k x_ik.
 * x, y: rows x cols.  y may be exactly x (in place, as [P1] allows); any other
 * overlap is ROWOPS_ERR_ALIAS.  cols == 0 is a no-op ([P3]'s softmax accepts
 * empty tensors).
 */
int rowops_softmax_fwd(const float *x, float *y, int64_t rows, int64_t cols,
                       rowops_stream stream);

/*
 * Softmax backward from the output.  [P1] softmax_rows_backward(y, dy, dx, ...);
 * [P2] softmax_backward(s, ds).
 *   dx_ij = y_ij * (dy_ij - sum_k y_ik * dy_ik).
 * y, dy, dx: rows x cols.  dx must not overlap y or dy ([P1]).  cols == 0 is a
 * no-op.
 */
int rowops_softmax_bwd(const float *y, const float *dy, float *dx, int64_t rows, int64_t cols,
                       rowops_stream stream);

/*
 * Scaled causal attention softmax.  [P2] fused_attn_softmax(scores, scale) on the
 * stacked (batch*heads*seq_len, seq_len) score rows of
 * causal_mask_batched(scores, seq_len): row r is query i = r mod seq_len and
 *   p_rj = exp(scale*s_rj - m_r) / sum_{k<=i} exp(scale*s_rk - m_r)  for j <= i,
 *   p_rj = 0 (exactly +0.0)                                       for j > i,
 * with m_r = max_{k<=i} scale*s_rk.  Only the entries j <= i of `scores` are
 * read.  Requires seq_len >= 1, cols == seq_len, rows % seq_len == 0 and
 * 0 < scale < inf (else ROWOPS_ERR_SHAPE).  p must not overlap scores.
 */
int rowops_attn_softmax_fwd(const float *scores, float *p, int64_t rows, int64_t cols,
                            int64_t seq_len, float scale, rowops_stream stream);

/*
 * Backward of rowops_attn_softmax_fwd with respect to the raw scores, from its
 * output p.  [P2] fused_attn_softmax_backward(s, ds, scale).
 *   c_r = sum_{k<=i} p_rk dp_rk,  ds_rj = scale * p_rj * (dp_rj - c_r) for j <= i,
 *   ds_rj = 0 (exactly +0.0) for j > i.
 * Only the entries j <= i of p and dp are read.  Same shape rules as the
 * forward.  ds must not overlap p or dp.
 */
int rowops_attn_softmax_bwd(const float *p, const float *dp, float *ds, int64_t rows,
                            int64_t cols, int64_t seq_len, float scale, rowops_stream stream);

/*
 * Hard-masked row softmax.  [P3] stable row-wise hard-masked softmax.
 *   A_i = { j : mask_ij != 0 },  y_ij = exp(x_ij - max_{A_i} x) / sum_{A_i} exp(.)
 *   for j in A_i;  y_ij = +0.0 for j not in A_i;  a row with empty A_i is all +0.0.
 * x, y: rows x cols fp32; mask: rows x cols bytes, any nonzero byte allows.  y may
 * be exactly x; any other overlap (with x or mask) is ROWOPS_ERR_ALIAS.  cols == 0
 * is a no-op.
 */
int rowops_masked_softmax(const float *x, const uint8_t *mask, float *y, int64_t rows,
                          int64_t cols, rowops_stream stream);

/*
 * Per-row log-sum-exp, max-subtracted.  [P1] logsumexp_rows(in, out, rows, cols).
 *   lse_i = m_i + log sum_j exp(x_ij - m_i).
 * x: rows x cols; lse: rows.  cols == 0 writes -inf (log of an empty sum); a row
 * whose maximum is +-inf gets that maximum.  lse must not overlap x.
 */
int rowops_logsumexp(const float *x, float *lse, int64_t rows, int64_t cols,
                     rowops_stream stream);

/*
 * Fused softmax cross-entropy loss and logits gradient for integer targets.
 * [P2] fused_softmax_ce_grad(logits, targets) -> (Float64 loss, grad).
 *   loss_i = lse_i - x_{i,t_i}
 *   grad_ij = grad_scale * (softmax(x_i)_j - [j == t_i])
 *   *mean_loss = (1/rows) * sum_i loss_i   (fixed summation order; summed as a
 *   double-word fp32 value, about 48 significant bits, and returned as a double;
 *   a sum that is not finite in that form is redone in double)
 * logits, grad: rows x cols fp32; targets: rows int32; row_loss: rows fp32
 * (written, then reduced into the mean); mean_loss: ONE double in device memory.
 * grad_scale = 1/rows gives the gradient of the mean loss.  A target outside
 * [0, cols) cannot be checked without a device sync, so it is defined instead:
 * that row's row_loss is NaN (hence *mean_loss is NaN) and its gradient row is
 * grad_scale * softmax with no one-hot term.  cols == 0 and a non-finite
 * grad_scale are ROWOPS_ERR_SHAPE.  No output may overlap another buffer.
 */
int rowops_softmax_ce(const float *logits, const int32_t *targets, float *grad,
                      float *row_loss, double *mean_loss, int64_t rows, int64_t cols,
                      float grad_scale, rowops_stream stream);

/*
 * LayerNorm forward over the columns.  [P1] layer_norm_forward(); [P2]
 * layer_norm_forward(x, gamma, beta); [P3] layer normalisation returning
 * (output, normalized, invStd).
 *   mu_i = mean_j x_ij,  v_i = mean_j (x_ij - mu_i)^2 (population variance),
 *   inv_std_i = 1/sqrt(v_i + eps),  xhat_ij = (x_ij - mu_i) * inv_std_i,
 *   out_ij = gamma_j * xhat_ij + beta_j.
 * x, out, xhat: rows x cols; gamma, beta: cols; inv_std: rows.  cols == 0,
 * eps < 0 or non-finite eps are ROWOPS_ERR_SHAPE.  No output may overlap another
 * buffer.
 */
int rowops_layernorm_fwd(const float *x, const float *gamma, const float *beta, float *out,
                         float *xhat, float *inv_std, int64_t rows, int64_t cols, float eps,
                         rowops_stream stream);

/* Bytes of device workspace rowops_layernorm_bwd needs for this shape (a pure
 * function of rows and cols; 0 when rows or cols is 0 or negative). */
size_t rowops_layernorm_bwd_workspace(int64_t rows, int64_t cols);

/*
 * LayerNorm backward.  [P3] layer-normalisation VJP returning (dX, dGamma,
 * dBeta); [P2] layer_norm_backward(grad, norm, std_inv, gamma); [P1]
 * layer_norm_backward() for dX and column_sums() for the parameter sums.
 *   g'_ij = dy_ij * gamma_j
 *   dx_ij = inv_std_i * (g'_ij - mean_k g'_ik - xhat_ij * mean_k (g'_ik xhat_ik))
 *   dgamma_j = sum_i dy_ij * xhat_ij,   dbeta_j = sum_i dy_ij   (overwritten)
 * dy, xhat, dx: rows x cols; gamma, dgamma, dbeta: cols; inv_std: rows.  The
 * column sums are deterministic: fixed blocks of rows write partial sums into
 * `workspace` (at least rowops_layernorm_bwd_workspace(rows, cols) bytes of
 * 16-byte aligned device memory; its contents need not be initialised and are
 * garbage afterwards), then a second kernel, a programmatic dependent of the
 * first, adds the partials in a fixed order.  The workspace size depends on
 * rows, cols and the current device's SM count (the partials are per CTA or
 * per cluster of a grid sized to one wave); query it with the device current
 * that will run the call.  Concurrent calls need separate workspaces.
 * cols == 0 is ROWOPS_ERR_SHAPE; a short, NULL or misaligned workspace is
 * ROWOPS_ERR_WORKSPACE.  No output may overlap another buffer.  Rows of
 * 384..1024 floats whose CTA blocks are too large for shared memory stream
 * through a bulk-copy ring whose waits are bounded: a wait that runs out (a
 * defect) leaves dx, dgamma and dbeta incomplete and counts one timeout, so
 * callers that must know check rowops_pipeline_timeouts() after
 * synchronizing.
 */
int rowops_layernorm_bwd(const float *dy, const float *gamma, const float *xhat,
                         const float *inv_std, float *dx, float *dgamma, float *dbeta,
                         int64_t rows, int64_t cols, void *workspace, size_t workspace_bytes,
                         rowops_stream stream);

/*
 * LayerNorm backward that allocates nothing and takes no workspace.  The pages
 * have no counterpart; this is a convenience of this library.
 *
 * Some callers cannot obtain device memory when they need this op: code that
 * runs under a fixed device-memory budget set aside up front, plugins whose
 * host framework owns every allocation and offers no scratch space, or code
 * that must not enter an allocator at all (inside an allocator's own
 * out-of-memory path, for instance).  For them this entry point computes
 * what rowops_layernorm_bwd computes (bit for bit wherever both run the same
 * CTA count; see below), with the same argument rules, using a workspace that
 * lives inside the library: a fixed array of
 * rowops_layernorm_bwd_noalloc_max_bytes() bytes (1 MiB) of device memory,
 * which every GPU that loads the library holds until the process exits.
 *
 *   - The first call on each device looks up that array's device address
 *     (with the device current); make that first call before any stream
 *     capture.  Later calls reuse the address for the life of the process, so
 *     a device reset (cudaDeviceReset) after the first call on that device is
 *     not supported.
 *   - Errors are reported in this order: the argument checks of
 *     rowops_layernorm_bwd (shape, NULL, alignment, overlap), then the size
 *     check below, then a failed address lookup (ROWOPS_ERR_CUDA).
 *   - Each CTA's partial sums take 8 * cols bytes.  Rows of up to 1024 floats
 *     fit for every row count: the launch uses only as many CTAs as the array
 *     holds partials for (rows of 863..1024 floats then run on fewer CTAs
 *     than rowops_layernorm_bwd uses where a CTA's rows fit in shared memory,
 *     so dgamma and dbeta are added in another order and dx may come from the
 *     other stage-1 kernel; both agree with rowops_layernorm_bwd within the
 *     parity bounds).  Wider rows fit while rows is small enough
 *     (e.g. 64 rows of 2048 floats, 8 rows of 16384); larger shapes are
 *     refused with ROWOPS_ERR_WORKSPACE.
 *   - All calls on a device share the one array, and it keeps the contents of
 *     the last call.  Nothing in it needs to start at zero: each call writes
 *     every partial sum it later reads.  Calls that can overlap on the GPU
 *     (different streams, no ordering between them) race on the array and may
 *     return wrong dgamma/dbeta; order them, or use rowops_layernorm_bwd with
 *     separate workspaces.
 *   - Bounded waits that run out are counted as for rowops_layernorm_bwd:
 *     check rowops_pipeline_timeouts() after synchronizing.
 *   - It never calls cudaMalloc, cudaFree or any other allocating routine.
 */
int rowops_layernorm_bwd_noalloc(const float *dy, const float *gamma, const float *xhat,
                                 const float *inv_std, float *dx, float *dgamma, float *dbeta,
                                 int64_t rows, int64_t cols, rowops_stream stream);

/* Size in bytes of the array rowops_layernorm_bwd_noalloc uses (1 MiB). */
size_t rowops_layernorm_bwd_noalloc_max_bytes(void);

/*
 * Top-k kept mask.  [P3] kept mask (Spec.MoE.kept): entry i of a row is kept
 * when fewer than k entries of the row beat it; entry j beats entry i when
 * x_j > x_i, or when neither is larger and j < i.
 *   kept_ij = 1.0f if #{ j' : j' beats j } < k, else 0.0f.
 * The result is exact (comparisons and counts only) and equals the literal
 * compare-and-count for every input, NaN included (a NaN is neither larger nor
 * smaller than anything, so it ties).  x, kept: rows x cols fp32.  Requires
 * 1 <= k <= cols ([P1] top_k_rows precondition), else ROWOPS_ERR_SHAPE.  kept
 * must not overlap x.
 */
int rowops_topk_kept(const float *x, float *kept, int64_t rows, int64_t cols, int64_t k,
                     rowops_stream stream);

/*
 * Fused MoE router: hard-masked softmax and the top-k kept mask of its output in
 * one pass.  [P3] hard-masked softmax followed by [P3] kept mask (Spec.MoE.kept)
 * on the probabilities.
 *   p = rowops_masked_softmax(x, mask);  kept = rowops_topk_kept(p, k)
 * computed together: p is stored and the mask is decided on the same fp32
 * values, so both outputs equal the two separate calls bit for bit, while p is
 * never read back (13 instead of 17 bytes of HBM traffic per element).
 * x, p, kept: rows x cols fp32; mask: rows x cols bytes.  p may be exactly x;
 * kept must not overlap x, mask or p.  1 <= k <= cols, else ROWOPS_ERR_SHAPE.
 */
int rowops_router_masked_topk(const float *x, const uint8_t *mask, float *p, float *kept,
                              int64_t rows, int64_t cols, int64_t k, rowops_stream stream);

/*
 * Per-row top k values and their columns.  [P1] top_k_rows(in, values, indices,
 * rows, cols, k, largest).
 *   values[i][r], indices[i][r]: the entry of row i ranked r (0-based) among the
 *   k largest (largest != 0) or smallest, its column as a whole-number float.
 * Rank order: NaN ranks above every number (first for largest, last for
 * smallest); equal values (NaNs among themselves, -0 with +0) keep the lower
 * column first.  The output values are the input's bits (sign of zero and NaN
 * payload kept).  x: rows x cols; values, indices: rows x k.  Requires
 * 1 <= k <= cols <= 2^24 ([P1] precondition), else ROWOPS_ERR_SHAPE.  Outputs
 * must not overlap x or each other.  Exact (selection only).
 */
int rowops_top_k_rows(const float *x, float *values, float *indices, int64_t rows, int64_t cols,
                      int64_t k, int largest, rowops_stream stream);

/*
 * RMSNorm forward.  [P1] rms_norm_forward(in, gamma, out, row_rms, rows, cols, eps).
 *   rms_i = sqrt(mean_j x_ij^2 + eps),  out_ij = gamma_j * x_ij / rms_i,
 *   row_rms_i = rms_i (the cached statistic).
 * x, out: rows x cols; gamma: cols; row_rms: rows.  cols == 0, eps < 0 or
 * non-finite eps are ROWOPS_ERR_SHAPE.  Outputs must not overlap inputs or each
 * other.
 */
int rowops_rmsnorm_fwd(const float *x, const float *gamma, float *out, float *row_rms, int64_t rows,
                       int64_t cols, float eps, rowops_stream stream);

/*
 * RMSNorm backward.  [P1] rms_norm_backward(grad_out, gamma, in, row_rms,
 * grad_in, gamma_terms, rows, cols).
 *   g'_ij = dy_ij * gamma_j,  dx_ij = (g'_ij - x_ij * mean_k(g'_ik x_ik) / rms_i^2) / rms_i,
 *   gamma_terms_ij = dy_ij * x_ij / rms_i
 * (gamma's gradient is rowops_column_sums(gamma_terms), as [P1] intends).
 * dy, x, dx, gamma_terms: rows x cols; gamma: cols; row_rms: rows.  cols == 0 is
 * ROWOPS_ERR_SHAPE.  Outputs must not overlap inputs or each other.
 */
int rowops_rmsnorm_bwd(const float *dy, const float *gamma, const float *x, const float *row_rms,
                       float *dx, float *gamma_terms, int64_t rows, int64_t cols,
                       rowops_stream stream);

/*
 * Column sums.  [P1] column_sums(in, out, rows, cols, beta).
 *   out_j = beta * out_j + sum_i in_ij;  beta == 0 does not read out.
 * in: rows x cols; out: cols.  Deterministic: fixed blocks of consecutive rows
 * are added in row order, then the blocks in block order (no workspace: a
 * thread-block cluster per 32-column tile).  Exception to the common contract:
 * rows == 0 still applies beta.  Non-finite beta is ROWOPS_ERR_SHAPE; out must not
 * overlap in ([P1]).
 */
int rowops_column_sums(const float *in, float *out, int64_t rows, int64_t cols, float beta,
                       rowops_stream stream);

/*
 * Hard-masked softmax with a floating-point mask.  [P3] hard-masked softmax: an
 * entry is allowed when its mask value is not zero (mask != 0.0f: -0.0 blocks,
 * NaN allows); otherwise exactly rowops_masked_softmax.  mask: rows x cols fp32.
 * y may be exactly x; any other overlap is ROWOPS_ERR_ALIAS.
 */
int rowops_masked_softmax_fmask(const float *x, const float *mask, float *y, int64_t rows,
                                int64_t cols, rowops_stream stream);

/*
 * Softmax relevance rule.  [P1] lrp_softmax_rows(x, y, r, r_in, rows, cols):
 *   r_in_ij = x_ij * (r_ij - y_ij * sum_k r_ik).
 * x, y, r, r_in: rows x cols (y is the softmax output).  r_in must not overlap the
 * inputs.  cols == 0 is a no-op.
 */
int rowops_lrp_softmax_rows(const float *x, const float *y, const float *r, float *r_in,
                            int64_t rows, int64_t cols, rowops_stream stream);

/*
 * First-max one-hot.  [P3]: 1.0f at the first maximal coordinate of each
 * nonempty row and 0.0f elsewhere (the input dtype).  A coordinate is maximal
 * when no entry is larger than it, so a NaN is maximal and, without NaN, this is
 * the first index of the maximum.  x, out: rows x cols; out must not overlap x.
 * cols == 0 is a no-op (empty rows give an empty result).
 */
int rowops_argmax_onehot(const float *x, float *out, int64_t rows, int64_t cols,
                         rowops_stream stream);

/*
 * Weighted-logits (soft-target) cross-entropy.  [P3] mean weighted-logits
 * cross-entropy, read as cross-entropy against a weight row, with every
 * log-probability taken from the original logits (x - lse) so that a weighted
 * term whose probability underflows stays finite:
 *   loss_i = sum_j w_ij (lse_i - x_ij),  *mean_loss = (1/rows) sum_i loss_i,
 *   grad_ij = grad_scale * (softmax(x_i)_j * sum_k w_ik - w_ij).
 * A one-hot w gives rowops_softmax_ce.  logits, weights, grad: rows x cols;
 * row_loss: rows; mean_loss: one device double.  cols == 0 or non-finite
 * grad_scale is ROWOPS_ERR_SHAPE; outputs must not overlap inputs or each other.
 */
int rowops_soft_ce(const float *logits, const float *weights, float *grad, float *row_loss,
                   double *mean_loss, int64_t rows, int64_t cols, float grad_scale,
                   rowops_stream stream);

/*
 * Fixed-teacher cross-entropy and the student gradient.  [P3] fixed-teacher mean
 * cross-entropy, or its student gradient: q = softmax(teacher) is a constant,
 *   loss_i = sum_j q_ij (lse(student)_i - student_ij),  mean over rows,
 *   grad_ij = grad_scale * (softmax(student_i)_j - q_ij)   (written when grad != NULL).
 * Shapes and rules as rowops_soft_ce; grad may be NULL (loss only).
 */
int rowops_teacher_ce(const float *student, const float *teacher, float *grad, float *row_loss,
                      double *mean_loss, int64_t rows, int64_t cols, float grad_scale,
                      rowops_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* ROWOPS_H */
