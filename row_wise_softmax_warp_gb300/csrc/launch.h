// launch.h - host-side glue between the C ABI (abi.cu) and the kernels.
//
// Each launch_* function queues the kernel(s) of one op on `stream` for
// arguments that abi.cu has already validated, and returns the CUDA error of
// the launch.  `vec4` says that every row-major matrix argument is 16-byte
// aligned with cols % 4 == 0 (and byte masks 4-byte aligned), which enables the
// 128-bit path.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace rowops {

// ------------------------------------------------------------ bookkeeping

void note_launches(int n);  // counts kernels queued (rowops_kernel_launches)
int sm_count();             // SMs of the current device (cached; 0 if unknown)

template <int L, int N, int V>
struct Geom {
    static constexpr int LANES = L;
    static constexpr int NV = N;
    static constexpr int VEC = V;
};

// Calls f(Geom<LANES, NV, VEC>{}) with the group geometry for rows of `cols`
// floats (see common.cuh), or returns false when a row is longer than one
// warp holds in registers (1024 floats, vectorised or scalar).  Scalar rows
// keep the floats per lane of vectorised rows of the same length (NV = 32
// scalars against NV = 8 float4s); groups of at least 8 lanes make each row's
// share of a warp load one full 32-byte sector.
template <typename F>
bool with_geometry(bool vec4, int64_t cols, F&& f) {
    if (vec4) {
        const int64_t nc = cols / 4;
        if (nc <= 4) f(Geom<4, 1, 4>{});
        else if (nc <= 8) f(Geom<4, 2, 4>{});
        else if (nc <= 16) f(Geom<8, 2, 4>{});
        else if (nc <= 32) f(Geom<16, 2, 4>{});
        else if (nc <= 64) f(Geom<32, 2, 4>{});
        else if (nc <= 128) f(Geom<32, 4, 4>{});
        else if (nc <= 192) f(Geom<32, 6, 4>{});
        else if (nc <= 256) f(Geom<32, 8, 4>{});
        else return false;
    } else {
        if (cols <= 4) f(Geom<4, 1, 1>{});
        else if (cols <= 8) f(Geom<8, 1, 1>{});
        else if (cols <= 16) f(Geom<8, 2, 1>{});
        else if (cols <= 32) f(Geom<8, 4, 1>{});
        else if (cols <= 64) f(Geom<8, 8, 1>{});
        else if (cols <= 128) f(Geom<16, 8, 1>{});
        else if (cols <= 256) f(Geom<32, 8, 1>{});
        else if (cols <= 512) f(Geom<32, 16, 1>{});
        else if (cols <= 768) f(Geom<32, 24, 1>{});
        else if (cols <= 1024) f(Geom<32, 32, 1>{});
        else return false;
    }
    return true;
}

// Blocks of 256 threads for a group kernel over `rows` rows (grid-stride
// beyond the cap).
inline unsigned group_grid(int64_t rows, int lanes) {
    const int64_t groups_per_block = 256 / lanes;
    int64_t b = (rows + groups_per_block - 1) / groups_per_block;
    if (b > (1 << 20)) b = 1 << 20;
    return static_cast<unsigned>(b < 1 ? 1 : b);
}

// Balanced launch for a group kernel whose block is any whole number of warps
// (up to 1024 threads, GPB = blockDim.x / LANES): one block per SM holding
// ceil(rows / SMs) groups, so no SM carries a block more than another (with
// 256-thread blocks, 4096 rows of 768 floats put 4 blocks on 56 SMs and 3 on
// the other 96).  threads = 0 when that block would be smaller than
// kBlockThreads-equivalent work or larger than 1024 threads (use group_grid).
struct BalancedLaunch {
    unsigned grid = 0, threads = 0;
};
inline BalancedLaunch balanced_groups(int64_t rows, int lanes) {
    BalancedLaunch b;
    const int sms = sm_count();
    if (sms <= 0 || rows <= 0) return b;
    const int64_t per_sm = (rows + sms - 1) / sms;  // groups per block
    const int64_t nt = (per_sm * lanes + 31) / 32 * 32;
    if (nt < 256 || nt > 1024) return b;
    b.grid = static_cast<unsigned>((rows + per_sm - 1) / per_sm);
    b.threads = static_cast<unsigned>(nt);
    return b;
}

// Blocks for a group kernel whose loop loads the next rows while it works on
// the current ones: at most `per_sm` blocks per SM, so each group walks several
// rows and its loads stay in flight across the selection work.
inline unsigned stream_grid(int64_t rows, int lanes, int per_sm = 8) {
    const unsigned g = group_grid(rows, lanes);
    const int sms = sm_count();
    const int64_t cap = int64_t(sms > 0 ? sms : 132) * per_sm;
    return int64_t(g) > cap ? static_cast<unsigned>(cap) : g;
}

// Blocks for a one-row-per-block (or per-cluster) kernel.
inline unsigned row_grid(int64_t rows, int per_row = 1) {
    int64_t b = rows;
    const int64_t cap = (int64_t(1) << 20);
    if (b > cap) b = cap;
    return static_cast<unsigned>((b < 1 ? 1 : b) * per_row);
}

// ----------------------------------------------------------------- ops

cudaError_t launch_softmax_fwd(const float* x, float* y, int64_t rows, int64_t cols, bool vec4,
                               cudaStream_t stream);
// TMA-streamed long rows (tma_rows.cu): rows of more than 1024 floats from
// 4-byte aligned buffers (an output row must share its input row's alignment
// modulo 16 bytes); each returns false, launching nothing, when the shape does
// not suit it (the row does not fit in shared memory where it must stay
// resident, or the alignments differ).
bool launch_lse_tma(const float* x, float* lse, int64_t rows, int64_t cols, cudaStream_t stream,
                    cudaError_t* err);
bool launch_ce_tma(const float* x, const int32_t* targets, float* grad, float* row_loss, int64_t rows,
                   int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err);
bool launch_softmax_tma(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t stream,
                        cudaError_t* err);
// Two-input long rows (weighted-logits and fixed-teacher CE): x and w must
// share their alignment modulo 16 bytes; grad (which may be NULL) may differ.
bool launch_soft_ce_tma(const float* x, const float* w, float* grad, float* row_loss, int64_t rows, int64_t cols,
                        float grad_scale, cudaStream_t stream, cudaError_t* err);
bool launch_teacher_ce_tma(const float* s, const float* t, float* grad, float* row_loss, int64_t rows,
                           int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err);
// Timeouts counted by the bounded waits of each bulk-copy translation unit
// (rowops_pipeline_timeouts adds them up).
uint32_t pipeline_timeouts_rows();
uint32_t pipeline_timeouts_pairs();
uint32_t pipeline_timeouts_ln();
// LayerNorm backward stage 1 on rows of 384..1024 floats on 16-byte
// boundaries through the bulk-copy ring (one CTA per SM, at most 2^17 / cols
// and at most max_ctas, 0: no further limit); writes
// ln_bwd_tma_ctas(rows, cols, max_ctas) partials to ws.
// ln_bwd_tma_ctas is 0 for shapes it does not take.
int64_t ln_bwd_tma_ctas(int64_t rows, int64_t cols, int64_t max_ctas);
bool launch_ln_bwd_tma(const float* dy, const float* gamma, const float* xhat, const float* inv_std, float* dx,
                       float* ws, int64_t rows, int64_t cols, int64_t max_ctas, cudaStream_t stream,
                       cudaError_t* err);
// Softmax backward on long rows (two passes through the ring); y and dy must
// share their alignment modulo 16 bytes.
bool launch_softmax_bwd_tma(const float* y, const float* dy, float* dx, int64_t rows, int64_t cols,
                            cudaStream_t stream, cudaError_t* err);
cudaError_t launch_softmax_bwd(const float* y, const float* dy, float* dx, int64_t rows,
                               int64_t cols, bool vec4, cudaStream_t stream);
cudaError_t launch_attn_fwd(const float* s, float* p, int64_t rows, int64_t cols, int64_t seq_len,
                            float scale, bool vec4, cudaStream_t stream);
cudaError_t launch_attn_bwd(const float* p, const float* dp, float* ds, int64_t rows,
                            int64_t cols, int64_t seq_len, float scale, bool vec4,
                            cudaStream_t stream);
cudaError_t launch_masked_softmax(const float* x, const uint8_t* mask, float* y, int64_t rows,
                                  int64_t cols, bool vec4, cudaStream_t stream);
cudaError_t launch_logsumexp(const float* x, float* lse, int64_t rows, int64_t cols, bool vec4,
                             cudaStream_t stream);
cudaError_t launch_softmax_ce(const float* logits, const int32_t* targets, float* grad,
                              float* row_loss, double* mean_loss, int64_t rows, int64_t cols,
                              float grad_scale, bool vec4, cudaStream_t stream);
cudaError_t launch_layernorm_fwd(const float* x, const float* gamma, const float* beta,
                                 float* out, float* xhat, float* inv_std, int64_t rows,
                                 int64_t cols, float eps, bool vec4, cudaStream_t stream);
// The argument checks of rowops_layernorm_bwd other than the workspace's
// (dimensions, null and misaligned pointers, overlaps of the inputs and
// outputs), in the order that entry point reports them; sets *vec4.
int layernorm_bwd_checks(const float* dy, const float* gamma, const float* xhat, const float* inv_std, float* dx,
                         float* dgamma, float* dbeta, int64_t rows, int64_t cols, bool* vec4);
// budget (bytes, 0: none) caps the workspace the launch may use: the
// allocation-free entry point passes the size of its fixed array.
size_t layernorm_bwd_workspace(int64_t rows, int64_t cols, size_t budget = 0);
cudaError_t launch_layernorm_bwd(const float* dy, const float* gamma, const float* xhat,
                                 const float* inv_std, float* dx, float* dgamma, float* dbeta,
                                 int64_t rows, int64_t cols, float* workspace, bool vec4,
                                 cudaStream_t stream, size_t budget = 0);
cudaError_t launch_router(const float* x, const uint8_t* mask, float* p, float* kept, int64_t rows,
                          int64_t cols, int64_t k, bool vec4, cudaStream_t stream);
cudaError_t launch_top_k_rows(const float* x, float* values, float* indices, int64_t rows, int64_t cols,
                              int64_t k, bool largest, bool vec4, cudaStream_t stream);
cudaError_t launch_rmsnorm_fwd(const float* x, const float* gamma, float* out, float* row_rms, int64_t rows,
                               int64_t cols, float eps, bool vec4, cudaStream_t stream);
cudaError_t launch_rmsnorm_bwd(const float* dy, const float* gamma, const float* x, const float* row_rms,
                               float* dx, float* terms, int64_t rows, int64_t cols, bool vec4,
                               cudaStream_t stream);
cudaError_t launch_column_sums(const float* in, float* out, int64_t rows, int64_t cols, float beta,
                               cudaStream_t stream);
cudaError_t launch_masked_softmax_fmask(const float* x, const float* mask, float* y, int64_t rows,
                                        int64_t cols, bool vec4, cudaStream_t stream);
cudaError_t launch_lrp_softmax(const float* x, const float* y, const float* r, float* r_in, int64_t rows,
                               int64_t cols, bool vec4, cudaStream_t stream);
cudaError_t launch_argmax_onehot(const float* x, float* out, int64_t rows, int64_t cols, bool vec4,
                                 cudaStream_t stream);
// Fixed-order mean of the row losses into one double (programmatic dependent).
cudaError_t launch_row_mean(const float* row_loss, int64_t rows, double* mean_loss, cudaStream_t stream);
cudaError_t launch_soft_ce(const float* x, const float* w, float* grad, float* row_loss, double* mean_loss,
                           int64_t rows, int64_t cols, float grad_scale, bool vec4, cudaStream_t stream);
cudaError_t launch_teacher_ce(const float* s, const float* t, float* grad, float* row_loss, double* mean_loss,
                              int64_t rows, int64_t cols, float grad_scale, bool vec4, cudaStream_t stream);
cudaError_t launch_topk_kept(const float* x, float* kept, int64_t rows, int64_t cols, int64_t k,
                             bool vec4, cudaStream_t stream);

}  // namespace rowops
