// abi.cu - the extern "C" entry points of librowops (include/rowops.h).
//
// Each entry point validates its arguments on the host in a fixed order
// (sizes, scalar parameters, empty problem, NULL pointers, overlap), decides
// whether the 128-bit path applies, and hands over to the op's launcher.  No
// exception crosses this boundary and nothing here allocates or synchronises.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include <initializer_list>
#include <utility>

#include "rowops.h"
#include "launch.h"

namespace rowops {

static std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }

int sm_count() {
    // Per-device cache; concurrent first calls store the same value.
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace rowops

namespace {

using rowops::launch_attn_bwd;

struct Buf {
    const void* p;
    int64_t bytes;
};

bool overlap(Buf a, Buf b) {
    if (a.p == nullptr || b.p == nullptr || a.bytes <= 0 || b.bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + uint64_t(b.bytes) && b0 < a0 + uint64_t(a.bytes);
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

// Every pointer aligned to its element type (4 bytes for float and int32, 8 for
// double): the scalar paths need no more, and less would make the kernels'
// accesses misaligned on the GPU.
bool elems_aligned(std::initializer_list<std::pair<const void*, uintptr_t>> ps) {
    for (const auto& p : ps)
        if (!aligned(p.first, p.second)) return false;
    return true;
}

// rows, cols >= 0; cols < 2^31; rows*cols*8 bytes fits in int64.
int check_dims(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0 || cols > INT32_MAX) return ROWOPS_ERR_SHAPE;
    if (cols > 0 && rows > (INT64_MAX / 8) / cols) return ROWOPS_ERR_SHAPE;
    return ROWOPS_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? ROWOPS_OK : ROWOPS_ERR_CUDA; }

cudaStream_t st(rowops_stream s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

namespace rowops {

int layernorm_bwd_checks(const float* dy, const float* gamma, const float* xhat, const float* inv_std, float* dx,
                         float* dgamma, float* dbeta, int64_t rows, int64_t cols, bool* vec4) {
    if (int e = check_dims(rows, cols)) return e;
    if (cols == 0) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!dy || !gamma || !xhat || !inv_std || !dx || !dgamma || !dbeta) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{dy, 4}, {gamma, 4}, {xhat, 4}, {inv_std, 4}, {dx, 4}, {dgamma, 4}, {dbeta, 4}}))
        return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    const Buf in[4] = {{dy, n}, {gamma, cols * 4}, {xhat, n}, {inv_std, rows * 4}};
    const Buf o[3] = {{dx, n}, {dgamma, cols * 4}, {dbeta, cols * 4}};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 4; ++b)
            if (overlap(o[a], in[b])) return ROWOPS_ERR_ALIAS;
        for (int b = 0; b < 3; ++b)
            if (a != b && overlap(o[a], o[b])) return ROWOPS_ERR_ALIAS;
    }
    *vec4 = cols % 4 == 0 && aligned(dy, 16) && aligned(gamma, 16) && aligned(xhat, 16) && aligned(dx, 16);
    return ROWOPS_OK;
}

}  // namespace rowops

extern "C" {

const char* rowops_status_string(int status) {
    switch (status) {
        case ROWOPS_OK: return "ROWOPS_OK";
        case ROWOPS_ERR_NULL: return "ROWOPS_ERR_NULL: a required pointer is NULL";
        case ROWOPS_ERR_SHAPE: return "ROWOPS_ERR_SHAPE: invalid size or scalar parameter";
        case ROWOPS_ERR_ALIAS: return "ROWOPS_ERR_ALIAS: buffers overlap where the op forbids it";
        case ROWOPS_ERR_WORKSPACE: return "ROWOPS_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case ROWOPS_ERR_CUDA: return "ROWOPS_ERR_CUDA: the CUDA runtime reported a launch error";
        case ROWOPS_ERR_ALIGN: return "ROWOPS_ERR_ALIGN: a pointer is not aligned to its element type";
        default: return "ROWOPS: unknown status";
    }
}

uint64_t rowops_kernel_launches(void) { return rowops::g_launches.load(std::memory_order_relaxed); }

int rowops_softmax_fwd(const float* x, float* y, int64_t rows, int64_t cols, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0 || cols == 0) return ROWOPS_OK;
    if (!x || !y) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {y, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (static_cast<const void*>(x) != y && overlap({x, n}, {y, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(y, 16);
    return to_status(rowops::launch_softmax_fwd(x, y, rows, cols, vec4, st(stream)));
}

int rowops_softmax_bwd(const float* y, const float* dy, float* dx, int64_t rows, int64_t cols,
                       rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0 || cols == 0) return ROWOPS_OK;
    if (!y || !dy || !dx) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{y, 4}, {dy, 4}, {dx, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (overlap({dx, n}, {y, n}) || overlap({dx, n}, {dy, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(y, 16) && aligned(dy, 16) && aligned(dx, 16);
    return to_status(rowops::launch_softmax_bwd(y, dy, dx, rows, cols, vec4, st(stream)));
}

static int check_attn(int64_t rows, int64_t cols, int64_t seq_len, float scale) {
    if (int e = check_dims(rows, cols)) return e;
    if (seq_len < 1 || cols != seq_len || rows % seq_len != 0) return ROWOPS_ERR_SHAPE;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ROWOPS_ERR_SHAPE;
    return ROWOPS_OK;
}

int rowops_attn_softmax_fwd(const float* scores, float* p, int64_t rows, int64_t cols,
                            int64_t seq_len, float scale, rowops_stream stream) {
    if (int e = check_attn(rows, cols, seq_len, scale)) return e;
    if (rows == 0) return ROWOPS_OK;
    if (!scores || !p) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{scores, 4}, {p, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (overlap({scores, n}, {p, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(scores, 16) && aligned(p, 16);
    return to_status(rowops::launch_attn_fwd(scores, p, rows, cols, seq_len, scale, vec4, st(stream)));
}

int rowops_attn_softmax_bwd(const float* p, const float* dp, float* ds, int64_t rows, int64_t cols,
                            int64_t seq_len, float scale, rowops_stream stream) {
    if (int e = check_attn(rows, cols, seq_len, scale)) return e;
    if (rows == 0) return ROWOPS_OK;
    if (!p || !dp || !ds) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{p, 4}, {dp, 4}, {ds, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (overlap({ds, n}, {p, n}) || overlap({ds, n}, {dp, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(p, 16) && aligned(dp, 16) && aligned(ds, 16);
    return to_status(launch_attn_bwd(p, dp, ds, rows, cols, seq_len, scale, vec4, st(stream)));
}

int rowops_masked_softmax(const float* x, const uint8_t* mask, float* y, int64_t rows, int64_t cols,
                          rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0 || cols == 0) return ROWOPS_OK;
    if (!x || !mask || !y) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {y, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (static_cast<const void*>(x) != y && overlap({x, n}, {y, n})) return ROWOPS_ERR_ALIAS;
    if (overlap({mask, rows * cols}, {y, n}) || overlap({mask, rows * cols}, {x, n}))
        return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(y, 16) && aligned(mask, 4);
    return to_status(rowops::launch_masked_softmax(x, mask, y, rows, cols, vec4, st(stream)));
}

int rowops_logsumexp(const float* x, float* lse, int64_t rows, int64_t cols, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0) return ROWOPS_OK;
    if (!lse || (cols > 0 && !x)) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {lse, 4}})) return ROWOPS_ERR_ALIGN;
    if (overlap({x, rows * cols * 4}, {lse, rows * 4})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16);
    return to_status(rowops::launch_logsumexp(x, lse, rows, cols, vec4, st(stream)));
}

int rowops_softmax_ce(const float* logits, const int32_t* targets, float* grad, float* row_loss,
                      double* mean_loss, int64_t rows, int64_t cols, float grad_scale,
                      rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (cols == 0 || !std::isfinite(grad_scale)) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!logits || !targets || !grad || !row_loss || !mean_loss) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{logits, 4}, {targets, 4}, {grad, 4}, {row_loss, 4}, {mean_loss, 8}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    const Buf in[2] = {{logits, n}, {targets, rows * 4}};
    const Buf out[3] = {{grad, n}, {row_loss, rows * 4}, {mean_loss, 8}};
    for (const Buf& o : out) {
        for (const Buf& i : in)
            if (overlap(o, i)) return ROWOPS_ERR_ALIAS;
        for (const Buf& o2 : out)
            if (&o != &o2 && overlap(o, o2)) return ROWOPS_ERR_ALIAS;
    }
    const bool vec4 = cols % 4 == 0 && aligned(logits, 16) && aligned(grad, 16);
    return to_status(rowops::launch_softmax_ce(logits, targets, grad, row_loss, mean_loss, rows, cols,
                                               grad_scale, vec4, st(stream)));
}

int rowops_layernorm_fwd(const float* x, const float* gamma, const float* beta, float* out,
                         float* xhat, float* inv_std, int64_t rows, int64_t cols, float eps,
                         rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (cols == 0 || !std::isfinite(eps) || eps < 0.f) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!x || !gamma || !beta || !out || !xhat || !inv_std) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {gamma, 4}, {beta, 4}, {out, 4}, {xhat, 4}, {inv_std, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    const Buf in[3] = {{x, n}, {gamma, cols * 4}, {beta, cols * 4}};
    const Buf o[3] = {{out, n}, {xhat, n}, {inv_std, rows * 4}};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 3; ++b)
            if (overlap(o[a], in[b]) || (a != b && overlap(o[a], o[b]))) return ROWOPS_ERR_ALIAS;
    }
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(gamma, 16) && aligned(beta, 16) &&
                      aligned(out, 16) && aligned(xhat, 16);
    return to_status(rowops::launch_layernorm_fwd(x, gamma, beta, out, xhat, inv_std, rows, cols, eps,
                                                  vec4, st(stream)));
}

size_t rowops_layernorm_bwd_workspace(int64_t rows, int64_t cols) {
    if (check_dims(rows, cols) != ROWOPS_OK) return 0;
    return rowops::layernorm_bwd_workspace(rows, cols);
}

int rowops_layernorm_bwd(const float* dy, const float* gamma, const float* xhat,
                         const float* inv_std, float* dx, float* dgamma, float* dbeta,
                         int64_t rows, int64_t cols, void* workspace, size_t workspace_bytes,
                         rowops_stream stream) {
    bool vec4 = false;
    if (int e = rowops::layernorm_bwd_checks(dy, gamma, xhat, inv_std, dx, dgamma, dbeta, rows, cols, &vec4))
        return e;
    if (rows == 0) return ROWOPS_OK;
    const size_t need = rowops::layernorm_bwd_workspace(rows, cols);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return ROWOPS_ERR_WORKSPACE;
    const int64_t n = rows * cols * 4;
    const Buf w{workspace, int64_t(need)};
    const Buf all[7] = {{dy, n}, {gamma, cols * 4}, {xhat, n}, {inv_std, rows * 4},
                        {dx, n}, {dgamma, cols * 4}, {dbeta, cols * 4}};
    for (const Buf& b : all)
        if (overlap(w, b)) return ROWOPS_ERR_ALIAS;
    return to_status(rowops::launch_layernorm_bwd(dy, gamma, xhat, inv_std, dx, dgamma, dbeta, rows,
                                                  cols, static_cast<float*>(workspace), vec4,
                                                  st(stream)));
}

int rowops_topk_kept(const float* x, float* kept, int64_t rows, int64_t cols, int64_t k,
                     rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (k < 1 || k > cols) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!x || !kept) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {kept, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (overlap({x, n}, {kept, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(kept, 16);
    return to_status(rowops::launch_topk_kept(x, kept, rows, cols, k, vec4, st(stream)));
}

int rowops_router_masked_topk(const float* x, const uint8_t* mask, float* p, float* kept, int64_t rows,
                              int64_t cols, int64_t k, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (k < 1 || k > cols) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!x || !mask || !p || !kept) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {p, 4}, {kept, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (static_cast<const void*>(x) != p && overlap({x, n}, {p, n})) return ROWOPS_ERR_ALIAS;
    if (overlap({mask, rows * cols}, {p, n}) || overlap({mask, rows * cols}, {x, n}) ||
        overlap({kept, n}, {x, n}) || overlap({kept, n}, {p, n}) || overlap({kept, n}, {mask, rows * cols}))
        return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(p, 16) && aligned(kept, 16) &&
                      aligned(mask, 4);
    return to_status(rowops::launch_router(x, mask, p, kept, rows, cols, k, vec4, st(stream)));
}

int rowops_top_k_rows(const float* x, float* values, float* indices, int64_t rows, int64_t cols,
                      int64_t k, int largest, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (k < 1 || k > cols || cols > (int64_t(1) << 24)) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!x || !values || !indices) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {values, 4}, {indices, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4, nk = rows * k * 4;
    if (overlap({values, nk}, {x, n}) || overlap({indices, nk}, {x, n}) ||
        overlap({values, nk}, {indices, nk}))
        return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16);
    return to_status(rowops::launch_top_k_rows(x, values, indices, rows, cols, k, largest != 0, vec4,
                                               st(stream)));
}

int rowops_rmsnorm_fwd(const float* x, const float* gamma, float* out, float* row_rms, int64_t rows,
                       int64_t cols, float eps, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (cols == 0 || !std::isfinite(eps) || eps < 0.f) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!x || !gamma || !out || !row_rms) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {gamma, 4}, {out, 4}, {row_rms, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    const Buf in[2] = {{x, n}, {gamma, cols * 4}};
    const Buf o[2] = {{out, n}, {row_rms, rows * 4}};
    for (int a = 0; a < 2; ++a)
        for (int b = 0; b < 2; ++b)
            if (overlap(o[a], in[b]) || (a != b && overlap(o[a], o[b]))) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(gamma, 16) && aligned(out, 16);
    return to_status(rowops::launch_rmsnorm_fwd(x, gamma, out, row_rms, rows, cols, eps, vec4, st(stream)));
}

int rowops_rmsnorm_bwd(const float* dy, const float* gamma, const float* x, const float* row_rms, float* dx,
                       float* gamma_terms, int64_t rows, int64_t cols, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (cols == 0) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return ROWOPS_OK;
    if (!dy || !gamma || !x || !row_rms || !dx || !gamma_terms) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{dy, 4}, {gamma, 4}, {x, 4}, {row_rms, 4}, {dx, 4}, {gamma_terms, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    const Buf in[4] = {{dy, n}, {gamma, cols * 4}, {x, n}, {row_rms, rows * 4}};
    const Buf o[2] = {{dx, n}, {gamma_terms, n}};
    for (int a = 0; a < 2; ++a) {
        for (int b = 0; b < 4; ++b)
            if (overlap(o[a], in[b])) return ROWOPS_ERR_ALIAS;
    }
    if (overlap(o[0], o[1])) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(dy, 16) && aligned(gamma, 16) && aligned(x, 16) &&
                      aligned(dx, 16) && aligned(gamma_terms, 16);
    return to_status(rowops::launch_rmsnorm_bwd(dy, gamma, x, row_rms, dx, gamma_terms, rows, cols, vec4,
                                                st(stream)));
}

int rowops_column_sums(const float* in, float* out, int64_t rows, int64_t cols, float beta,
                       rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (!std::isfinite(beta)) return ROWOPS_ERR_SHAPE;
    if (cols == 0) return ROWOPS_OK;
    if (!out || (rows > 0 && !in)) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{in, 4}, {out, 4}})) return ROWOPS_ERR_ALIGN;
    if (overlap({in, rows * cols * 4}, {out, cols * 4})) return ROWOPS_ERR_ALIAS;
    return to_status(rowops::launch_column_sums(in, out, rows, cols, beta, st(stream)));
}

int rowops_masked_softmax_fmask(const float* x, const float* mask, float* y, int64_t rows, int64_t cols,
                                rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0 || cols == 0) return ROWOPS_OK;
    if (!x || !mask || !y) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {mask, 4}, {y, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (static_cast<const void*>(x) != y && overlap({x, n}, {y, n})) return ROWOPS_ERR_ALIAS;
    if (overlap({mask, n}, {y, n}) || overlap({mask, n}, {x, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(y, 16) && aligned(mask, 16);
    return to_status(rowops::launch_masked_softmax_fmask(x, mask, y, rows, cols, vec4, st(stream)));
}

int rowops_lrp_softmax_rows(const float* x, const float* y, const float* r, float* r_in, int64_t rows,
                            int64_t cols, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0 || cols == 0) return ROWOPS_OK;
    if (!x || !y || !r || !r_in) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {y, 4}, {r, 4}, {r_in, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (overlap({r_in, n}, {x, n}) || overlap({r_in, n}, {y, n}) || overlap({r_in, n}, {r, n}))
        return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(y, 16) && aligned(r, 16) &&
                      aligned(r_in, 16);
    return to_status(rowops::launch_lrp_softmax(x, y, r, r_in, rows, cols, vec4, st(stream)));
}

int rowops_argmax_onehot(const float* x, float* out, int64_t rows, int64_t cols, rowops_stream stream) {
    if (int e = check_dims(rows, cols)) return e;
    if (rows == 0 || cols == 0) return ROWOPS_OK;
    if (!x || !out) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {out, 4}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    if (overlap({x, n}, {out, n})) return ROWOPS_ERR_ALIAS;
    const bool vec4 = cols % 4 == 0 && aligned(x, 16) && aligned(out, 16);
    return to_status(rowops::launch_argmax_onehot(x, out, rows, cols, vec4, st(stream)));
}

static int ce2_checks(const float* x, const float* w, float* grad, float* row_loss, double* mean_loss,
                      int64_t rows, int64_t cols, float grad_scale, bool grad_required) {
    if (int e = check_dims(rows, cols)) return e;
    if (cols == 0 || !std::isfinite(grad_scale)) return ROWOPS_ERR_SHAPE;
    if (rows == 0) return -1;  // nothing to do
    if (!x || !w || !row_loss || !mean_loss || (grad_required && !grad)) return ROWOPS_ERR_NULL;
    if (!elems_aligned({{x, 4}, {w, 4}, {grad, 4}, {row_loss, 4}, {mean_loss, 8}})) return ROWOPS_ERR_ALIGN;
    const int64_t n = rows * cols * 4;
    const Buf in[2] = {{x, n}, {w, n}};
    const Buf out[3] = {{grad, grad ? n : 0}, {row_loss, rows * 4}, {mean_loss, 8}};
    for (const Buf& o : out) {
        for (const Buf& i : in)
            if (overlap(o, i)) return ROWOPS_ERR_ALIAS;
        for (const Buf& o2 : out)
            if (&o != &o2 && overlap(o, o2)) return ROWOPS_ERR_ALIAS;
    }
    return ROWOPS_OK;
}

int rowops_soft_ce(const float* logits, const float* weights, float* grad, float* row_loss, double* mean_loss,
                   int64_t rows, int64_t cols, float grad_scale, rowops_stream stream) {
    const int e = ce2_checks(logits, weights, grad, row_loss, mean_loss, rows, cols, grad_scale, true);
    if (e != ROWOPS_OK) return e < 0 ? ROWOPS_OK : e;
    const bool vec4 = cols % 4 == 0 && aligned(logits, 16) && aligned(weights, 16) && aligned(grad, 16);
    return to_status(rowops::launch_soft_ce(logits, weights, grad, row_loss, mean_loss, rows, cols, grad_scale,
                                            vec4, st(stream)));
}

int rowops_teacher_ce(const float* student, const float* teacher, float* grad, float* row_loss,
                      double* mean_loss, int64_t rows, int64_t cols, float grad_scale, rowops_stream stream) {
    const int e = ce2_checks(student, teacher, grad, row_loss, mean_loss, rows, cols, grad_scale, false);
    if (e != ROWOPS_OK) return e < 0 ? ROWOPS_OK : e;
    const bool vec4 = cols % 4 == 0 && aligned(student, 16) && aligned(teacher, 16) &&
                      (grad == nullptr || aligned(grad, 16));
    return to_status(rowops::launch_teacher_ce(student, teacher, grad, row_loss, mean_loss, rows, cols,
                                               grad_scale, vec4, st(stream)));
}

}  // extern "C"
