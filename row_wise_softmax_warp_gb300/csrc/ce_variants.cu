// ce_variants.cu - TorchLean's weighted-logits (soft-target) cross-entropy and
// fixed-teacher cross-entropy with the student gradient.
//
//   soft     loss_i = sum_j w_ij (lse_i - x_ij),  g_ij = scale (p_ij sum_k w_ik - w_ij)
//   teacher  q = softmax(t), loss_i = sum_j q_ij (lse(s)_i - s_ij),  g_ij = scale (p_ij - q_ij)
//
// Log-probabilities are formed as x - lse from the original logits, so a term
// whose probability underflows keeps a finite value.  Group kernels hold both
// rows in registers (geometry of common.cuh), block-row kernels rows of
// 1025..16384 floats (block_rows.cuh); longer rows stream two passes through
// the L2, by bulk copies (tma_rows.cu) or, when x and w differ in alignment,
// by plain loads (ce2_stream).
// The mean over rows is the fixed-order mean kernel of the integer-target loss.
#include "block_rows.cuh"
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

template <bool TEACHER, int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
ce2_group(const float* __restrict__ x, const float* __restrict__ w, float* __restrict__ grad,
          float* __restrict__ row_loss, int64_t rows, int cols, float grad_scale) {
    const int GPB = int(blockDim.x) / LANES;  // blocks of up to kBlockThreads
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float a[NV][VEC], b[NV][VEC];
        bool valid[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            valid[k] = live && c < nch;
            if (valid[k]) {
                ld_chunk<VEC>(x + off + c * VEC, a[k]);
                ld_chunk<VEC>(w + off + c * VEC, b[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    a[k][e] = -INFINITY;
                    b[k][e] = TEACHER ? -INFINITY : 0.f;
                }
            }
        }
        float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                ma = fmaxf(ma, a[k][e]);
                if constexpr (TEACHER) mb = fmaxf(mb, b[k][e]);
            }
        ma = group_max<LANES>(ma);
        if constexpr (TEACHER) mb = group_max<LANES>(mb);
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                sa += exp_shifted(a[k][e], ma);
                if constexpr (TEACHER) {
                    b[k][e] = exp_shifted(b[k][e], mb);  // unnormalised teacher weights
                }
                sb += b[k][e];                            // soft: the weight sum
            }
        sa = group_sum<LANES>(sa);
        sb = group_sum<LANES>(sb);
        const float lse = ma + logf(sa);
        const float inv_sa = 1.0f / sa;
        const float qs = TEACHER ? 1.0f / sb : 1.f;  // teacher: q = b / sb
        float loss = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (valid[k])
#pragma unroll
                for (int e = 0; e < VEC; ++e) loss = fmaf(b[k][e] * qs, lse - a[k][e], loss);
        loss = group_sum<LANES>(loss);
        if (grad != nullptr) {
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int c = g + k * LANES;
                if (valid[k]) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float p = exp_shifted(a[k][e], ma) * inv_sa;
                        o[e] = TEACHER ? grad_scale * (p - b[k][e] * qs) : grad_scale * (p * sb - b[k][e]);
                    }
                    st_chunk<VEC>(grad + off + c * VEC, o);
                }
            }
        }
        if (live && g == 0) row_loss[row] = loss;
    }
}

// Rows of 1025..16384 floats: one CTA per row pair in registers
// (block_rows.cuh), the arithmetic of ce2_group with block reductions.
template <bool TEACHER, int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
ce2_brow(const float* __restrict__ x, const float* __restrict__ w, float* __restrict__ grad,
         float* __restrict__ row_loss, int64_t rows, int cols, float grad_scale) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float a[NV][VEC], b[NV][VEC];
        float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(x + off + c * VEC, a[k]);
                ld_chunk<VEC>(w + off + c * VEC, b[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    a[k][e] = -INFINITY;
                    b[k][e] = TEACHER ? -INFINITY : 0.f;
                }
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                ma = fmaxf(ma, a[k][e]);
                if constexpr (TEACHER) mb = fmaxf(mb, b[k][e]);
            }
        }
        if constexpr (TEACHER)
            red.max2(ma, mb);
        else
            ma = red.max(ma);
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                sa += exp_shifted(a[k][e], ma);
                if constexpr (TEACHER) b[k][e] = exp_shifted(b[k][e], mb);  // unnormalised teacher weights
                sb += b[k][e];                                               // soft: the weight sum
            }
        red.sum2(sa, sb);
        const float lse = ma + logf(sa);
        const float inv_sa = 1.0f / sa;
        const float qs = TEACHER ? 1.0f / sb : 1.f;  // teacher: q = b / sb
        float loss = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    loss = fmaf(b[k][e] * qs, lse - a[k][e], loss);
                    const float p = exp_shifted(a[k][e], ma) * inv_sa;
                    o[e] = TEACHER ? grad_scale * (p - b[k][e] * qs) : grad_scale * (p * sb - b[k][e]);
                }
                if (grad != nullptr) st_chunk<VEC>(grad + off + c * VEC, o);
            }
        }
        loss = red.sum(loss);
        if (threadIdx.x == 0) row_loss[row] = loss;
    }
}

// Rows of more than 16384 floats go to the bulk-copy pipeline (tma_rows.cu)
// when x and w share their alignment modulo 16 bytes; otherwise to this
// kernel: one 1024-thread CTA per SM walks rows and
// reads each row pair twice, (max, sum) in the first pass and loss and
// gradient in the second.  With one row pair in flight per SM (61 MB for
// 50304-float rows on 152 SMs) the second pass finds the rows in the L2, so
// HBM sees one read of each input and one write of the gradient.  Each thread
// keeps UNROLL chunks of both rows in flight per step.
constexpr int kStreamThreads = 1024;

template <bool TEACHER, int VEC>
__global__ void __launch_bounds__(kStreamThreads, 1)
ce2_stream(const float* __restrict__ x, const float* __restrict__ w, float* __restrict__ grad,
           float* __restrict__ row_loss, int64_t rows, int64_t cols, float grad_scale) {
    constexpr int UNROLL = VEC == 4 ? 2 : 8;  // 64 bytes of the row pair in flight per thread
    constexpr int NW = kStreamThreads / 32;
    __shared__ float part[2][4][NW];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t nch = cols / VEC;
    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const int64_t off = row * cols;
        float ma = -INFINITY, sa = 0.f, mb = -INFINITY, sb = 0.f;
        for (int64_t base = threadIdx.x; base < nch; base += int64_t(UNROLL) * kStreamThreads) {
            float a[UNROLL][VEC], b[UNROLL][VEC];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t c = base + int64_t(u) * kStreamThreads;
                if (c < nch) {
                    ld_chunk<VEC>(x + off + c * VEC, a[u]);
                    ld_chunk<VEC>(w + off + c * VEC, b[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        a[u][e] = -INFINITY;
                        b[u][e] = TEACHER ? -INFINITY : 0.f;
                    }
                }
            }
            float na = ma, nb = mb;
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    na = fmaxf(na, a[u][e]);
                    if constexpr (TEACHER) nb = fmaxf(nb, b[u][e]);
                }
            if (na > ma) {  // rescale the running sum to the new maximum
                sa *= exp_shifted(ma, na);
                ma = na;
            }
            if constexpr (TEACHER) {
                if (nb > mb) {
                    sb *= exp_shifted(mb, nb);
                    mb = nb;
                }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    if (ma != -INFINITY) sa += exp_shifted(a[u][e], ma);
                    if constexpr (TEACHER) {
                        if (mb != -INFINITY) sb += exp_shifted(b[u][e], mb);
                    } else {
                        sb += b[u][e];  // the weight sum
                    }
                }
        }
        // (max, sum) pairs of the block: warp butterfly, then warps in order.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const MaxSum ta =
                ms_merge({ma, sa}, {__shfl_xor_sync(kFullMask, ma, o), __shfl_xor_sync(kFullMask, sa, o)});
            ma = ta.m;
            sa = ta.s;
            if constexpr (TEACHER) {
                const MaxSum tb =
                    ms_merge({mb, sb}, {__shfl_xor_sync(kFullMask, mb, o), __shfl_xor_sync(kFullMask, sb, o)});
                mb = tb.m;
                sb = tb.s;
            } else {
                sb += __shfl_xor_sync(kFullMask, sb, o);
            }
        }
        const int par = it & 1;  // alternating buffers: one barrier per reduction
        if (lane == 0) {
            part[par][0][wid] = ma;
            part[par][1][wid] = sa;
            part[par][2][wid] = mb;  // soft: unused
            part[par][3][wid] = sb;  // soft: the weight sum
        }
        __syncthreads();
        MaxSum A{part[par][0][0], part[par][1][0]};
        MaxSum B{part[par][2][0], part[par][3][0]};
        float wsum = part[par][3][0];
        for (int q = 1; q < NW; ++q) {
            A = ms_merge(A, MaxSum{part[par][0][q], part[par][1][q]});
            if constexpr (TEACHER)
                B = ms_merge(B, MaxSum{part[par][2][q], part[par][3][q]});
            else
                wsum += part[par][3][q];
        }
        const float lse = A.m + logf(A.s);
        const float inv_sa = 1.0f / A.s;
        const float inv_sb = TEACHER ? 1.0f / B.s : 1.f;
        float loss = 0.f;
        for (int64_t base = threadIdx.x; base < nch; base += int64_t(UNROLL) * kStreamThreads) {
            float a[UNROLL][VEC], b[UNROLL][VEC];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t c = base + int64_t(u) * kStreamThreads;
                if (c < nch) {
                    ld_chunk<VEC>(x + off + c * VEC, a[u]);
                    ld_chunk<VEC>(w + off + c * VEC, b[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t c = base + int64_t(u) * kStreamThreads;
                if (c < nch) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float q = TEACHER ? exp_shifted(b[u][e], B.m) * inv_sb : b[u][e];
                        loss = fmaf(q, lse - a[u][e], loss);
                        const float p = exp_shifted(a[u][e], A.m) * inv_sa;
                        o[e] = TEACHER ? grad_scale * (p - q) : grad_scale * (p * wsum - q);
                    }
                    if (grad != nullptr) st_chunk<VEC>(grad + off + c * VEC, o);
                }
            }
        }
        loss = group_sum<32>(loss);
        __syncthreads();  // all threads have read this row's part[par]
        if (lane == 0) part[par][0][wid] = loss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float l = part[par][0][0];
            for (int q = 1; q < NW; ++q) l += part[par][0][q];
            row_loss[row] = l;
        }
    }
}

template <bool TEACHER>
cudaError_t launch_ce2(const float* x, const float* w, float* grad, float* row_loss, double* mean_loss,
                       int64_t rows, int64_t cols, float grad_scale, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        // blocks of 128 threads: finer than 256 when a row takes a warp of
        // ~90 registers and the rows do not fit one wave (on GB300, 4096 x 768
        // back to back: soft 11.2 -> 10.9 us, teacher 12.6 -> 12.4)
        constexpr int nt = 128;
        const int64_t gpb = nt / G::LANES;
        const int64_t blocks = (rows + gpb - 1) / gpb;
        ce2_group<TEACHER, G::LANES, G::NV, G::VEC>
            <<<unsigned(blocks < (1 << 20) ? blocks : (1 << 20)), nt, 0, stream>>>(x, w, grad, row_loss, rows,
                                                                               int(cols), grad_scale);
    });
    cudaError_t err = cudaSuccess;
    if (!done && !with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
            using G = decltype(geo);
            ce2_brow<TEACHER, G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                x, w, grad, row_loss, rows, int(cols), grad_scale);
        }) &&
        !(TEACHER ? launch_teacher_ce_tma(x, w, grad, row_loss, rows, cols, grad_scale, stream, &err)
                  : launch_soft_ce_tma(x, w, grad, row_loss, rows, cols, grad_scale, stream, &err))) {
        const int sms = sm_count();
        const unsigned grid = unsigned(rows < sms ? rows : (sms > 0 ? sms : 1));
        if (vec4)
            ce2_stream<TEACHER, 4><<<grid, kStreamThreads, 0, stream>>>(x, w, grad, row_loss, rows, cols, grad_scale);
        else
            ce2_stream<TEACHER, 1><<<grid, kStreamThreads, 0, stream>>>(x, w, grad, row_loss, rows, cols, grad_scale);
    }
    note_launches(1);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_row_mean(row_loss, rows, mean_loss, stream);
}

}  // namespace

cudaError_t launch_soft_ce(const float* x, const float* w, float* grad, float* row_loss, double* mean_loss,
                           int64_t rows, int64_t cols, float grad_scale, bool vec4, cudaStream_t stream) {
    return launch_ce2<false>(x, w, grad, row_loss, mean_loss, rows, cols, grad_scale, vec4, stream);
}

cudaError_t launch_teacher_ce(const float* s, const float* t, float* grad, float* row_loss, double* mean_loss,
                              int64_t rows, int64_t cols, float grad_scale, bool vec4, cudaStream_t stream) {
    return launch_ce2<true>(s, t, grad, row_loss, mean_loss, rows, cols, grad_scale, vec4, stream);
}

}  // namespace rowops
