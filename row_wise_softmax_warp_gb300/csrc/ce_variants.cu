// ce_variants.cu - TorchLean's weighted-logits (soft-target) cross-entropy and
// fixed-teacher cross-entropy with the student gradient.
//
//   soft     loss_i = sum_j w_ij (lse_i - x_ij),  g_ij = scale (p_ij sum_k w_ik - w_ij)
//   teacher  q = softmax(t), loss_i = sum_j q_ij (lse(s)_i - s_ij),  g_ij = scale (p_ij - q_ij)
//
// Log-probabilities are formed as x - lse from the original logits, so a term
// whose probability underflows keeps a finite value.  Group kernels hold both
// rows in registers (geometry of common.cuh); longer rows stream two passes.
// The mean over rows is the fixed-order mean kernel of the integer-target loss.
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

template <bool TEACHER, int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
ce2_group(const float* __restrict__ x, const float* __restrict__ w, float* __restrict__ grad,
          float* __restrict__ row_loss, int64_t rows, int cols, float grad_scale) {
    constexpr int GPB = kBlockThreads / LANES;
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

template <bool TEACHER, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
ce2_rowblock(const float* __restrict__ x, const float* __restrict__ w, float* __restrict__ grad,
             float* __restrict__ row_loss, int64_t rows, int64_t cols, float grad_scale) {
    __shared__ float scratch[2 * kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        MaxSum sa{-INFINITY, 0.f}, sb{-INFINITY, 0.f};
        float wsum = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float a[VEC], b[VEC];
            ld_chunk<VEC>(x + off + c * VEC, a);
            ld_chunk<VEC>(w + off + c * VEC, b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                sa = ms_push(sa, a[e]);
                if constexpr (TEACHER)
                    sb = ms_push(sb, b[e]);
                else
                    wsum += b[e];
            }
        }
        sa = block_maxsum<kBlockThreads>(sa, scratch);
        if constexpr (TEACHER)
            sb = block_maxsum<kBlockThreads>(sb, scratch);
        else
            wsum = block_sum<kBlockThreads>(wsum, scratch);
        const float lse = sa.m + logf(sa.s);
        const float inv_sa = 1.0f / sa.s;
        const float inv_sb = TEACHER ? 1.0f / sb.s : 1.f;
        float loss = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float a[VEC], b[VEC], o[VEC];
            ld_chunk<VEC>(x + off + c * VEC, a);
            ld_chunk<VEC>(w + off + c * VEC, b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float q = TEACHER ? expf(b[e] - sb.m) * inv_sb : b[e];
                loss = fmaf(q, lse - a[e], loss);
                const float p = expf(a[e] - sa.m) * inv_sa;
                o[e] = TEACHER ? grad_scale * (p - q) : grad_scale * (p * wsum - q);
            }
            if (grad != nullptr) st_chunk<VEC>(grad + off + c * VEC, o);
        }
        loss = block_sum<kBlockThreads>(loss, scratch);
        if (threadIdx.x == 0) row_loss[row] = loss;
    }
}

template <bool TEACHER>
cudaError_t launch_ce2(const float* x, const float* w, float* grad, float* row_loss, double* mean_loss,
                       int64_t rows, int64_t cols, float grad_scale, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        ce2_group<TEACHER, G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            x, w, grad, row_loss, rows, int(cols), grad_scale);
    });
    if (!done) {
        if (vec4)
            ce2_rowblock<TEACHER, 4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, w, grad, row_loss, rows, cols,
                                                                                  grad_scale);
        else
            ce2_rowblock<TEACHER, 1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, w, grad, row_loss, rows, cols,
                                                                                  grad_scale);
    }
    note_launches(1);
    const cudaError_t err = cudaGetLastError();
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
