// misc_rows.cu - pulsatrix lrp_softmax_rows and TorchLean's first-max one-hot.
//
//   lrp_softmax_rows  r_in_j = x_j * (r_j - y_j * sum_k r_k)   (SoftmaxModule rule)
//   argmax_onehot     1 at the first maximal coordinate of the row, 0 elsewhere:
//                     maximal = exceeded by no entry (x_i > x_j for no i), so
//                     the first entry that is a NaN or equals the numeric max.
// Group kernels (geometry of common.cuh), block-row kernels for rows of
// 1025..16384 floats (block_rows.cuh) and streaming fallbacks.
#include <climits>

#include "block_rows.cuh"
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
lrp_group(const float* __restrict__ x, const float* __restrict__ y, const float* __restrict__ r,
          float* __restrict__ r_in, int64_t rows, int cols) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float rv[NV][VEC];
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk<VEC>(r + off + c * VEC, rv[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) rv[k][e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) s += rv[k][e];
        }
        s = group_sum<LANES>(s);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float xv[VEC], yv[VEC], o[VEC];
                ld_chunk<VEC>(x + off + c * VEC, xv);
                ld_chunk<VEC>(y + off + c * VEC, yv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = xv[e] * (rv[k][e] - yv[e] * s);
                st_chunk<VEC>(r_in + off + c * VEC, o);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
lrp_rowblock(const float* __restrict__ x, const float* __restrict__ y, const float* __restrict__ r,
             float* __restrict__ r_in, int64_t rows, int64_t cols) {
    __shared__ float scratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        float s = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float rv[VEC];
            ld_chunk<VEC>(r + off + c * VEC, rv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) s += rv[e];
        }
        s = block_sum<kBlockThreads>(s, scratch);
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float xv[VEC], yv[VEC], rv[VEC];
            ld_chunk<VEC>(x + off + c * VEC, xv);
            ld_chunk<VEC>(y + off + c * VEC, yv);
            ld_chunk<VEC>(r + off + c * VEC, rv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) rv[e] = xv[e] * (rv[e] - yv[e] * s);
            st_chunk<VEC>(r_in + off + c * VEC, rv);
        }
    }
}

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
argmax_group(const float* __restrict__ x, float* __restrict__ out, int64_t rows, int cols) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float v[NV][VEC];
        float m = -INFINITY;  // numeric maximum (fmaxf skips NaN)
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk<VEC>(x + off + c * VEC, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
            }
        }
        m = group_max<LANES>(m);
        int first = INT_MAX;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (isnan(v[k][e]) || v[k][e] == m) first = min(first, c * VEC + e);
        }
        first = group_min_int<LANES>(first);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = (c * VEC + e == first) ? 1.f : 0.f;
                st_chunk<VEC>(out + off + c * VEC, o);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
argmax_rowblock(const float* __restrict__ x, float* __restrict__ out, int64_t rows, int64_t cols) {
    __shared__ float fscratch[kBlockThreads / 32];
    __shared__ int iscratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        float m = -INFINITY;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(x + off + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[e]);
        }
        m = block_max<kBlockThreads>(m, fscratch);
        int first = INT_MAX;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(x + off + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (isnan(v[e]) || v[e] == m) first = min(first, int(c * VEC + e));
        }
        first = group_min_int<32>(first);
        if ((threadIdx.x & 31) == 0) iscratch[threadIdx.x >> 5] = first;
        __syncthreads();
        first = iscratch[0];
        for (int q = 1; q < kBlockThreads / 32; ++q) first = min(first, iscratch[q]);
        __syncthreads();
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float o[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = (c * VEC + e == first) ? 1.f : 0.f;
            st_chunk<VEC>(out + off + c * VEC, o);
        }
    }
}

// ------------------------------------------------------ block-row kernels

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
lrp_brow(const float* __restrict__ x, const float* __restrict__ y, const float* __restrict__ r,
         float* __restrict__ r_in, int64_t rows, int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float rv[NV][VEC];
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(r + off + c * VEC, rv[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s += rv[k][e];
            }
        }
        s = red.sum(s);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float xv[VEC], yv[VEC], o[VEC];
                ld_chunk<VEC>(x + off + c * VEC, xv);
                ld_chunk<VEC>(y + off + c * VEC, yv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = xv[e] * (rv[k][e] - yv[e] * s);
                st_chunk<VEC>(r_in + off + c * VEC, o);
            }
        }
    }
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
argmax_brow(const float* __restrict__ x, float* __restrict__ out, int64_t rows, int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float v[NV][VEC];
        float m = -INFINITY;  // numeric maximum (fmaxf skips NaN)
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(x + off + c * VEC, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
            }
        }
        m = red.max(m);
        int first = INT_MAX;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (isnan(v[k][e]) || v[k][e] == m) first = min(first, c * VEC + e);
        }
        first = red.min_int(first);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = (c * VEC + e == first) ? 1.f : 0.f;
                st_chunk<VEC>(out + off + c * VEC, o);
            }
        }
    }
}

}  // namespace

cudaError_t launch_lrp_softmax(const float* x, const float* y, const float* r, float* r_in, int64_t rows,
                               int64_t cols, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        lrp_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            x, y, r, r_in, rows, int(cols));
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                lrp_brow<G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                    x, y, r, r_in, rows, int(cols));
            })) {
        } else if (vec4)
            lrp_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, y, r, r_in, rows, cols);
        else
            lrp_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, y, r, r_in, rows, cols);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_argmax_onehot(const float* x, float* out, int64_t rows, int64_t cols, bool vec4,
                                 cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        argmax_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            x, out, rows, int(cols));
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                argmax_brow<G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                    x, out, rows, int(cols));
            })) {
        } else if (vec4)
            argmax_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, out, rows, cols);
        else
            argmax_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, out, rows, cols);
    }
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace rowops
