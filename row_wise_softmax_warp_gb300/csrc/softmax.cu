// softmax.cu - softmax forward/backward, scaled causal attention softmax
// forward/backward and hard-masked softmax.
//
// Kernel shapes per op:
//   *_group    : rows of up to 1024 floats held in registers by a group of
//                LANES lanes (geometry in common.cuh); one HBM read and one
//                HBM write per element.
//   *_brow     : rows of 1025..16384 floats held in registers by one CTA
//                (block_rows.cuh); one HBM read and one HBM write per element.
//   *_rowblock : any row length and alignment; one 256-thread block per row,
//                streaming the row from global memory once per pass.
#include "block_rows.cuh"
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

// ------------------------------------------------------------ softmax fwd
// pulsatrix HIPBackend::softmax_rows: y = exp(x - max) / sum exp(x - max).

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
softmax_fwd_group(const float* x, float* y, int64_t rows, int cols) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float v[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk_coherent<VEC>(x + off + c * VEC, v[k]);  // y may be x
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = -INFINITY;
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
        m = group_max<LANES>(m);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = exp_shifted(v[k][e], m);
                s += v[k][e];
            }
        s = group_sum<LANES>(s);
        const float inv = 1.0f / s;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = v[k][e] * inv;
                st_chunk<VEC>(y + off + c * VEC, o);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
softmax_fwd_rowblock(const float* x, float* y, int64_t rows, int64_t cols) {
    __shared__ float scratch[2 * kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * cols;
        float* yr = y + row * cols;
        MaxSum a{-INFINITY, 0.f};
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk_coherent<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) a = ms_push(a, v[e]);
        }
        a = block_maxsum<kBlockThreads>(a, scratch);
        const float inv = 1.0f / a.s;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk_coherent<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[e] = expf(v[e] - a.m) * inv;
            st_chunk<VEC>(yr + c * VEC, v);
        }
    }
}

// ------------------------------------------------------------ softmax bwd
// pulsatrix HIPBackend::softmax_rows_backward: dx = y * (dy - sum_k y_k dy_k).

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
softmax_bwd_group(const float* __restrict__ y, const float* __restrict__ dy,
                  float* __restrict__ dx, int64_t rows, int cols) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float a[NV][VEC], b[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk<VEC>(y + off + c * VEC, a[k]);
                ld_chunk<VEC>(dy + off + c * VEC, b[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = b[k][e] = 0.f;
            }
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) dot = fmaf(a[k][e], b[k][e], dot);
        dot = group_sum<LANES>(dot);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = a[k][e] * (b[k][e] - dot);
                st_chunk<VEC>(dx + off + c * VEC, o);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
softmax_bwd_rowblock(const float* __restrict__ y, const float* __restrict__ dy,
                     float* __restrict__ dx, int64_t rows, int64_t cols) {
    __shared__ float scratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        float dot = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float a[VEC], b[VEC];
            ld_chunk<VEC>(y + off + c * VEC, a);
            ld_chunk<VEC>(dy + off + c * VEC, b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) dot = fmaf(a[e], b[e], dot);
        }
        dot = block_sum<kBlockThreads>(dot, scratch);
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float a[VEC], b[VEC];
            ld_chunk<VEC>(y + off + c * VEC, a);
            ld_chunk<VEC>(dy + off + c * VEC, b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) a[e] = a[e] * (b[e] - dot);
            st_chunk<VEC>(dx + off + c * VEC, a);
        }
    }
}

// --------------------------------------------------- causal attention fwd
// MicroGPT CuBLASBackend::fused_attn_softmax with causal_mask_batched: row r is
// query q = r mod seq_len; keys j <= q keep scale*s_j, keys j > q get p = +0.
// Only the visible prefix of each row is read.

// Four 256-thread blocks per SM: the register cap (64) keeps the 1024-column
// row (32 floats per lane) spill-free and doubles the loads in flight.
template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads, 4)
attn_fwd_group(const float* __restrict__ s, float* __restrict__ p, int64_t rows, int cols,
               int64_t seq_len, float scale) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        const int q = live ? int(row % seq_len) : 0;
        const int nvis = q + 1 < cols ? q + 1 : cols;  // visible keys 0..q
        float v[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (g + k * LANES) * VEC;
            if (live && c0 < nvis) {
                ld_chunk<VEC>(s + off + c0, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = (c0 + e < nvis) ? v[k][e] : -INFINITY;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = -INFINITY;
            }
        }
        // max(scale * s) = scale * max(s) for scale > 0; exp(scale*s - max) is
        // evaluated as 2^((s - max(s)) * scale*log2(e)).
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
        m = group_max<LANES>(m);
        const float sl = scale * kLog2e;
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (g + k * LANES) * VEC;
            if (c0 < nvis) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    v[k][e] = (c0 + e < nvis) ? ex2_approx((v[k][e] - m) * sl) : 0.f;
                    sum += v[k][e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = 0.f;
            }
        }
        sum = group_sum<LANES>(sum);
        const float inv = 1.0f / sum;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = v[k][e] * inv;
                st_chunk<VEC>(p + off + c * VEC, o);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
attn_fwd_rowblock(const float* __restrict__ s, float* __restrict__ p, int64_t rows, int64_t cols,
                  int64_t seq_len, float scale) {
    __shared__ float scratch[2 * kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        const int64_t q = row % seq_len;
        const int64_t nvis = q + 1 < cols ? q + 1 : cols;
        MaxSum a{-INFINITY, 0.f};
        for (int64_t c = threadIdx.x; c * VEC < nvis; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(s + off + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (c * VEC + e < nvis) a = ms_push(a, scale * v[e]);
        }
        a = block_maxsum<kBlockThreads>(a, scratch);
        const float inv = 1.0f / a.s;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            if (c * VEC < nvis) {
                ld_chunk<VEC>(s + off + c * VEC, v);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    v[e] = (c * VEC + e < nvis) ? expf(scale * v[e] - a.m) * inv : 0.f;
                st_chunk<VEC>(p + off + c * VEC, v);
            } else {
                st_zero_chunk<VEC>(p + off + c * VEC);
            }
        }
    }
}

// --------------------------------------------------- causal attention bwd
// MicroGPT CuBLASBackend::fused_attn_softmax_backward: from the output p,
// ds = scale * p * (dp - sum_{k<=q} p_k dp_k) on the visible keys, +0 beyond.

// Three 256-thread blocks per SM (register cap 85) for the 2 x 32 floats per
// lane of a 1024-column row.
template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads, 3)
attn_bwd_group(const float* __restrict__ p, const float* __restrict__ dp, float* __restrict__ ds,
               int64_t rows, int cols, int64_t seq_len, float scale) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        const int q = live ? int(row % seq_len) : 0;
        const int nvis = q + 1 < cols ? q + 1 : cols;
        float a[NV][VEC], b[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (g + k * LANES) * VEC;
            if (live && c0 < nvis) {
                ld_chunk<VEC>(p + off + c0, a[k]);
                ld_chunk<VEC>(dp + off + c0, b[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (c0 + e >= nvis) a[k][e] = b[k][e] = 0.f;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = b[k][e] = 0.f;
            }
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) dot = fmaf(a[k][e], b[k][e], dot);
        dot = group_sum<LANES>(dot);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (g + k * LANES) * VEC;
            if (live && c0 < nch * VEC) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    o[e] = (c0 + e < nvis) ? scale * a[k][e] * (b[k][e] - dot) : 0.f;
                st_chunk<VEC>(ds + off + c0, o);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
attn_bwd_rowblock(const float* __restrict__ p, const float* __restrict__ dp,
                  float* __restrict__ ds, int64_t rows, int64_t cols, int64_t seq_len,
                  float scale) {
    __shared__ float scratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        const int64_t q = row % seq_len;
        const int64_t nvis = q + 1 < cols ? q + 1 : cols;
        float dot = 0.f;
        for (int64_t c = threadIdx.x; c * VEC < nvis; c += kBlockThreads) {
            float a[VEC], b[VEC];
            ld_chunk<VEC>(p + off + c * VEC, a);
            ld_chunk<VEC>(dp + off + c * VEC, b);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (c * VEC + e < nvis) dot = fmaf(a[e], b[e], dot);
        }
        dot = block_sum<kBlockThreads>(dot, scratch);
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            if (c * VEC < nvis) {
                float a[VEC], b[VEC];
                ld_chunk<VEC>(p + off + c * VEC, a);
                ld_chunk<VEC>(dp + off + c * VEC, b);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    a[e] = (c * VEC + e < nvis) ? scale * a[e] * (b[e] - dot) : 0.f;
                st_chunk<VEC>(ds + off + c * VEC, a);
            } else {
                st_zero_chunk<VEC>(ds + off + c * VEC);
            }
        }
    }
}

// ---------------------------------------- causal attention fwd, split rows
// Rows of 513..1024 floats (vectorised): two warps share a row, which halves the
// registers per thread and doubles the warps (and loads) in flight.  The row's
// float4 chunks go out in groups of 32 (128 columns): warp h of the pair takes
// groups h, h+2, h+4, ..., so every load is 512 contiguous bytes and the two
// warps split a causal row's visible prefix evenly.  A block (8 warps) covers 4
// rows per iteration; the halves combine their (max, sum) through shared
// memory, half 0 then half 1, so both warps see identical values.

template <int NVH>
__global__ void __launch_bounds__(kBlockThreads, 6)
attn_fwd_split2(const float* __restrict__ s, float* __restrict__ p, int64_t rows, int cols,
                int64_t seq_len, float scale) {
    __shared__ float part[2][kBlockThreads / 32][2];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int pair = w >> 1, half = w & 1;
    const int nch = cols / 4;
    const float sl = scale * kLog2e;
    int it = 0;
    for (int64_t base = int64_t(blockIdx.x) * 4; base < rows; base += int64_t(gridDim.x) * 4, ++it) {
        const int64_t row = base + pair;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        const int q = live ? int(row % seq_len) : -1;
        const int nvis = q + 1 < cols ? q + 1 : cols;  // 0 for a dead row
        float v[NVH][4];
#pragma unroll
        for (int k = 0; k < NVH; ++k) {
            const int c = (2 * k + half) * 32 + lane;
            const int c0 = c * 4;
            if (c < nch && c0 < nvis) {
                ld_chunk<4>(s + off + c0, v[k]);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[k][e] = (c0 + e < nvis) ? v[k][e] : -INFINITY;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[k][e] = -INFINITY;
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NVH; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) m = fmaxf(m, v[k][e]);
        m = group_max<32>(m);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NVH; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[k][e] = (m == -INFINITY || v[k][e] == -INFINITY) ? 0.f : ex2_approx((v[k][e] - m) * sl);
                sum += v[k][e];
            }
        sum = group_sum<32>(sum);
        const int par = it & 1;
        if (lane == 0) {
            part[par][w][0] = m;
            part[par][w][1] = sum;
        }
        __syncthreads();
        const float m0 = part[par][2 * pair][0], s0 = part[par][2 * pair][1];
        const float m1 = part[par][2 * pair + 1][0], s1 = part[par][2 * pair + 1][1];
        const float M = fmaxf(m0, m1);
        const float f0 = m0 == -INFINITY ? 0.f : ex2_approx((m0 - M) * sl);
        const float f1 = m1 == -INFINITY ? 0.f : ex2_approx((m1 - M) * sl);
        const float S = s0 * f0 + s1 * f1;
        const float alpha = (half == 0 ? f0 : f1) / S;
#pragma unroll
        for (int k = 0; k < NVH; ++k) {
            const int c = (2 * k + half) * 32 + lane;
            if (live && c < nch) {
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = v[k][e] * alpha;
                st_chunk<4>(p + off + c * 4, o);
            }
        }
    }
}

// ------------------------------------------------------ hard-masked softmax
// TorchLean hard-masked softmax: max and denominator over allowed entries
// (mask value != 0: a byte mask, or a float mask where -0.0 blocks and NaN
// allows); blocked entries +0; a row with nothing allowed is all +0.

template <typename MaskT, int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
masked_group(const float* x, const MaskT* __restrict__ mask, float* y, int64_t rows, int cols) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float v[NV][VEC];
        bool al[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk_coherent<VEC>(x + off + c * VEC, v[k]);  // y may be x
                ld_mask<VEC>(mask + off + c * VEC, al[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) al[k][e] = false;
            }
        }
        float m = -INFINITY;
        int n_allowed = 0;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (al[k][e]) {
                    m = fmaxf(m, v[k][e]);
                    ++n_allowed;
                }
        m = group_max<LANES>(m);
        n_allowed = group_sum_int<LANES>(n_allowed);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = al[k][e] ? exp_shifted(v[k][e], m) : 0.f;
                s += v[k][e];
            }
        s = group_sum<LANES>(s);
        const float inv = n_allowed > 0 ? 1.0f / s : 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = al[k][e] ? v[k][e] * inv : 0.f;
                st_chunk<VEC>(y + off + c * VEC, o);
            }
        }
    }
}

template <typename MaskT, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
masked_rowblock(const float* x, const MaskT* __restrict__ mask, float* y, int64_t rows,
                int64_t cols) {
    __shared__ float scratch[2 * kBlockThreads / 32];
    __shared__ int iscratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        MaxSum a{-INFINITY, 0.f};
        int n_allowed = 0;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            bool al[VEC];
            ld_chunk_coherent<VEC>(x + off + c * VEC, v);
            ld_mask<VEC>(mask + off + c * VEC, al);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (al[e]) {
                    a = ms_push(a, v[e]);
                    ++n_allowed;
                }
        }
        a = block_maxsum<kBlockThreads>(a, scratch);
        n_allowed = block_sum_int<kBlockThreads>(n_allowed, iscratch);
        const float inv = n_allowed > 0 ? 1.0f / a.s : 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            bool al[VEC];
            ld_chunk_coherent<VEC>(x + off + c * VEC, v);
            ld_mask<VEC>(mask + off + c * VEC, al);
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[e] = al[e] ? expf(v[e] - a.m) * inv : 0.f;
            st_chunk<VEC>(y + off + c * VEC, v);
        }
    }
}

// ------------------------------------------------------ block-row kernels
// Rows of 1025..16384 floats, one CTA per row in registers (block_rows.cuh);
// the same arithmetic as the group kernels above, with block reductions.

// Loads the thread's NV chunks of a row (fill for chunks past the row).
template <int NT, int NV, int VEC, bool COHERENT>
__device__ __forceinline__ void brow_load(const float* r, int nch, float (&v)[NV][VEC], float fill) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = int(threadIdx.x) + k * NT;
        if (c < nch) {
            if constexpr (COHERENT)
                ld_chunk_coherent<VEC>(r + c * VEC, v[k]);
            else
                ld_chunk<VEC>(r + c * VEC, v[k]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] = fill;
        }
    }
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
softmax_fwd_brow(const float* x, float* y, int64_t rows, int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float v[NV][VEC];
        brow_load<NT, NV, VEC, true>(x + off, nch, v, -INFINITY);  // y may be x
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
        m = red.max(m);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = exp_shifted(v[k][e], m);
                s += v[k][e];
            }
        s = red.sum(s);
        const float inv = 1.0f / s;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = v[k][e] * inv;
                st_chunk<VEC>(y + off + c * VEC, o);
            }
        }
    }
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
softmax_bwd_brow(const float* __restrict__ y, const float* __restrict__ dy, float* __restrict__ dx,
                 int64_t rows, int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float a[NV][VEC], b[NV][VEC];
        brow_load<NT, NV, VEC, false>(y + off, nch, a, 0.f);
        brow_load<NT, NV, VEC, false>(dy + off, nch, b, 0.f);
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) dot = fmaf(a[k][e], b[k][e], dot);
        dot = red.sum(dot);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = a[k][e] * (b[k][e] - dot);
                st_chunk<VEC>(dx + off + c * VEC, o);
            }
        }
    }
}

// Causal attention forward: only the visible prefix (keys 0..q) is read.
template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
attn_fwd_brow(const float* __restrict__ s, float* __restrict__ p, int64_t rows, int cols, int64_t seq_len,
              float scale) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    const float sl = scale * kLog2e;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        const int q = int(row % seq_len);
        const int nvis = q + 1 < cols ? q + 1 : cols;
        float v[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (int(threadIdx.x) + k * NT) * VEC;
            if (c0 < nvis) {
                ld_chunk<VEC>(s + off + c0, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = (c0 + e < nvis) ? v[k][e] : -INFINITY;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = -INFINITY;
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
        m = red.max(m);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (int(threadIdx.x) + k * NT) * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = (c0 + e < nvis) ? ex2_approx((v[k][e] - m) * sl) : 0.f;
                sum += v[k][e];
            }
        }
        sum = red.sum(sum);
        const float inv = 1.0f / sum;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = v[k][e] * inv;
                st_chunk<VEC>(p + off + c * VEC, o);
            }
        }
    }
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
attn_bwd_brow(const float* __restrict__ p, const float* __restrict__ dp, float* __restrict__ ds, int64_t rows,
              int cols, int64_t seq_len, float scale) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        const int q = int(row % seq_len);
        const int nvis = q + 1 < cols ? q + 1 : cols;
        float a[NV][VEC], b[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c0 = (int(threadIdx.x) + k * NT) * VEC;
            if (c0 < nvis) {
                ld_chunk<VEC>(p + off + c0, a[k]);
                ld_chunk<VEC>(dp + off + c0, b[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (c0 + e >= nvis) a[k][e] = b[k][e] = 0.f;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = b[k][e] = 0.f;
            }
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) dot = fmaf(a[k][e], b[k][e], dot);
        dot = red.sum(dot);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                const int c0 = c * VEC;
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = (c0 + e < nvis) ? scale * a[k][e] * (b[k][e] - dot) : 0.f;
                st_chunk<VEC>(ds + off + c0, o);
            }
        }
    }
}

template <typename MaskT, int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
masked_brow(const float* x, const MaskT* __restrict__ mask, float* y, int64_t rows, int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float v[NV][VEC];
        bool al[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk_coherent<VEC>(x + off + c * VEC, v[k]);  // y may be x
                ld_mask<VEC>(mask + off + c * VEC, al[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) al[k][e] = false;
            }
        }
        float m = -INFINITY;
        int n_allowed = 0;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (al[k][e]) {
                    m = fmaxf(m, v[k][e]);
                    ++n_allowed;
                }
        red.max_count(m, n_allowed);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = al[k][e] ? exp_shifted(v[k][e], m) : 0.f;
                s += v[k][e];
            }
        s = red.sum(s);
        const float inv = n_allowed > 0 ? 1.0f / s : 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = al[k][e] ? v[k][e] * inv : 0.f;
                st_chunk<VEC>(y + off + c * VEC, o);
            }
        }
    }
}

}  // namespace

// ------------------------------------------------------------ launchers

cudaError_t launch_softmax_fwd(const float* x, float* y, int64_t rows, int64_t cols, bool vec4,
                               cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        softmax_fwd_group<G::LANES, G::NV, G::VEC>
            <<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(x, y, rows, int(cols));
    });
    cudaError_t err = cudaSuccess;
    if (!done) {
        // Up to 8192 floats: on GB300 the TMA kernel is ahead at 16384 (51.8
        // against 64.2 us on 2048 rows), the block-row kernel below (45.7
        // against 66.2 us on 4096 x 8192, 45.8 against 195 us on 16384 x 2048).
        if (with_block_geometry(vec4, cols, 8192, [&](auto geo) {
                using G = decltype(geo);
                softmax_fwd_brow<G::NT, G::NV, G::VEC>
                    <<<block_row_grid(rows), G::NT, 0, stream>>>(x, y, rows, int(cols));
            })) {
        } else if (launch_softmax_tma(x, y, rows, cols, stream, &err)) {
        } else if (vec4) {
            softmax_fwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, y, rows, cols);
        } else {
            softmax_fwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, y, rows, cols);
        }
    }
    note_launches(1);
    const cudaError_t last = cudaGetLastError();
    return err != cudaSuccess ? err : last;
}

cudaError_t launch_softmax_bwd(const float* y, const float* dy, float* dx, int64_t rows,
                               int64_t cols, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        softmax_bwd_group<G::LANES, G::NV, G::VEC>
            <<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(y, dy, dx, rows, int(cols));
    });
    cudaError_t err = cudaSuccess;
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                softmax_bwd_brow<G::NT, G::NV, G::VEC>
                    <<<block_row_grid(rows), G::NT, 0, stream>>>(y, dy, dx, rows, int(cols));
            })) {
        } else if (launch_softmax_bwd_tma(y, dy, dx, rows, cols, stream, &err)) {
            // longer rows: (y, dy) chunk pairs through the bulk-copy ring, two passes
        } else if (vec4)
            softmax_bwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(y, dy, dx, rows, cols);
        else
            softmax_bwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(y, dy, dx, rows, cols);
    }
    note_launches(1);
    const cudaError_t last = cudaGetLastError();
    return err != cudaSuccess ? err : last;
}

// Split rows for vectorised rows of 513..1024 floats (two warps per row): the
// forward only.  On GB300 (98,304 x 1024 causal rows) the split took the forward
// from 100.7 to 96.0 us, but the backward from 125 to 153 us (it holds p and dp
// and synchronises the block every four rows), so the backward keeps one warp
// per row.
inline bool attn_split_applies(bool vec4, int64_t cols) { return vec4 && cols > 512 && cols <= 1024; }

inline unsigned split_grid(int64_t rows) {
    int64_t b = (rows + 3) / 4;
    if (b > (1 << 20)) b = 1 << 20;
    return unsigned(b < 1 ? 1 : b);
}

cudaError_t launch_attn_fwd(const float* s, float* p, int64_t rows, int64_t cols, int64_t seq_len,
                            float scale, bool vec4, cudaStream_t stream) {
    if (attn_split_applies(vec4, cols)) {
        attn_fwd_split2<4><<<split_grid(rows), kBlockThreads, 0, stream>>>(s, p, rows, int(cols), seq_len, scale);
        note_launches(1);
        return cudaGetLastError();
    }
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        attn_fwd_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0,
                                                  stream>>>(s, p, rows, int(cols), seq_len, scale);
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                attn_fwd_brow<G::NT, G::NV, G::VEC>
                    <<<block_row_grid(rows), G::NT, 0, stream>>>(s, p, rows, int(cols), seq_len, scale);
            })) {
        } else if (vec4)
            attn_fwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(s, p, rows, cols,
                                                                               seq_len, scale);
        else
            attn_fwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(s, p, rows, cols,
                                                                               seq_len, scale);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const float* p, const float* dp, float* ds, int64_t rows,
                            int64_t cols, int64_t seq_len, float scale, bool vec4,
                            cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        attn_bwd_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0,
                                                  stream>>>(p, dp, ds, rows, int(cols), seq_len,
                                                            scale);
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                attn_bwd_brow<G::NT, G::NV, G::VEC>
                    <<<block_row_grid(rows), G::NT, 0, stream>>>(p, dp, ds, rows, int(cols), seq_len, scale);
            })) {
        } else if (vec4)
            attn_bwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(p, dp, ds, rows, cols,
                                                                               seq_len, scale);
        else
            attn_bwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(p, dp, ds, rows, cols,
                                                                               seq_len, scale);
    }
    note_launches(1);
    return cudaGetLastError();
}

template <typename MaskT>
cudaError_t launch_masked_impl(const float* x, const MaskT* mask, float* y, int64_t rows, int64_t cols,
                               bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        masked_group<MaskT, G::LANES, G::NV, G::VEC>
            <<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(x, mask, y, rows, int(cols));
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                masked_brow<MaskT, G::NT, G::NV, G::VEC>
                    <<<block_row_grid(rows), G::NT, 0, stream>>>(x, mask, y, rows, int(cols));
            })) {
        } else if (vec4)
            masked_rowblock<MaskT, 4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, mask, y, rows, cols);
        else
            masked_rowblock<MaskT, 1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, mask, y, rows, cols);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_masked_softmax(const float* x, const uint8_t* mask, float* y, int64_t rows,
                                  int64_t cols, bool vec4, cudaStream_t stream) {
    return launch_masked_impl(x, mask, y, rows, cols, vec4, stream);
}

cudaError_t launch_masked_softmax_fmask(const float* x, const float* mask, float* y, int64_t rows,
                                        int64_t cols, bool vec4, cudaStream_t stream) {
    return launch_masked_impl(x, mask, y, rows, cols, vec4, stream);
}

}  // namespace rowops
