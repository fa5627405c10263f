// topk_kept.cu - top-k kept mask (TorchLean Spec.MoE.kept): entry i of a row is
// kept when fewer than k entries beat it; j beats i when x_j > x_i, or when
// neither is larger and j < i.
//
// The selection itself (exact for every input, NaN included) is in
// kept_core.cuh; this file holds the kernels that load rows and store the mask.
#include "common.cuh"
#include "kept_core.cuh"
#include "launch.h"

namespace rowops {
namespace {

using kept_detail::low_bits;
using kept_detail::make_key;

// Group kernel (geometry of common.cuh): a group of LANES lanes owns a row.
// Blocks walk the rows in a grid-stride loop and load a group's next row
// before selecting in the current one, so that load is in flight meanwhile.
template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
kept_group(const float* __restrict__ x, float* __restrict__ kept, int64_t rows, int cols, int k) {
    constexpr int GPB = kBlockThreads / LANES;
    __shared__ KeptScratch kscratch[kBlockThreads / 32];  // the candidate path's, one per warp
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    const int64_t stride = int64_t(gridDim.x) * GPB;
    float next[NV][VEC];
    kept_load_row<LANES, NV, VEC>(x, int64_t(blockIdx.x) * GPB + grp, rows, cols, next);
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += stride) {  // block-uniform
        float v[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[kk][e] = next[kk][e];
        if (base + stride < rows) kept_load_row<LANES, NV, VEC>(x, base + stride + grp, rows, cols, next);
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        bool valid[NV][VEC];
        float probe = 0.f;  // a NaN anywhere makes the sum non-finite
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                valid[kk][e] = live && g + kk * LANES < nch;
                probe += v[kk][e];
            }
        // A non-finite sum (NaN, or infinities / overflow) sends the warp to the
        // literal count, which is exact for every input.
        const bool any_nan = __any_sync(kFullMask, !(fabsf(probe) <= 3.402823466e38f));
        if (k <= 2 && !any_nan && cols == LANES * NV * VEC) {  // warp-uniform
            kept_store_top2_full<LANES, NV, VEC>(v, k, live, kept + off);
            continue;
        }
        bool keep[NV][VEC];
        kept_select<LANES, NV, VEC>(v, valid, any_nan, cols, k, keep, &kscratch[threadIdx.x >> 5]);
#pragma unroll
        for (int kk = 0; kk < NV; ++kk) {
            const int c = g + kk * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = keep[kk][e] ? 1.f : 0.f;
                st_chunk<VEC>(kept + off + c * VEC, o);
            }
        }
    }
}

// Any length and alignment: one block per row, re-reading the row from global
// memory (L1/L2) on every counting pass.
template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
kept_rowblock(const float* __restrict__ x, float* __restrict__ kept, int64_t rows, int cols, int k) {
    __shared__ int scratch[kBlockThreads / 32];
    const int nch = cols / VEC;
    const int lb = low_bits(cols);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * int64_t(cols);
        float* kr = kept + row * int64_t(cols);
        int nans = 0;
        for (int c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) nans += isnan(v[e]) ? 1 : 0;
        }
        nans = block_sum_int<kBlockThreads>(nans, scratch);
        if (nans > 0) {
            for (int c = threadIdx.x; c < nch; c += kBlockThreads) {
                float v[VEC], o[VEC];
                ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int i = c * VEC + e;
                    int n = 0;
                    for (int j = 0; j < cols; ++j) {
                        const float xj = __ldg(xr + j);
                        const bool larger = xj > v[e];
                        const bool neither = !(xj > v[e]) && !(v[e] > xj);
                        n += (larger || (neither && j < i)) ? 1 : 0;
                    }
                    o[e] = n < k ? 1.f : 0.f;
                }
                st_chunk<VEC>(kr + c * VEC, o);
            }
            continue;
        }
        uint64_t t = 0;
        for (int b = 63; b >= 0; --b) {
            if (b < 32 && b >= lb) continue;
            const uint64_t cand = t | (uint64_t(1) << b);
            int n = 0;
            for (int c = threadIdx.x; c < nch; c += kBlockThreads) {
                float v[VEC];
                ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
                for (int e = 0; e < VEC; ++e) n += make_key(v[e], c * VEC + e, cols) >= cand ? 1 : 0;
            }
            if (block_sum_int<kBlockThreads>(n, scratch) >= k) t = cand;
        }
        for (int c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC], o[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = make_key(v[e], c * VEC + e, cols) >= t ? 1.f : 0.f;
            st_chunk<VEC>(kr + c * VEC, o);
        }
    }
}

}  // namespace

cudaError_t launch_topk_kept(const float* x, float* kept, int64_t rows, int64_t cols, int64_t k,
                             bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        kept_group<G::LANES, G::NV, G::VEC><<<stream_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            x, kept, rows, int(cols), int(k));
    });
    if (!done) {
        if (vec4)
            kept_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, kept, rows, int(cols), int(k));
        else
            kept_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, kept, rows, int(cols), int(k));
    }
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace rowops
