// block_rows.cuh - mid-length rows (1025..16384 floats): one CTA per row, the
// row held in registers.
//
// A CTA of NT threads owns one row at a time (rows blockIdx.x, blockIdx.x +
// gridDim.x, ...).  Thread t holds the row's chunks t, t + NT, ...,
// t + (NV-1)*NT of VEC floats, so each load or store instruction of a warp
// covers consecutive addresses, and HBM sees one read and one write per
// element.  Row statistics are reduced across the block: a warp butterfly,
// then the warps' partials through shared memory, added in warp order by every
// thread, so all threads hold the bit-identical result.  The partials
// alternate between two shared-memory buffers, so a reduction costs one
// __syncthreads: a thread can only overwrite a buffer after the next
// reduction's barrier, which every thread reaches after reading it.
#pragma once

#include "common.cuh"

namespace rowops {

template <int T, int N, int V>
struct BGeom {
    static constexpr int NT = T;
    static constexpr int NV = N;
    static constexpr int VEC = V;
};

// Longest row of the block-row kernels, in floats.
constexpr int64_t kBlockRowMax = 16384;

// Calls f(BGeom<NT, NV, VEC>{}) for rows of 1025..max_cols floats (max_cols
// <= kBlockRowMax) and returns true, or returns false.  Every thread holds at
// most 16 floats of the row (4 float4 or 16 scalars).
template <typename F>
bool with_block_geometry(bool vec4, int64_t cols, int64_t max_cols, F&& f) {
    if (cols <= 1024 || cols > max_cols || cols > kBlockRowMax) return false;
    if (vec4) {
        if (cols <= 2048) f(BGeom<128, 4, 4>{});
        else if (cols <= 4096) f(BGeom<256, 4, 4>{});
        else if (cols <= 8192) f(BGeom<512, 4, 4>{});
        else f(BGeom<1024, 4, 4>{});
    } else {
        if (cols <= 2048) f(BGeom<128, 16, 1>{});
        else if (cols <= 4096) f(BGeom<256, 16, 1>{});
        else if (cols <= 8192) f(BGeom<512, 16, 1>{});
        else f(BGeom<1024, 16, 1>{});
    }
    return true;
}

// Block-wide reductions over NT threads with double-buffered partials.
// `sc` points to 2 * 2 * (NT / 32) floats of shared memory.  Every thread of
// the block must make the same sequence of calls.
template <int NT>
struct BlockReduce {
    static constexpr int W = NT / 32;
    float* sc;
    int buf;

    __device__ __forceinline__ explicit BlockReduce(float* s) : sc(s), buf(0) {}

    __device__ __forceinline__ float* next() {
        float* p = sc + buf * 2 * W;
        buf ^= 1;
        return p;
    }

    __device__ __forceinline__ float sum(float v) {
        v = group_sum<32>(v);
        float* p = next();
        if ((threadIdx.x & 31) == 0) p[threadIdx.x >> 5] = v;
        __syncthreads();
        float r = p[0];
#pragma unroll
        for (int i = 1; i < W; ++i) r += p[i];
        return r;
    }

    __device__ __forceinline__ float max(float v) {
        v = group_max<32>(v);
        float* p = next();
        if ((threadIdx.x & 31) == 0) p[threadIdx.x >> 5] = v;
        __syncthreads();
        float r = p[0];
#pragma unroll
        for (int i = 1; i < W; ++i) r = fmaxf(r, p[i]);
        return r;
    }

    // Two sums in one round.
    __device__ __forceinline__ void sum2(float& a, float& b) {
        a = group_sum<32>(a);
        b = group_sum<32>(b);
        float* p = next();
        if ((threadIdx.x & 31) == 0) {
            p[threadIdx.x >> 5] = a;
            p[W + (threadIdx.x >> 5)] = b;
        }
        __syncthreads();
        float ra = p[0], rb = p[W];
#pragma unroll
        for (int i = 1; i < W; ++i) {
            ra += p[i];
            rb += p[W + i];
        }
        a = ra;
        b = rb;
    }

    __device__ __forceinline__ int min_int(int v) {
        v = group_min_int<32>(v);
        float* p = next();
        if ((threadIdx.x & 31) == 0) p[threadIdx.x >> 5] = __int_as_float(v);
        __syncthreads();
        int r = __float_as_int(p[0]);
#pragma unroll
        for (int i = 1; i < W; ++i) r = min(r, __float_as_int(p[i]));
        return r;
    }

    // Two maxima in one round.
    __device__ __forceinline__ void max2(float& a, float& b) {
        a = group_max<32>(a);
        b = group_max<32>(b);
        float* p = next();
        if ((threadIdx.x & 31) == 0) {
            p[threadIdx.x >> 5] = a;
            p[W + (threadIdx.x >> 5)] = b;
        }
        __syncthreads();
        float ra = p[0], rb = p[W];
#pragma unroll
        for (int i = 1; i < W; ++i) {
            ra = fmaxf(ra, p[i]);
            rb = fmaxf(rb, p[W + i]);
        }
        a = ra;
        b = rb;
    }

    // Max of a float and sum of an int in one round (the int is carried as
    // its bit pattern; counts are far below 2^24, so float adds would do, but
    // the bits keep it exact whatever the count).
    __device__ __forceinline__ void max_count(float& m, int& n) {
        m = group_max<32>(m);
        n = group_sum_int<32>(n);
        float* p = next();
        if ((threadIdx.x & 31) == 0) {
            p[threadIdx.x >> 5] = m;
            p[W + (threadIdx.x >> 5)] = __int_as_float(n);
        }
        __syncthreads();
        float rm = p[0];
        int rn = __float_as_int(p[W]);
#pragma unroll
        for (int i = 1; i < W; ++i) {
            rm = fmaxf(rm, p[i]);
            rn += __float_as_int(p[W + i]);
        }
        m = rm;
        n = rn;
    }
};

// Grid of a block-row kernel: one CTA per row up to the grid-size cap; the
// kernels walk rows with a grid stride beyond it.
inline unsigned block_row_grid(int64_t rows) {
    int64_t b = rows;
    if (b > (int64_t(1) << 20)) b = int64_t(1) << 20;
    return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace rowops
