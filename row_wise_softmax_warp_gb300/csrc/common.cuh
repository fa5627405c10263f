// common.cuh - device helpers shared by the row-op kernels (sm_103a).
//
// Row geometry used by every "group" kernel: a row of `cols` floats is split
// into chunks of VEC consecutive floats (VEC = 4: one 128-bit access; VEC = 1:
// scalar).  A group of LANES consecutive lanes of a warp owns one row; lane g of
// the group holds chunks g, g + LANES, ..., g + (NV-1)*LANES, so every load and
// store instruction of a warp touches consecutive addresses.  A warp holds
// 32 / LANES rows at a time.  Reductions inside a group are xor-butterfly
// shuffles, which leave the bit-identical result in every lane of the group.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

namespace rowops {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kBlockThreads = 256;

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;     // ln(2)

// 2^x by the MUFU ex2 instruction (subnormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// exp(x - m) as 2^((x - m) * log2(e)).  The difference is taken first so that no
// intermediate overflows for finite x and m (m * log2(e) would for |m| > 2.3e38).
__device__ __forceinline__ float exp_shifted(float x, float m) {
    return ex2_approx((x - m) * kLog2e);
}

// ----------------------------------------------------------------- memory

template <int VEC>
__device__ __forceinline__ void ld_chunk(const float* p, float (&v)[VEC]) {
    if constexpr (VEC == 4) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        v[0] = __ldg(p);
    }
}

// Coherent load, for kernels whose output may be the same buffer as the input.
template <int VEC>
__device__ __forceinline__ void ld_chunk_coherent(const float* p, float (&v)[VEC]) {
    if constexpr (VEC == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        v[0] = *p;
    }
}

template <int VEC>
__device__ __forceinline__ void st_chunk(float* p, const float (&v)[VEC]) {
    if constexpr (VEC == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        *p = v[0];
    }
}

template <int VEC>
__device__ __forceinline__ void st_zero_chunk(float* p) {
    if constexpr (VEC == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        *p = 0.f;
    }
}

// VEC mask bytes; the VEC = 4 path needs the row's mask bytes 4-byte aligned.
template <int VEC>
__device__ __forceinline__ void ld_mask(const uint8_t* p, bool (&a)[VEC]) {
    if constexpr (VEC == 4) {
        const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
        a[0] = (w & 0xffu) != 0; a[1] = (w & 0xff00u) != 0;
        a[2] = (w & 0xff0000u) != 0; a[3] = (w & 0xff000000u) != 0;
    } else {
        a[0] = __ldg(p) != 0;
    }
}

// VEC float mask values; an entry is allowed when its mask value is not 0.0.
template <int VEC>
__device__ __forceinline__ void ld_mask(const float* p, bool (&a)[VEC]) {
    float m[VEC];
    ld_chunk<VEC>(p, m);
#pragma unroll
    for (int e = 0; e < VEC; ++e) a[e] = m[e] != 0.0f;
}

// ----------------------------------------------------------- group reductions

template <int LANES>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

template <int LANES>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

template <int LANES>
__device__ __forceinline__ int group_sum_int(int v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

template <int LANES>
__device__ __forceinline__ float group_min(float v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

template <int LANES>
__device__ __forceinline__ int group_min_int(int v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

template <int LANES>
__device__ __forceinline__ int group_max_int(int v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

// Sum across the groups of a warp that sit at the same position g (lanes
// g, g + LANES, ...): used to merge per-group column partials.
template <int LANES>
__device__ __forceinline__ float across_groups_sum(float v) {
#pragma unroll
    for (int o = LANES; o < 32; o <<= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

// ------------------------------------------------------ block reductions
// Every thread of the block gets the same value; partials are combined in
// warp order, so the result is deterministic.  `scratch` holds NT/32 floats and
// is free again when the function returns.

template <int NT>
__device__ __forceinline__ float block_max(float v, float* scratch) {
    v = group_max<32>(v);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    float r = scratch[0];
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) r = fmaxf(r, scratch[i]);
    __syncthreads();
    return r;
}

template <int NT>
__device__ __forceinline__ float block_sum(float v, float* scratch) {
    v = group_sum<32>(v);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    float r = scratch[0];
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) r += scratch[i];
    __syncthreads();
    return r;
}

template <int NT>
__device__ __forceinline__ int block_sum_int(int v, int* scratch) {
    v = group_sum_int<32>(v);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    int r = 0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) r += scratch[i];
    __syncthreads();
    return r;
}

// (max, sum of exp(x - max)) pairs: the state of a one-pass softmax reduction.
struct MaxSum {
    float m;
    float s;
};

__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    return {m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}

// Fold one value into a running (max, sum).
__device__ __forceinline__ MaxSum ms_push(MaxSum a, float x) {
    if (x > a.m) {
        const float s = (a.m == -INFINITY) ? 1.f : a.s * expf(a.m - x) + 1.f;
        return {x, s};
    }
    return {a.m, a.s + expf(x - a.m)};
}

template <int NT>
__device__ __forceinline__ MaxSum block_maxsum(MaxSum v, float* scratch /* 2*NT/32 */) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum t{__shfl_xor_sync(kFullMask, v.m, o), __shfl_xor_sync(kFullMask, v.s, o)};
        v = ms_merge(v, t);
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        scratch[2 * w] = v.m;
        scratch[2 * w + 1] = v.s;
    }
    __syncthreads();
    MaxSum r{scratch[0], scratch[1]};
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) r = ms_merge(r, MaxSum{scratch[2 * i], scratch[2 * i + 1]});
    __syncthreads();
    return r;
}

// Order-preserving map of a float to uint32 (-0 and +0 map to the same key,
// NaN is not handled: callers route rows with NaN elsewhere).
__device__ __forceinline__ uint32_t ordered_key(float x) {
    const uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace rowops
