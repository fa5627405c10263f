// lse_ce.cu - per-row logsumexp and fused softmax cross-entropy (loss + logits
// gradient), and the fixed-order mean of the row losses.
//
// Kernel shapes:
//   *_group    : rows of up to 1024 floats in registers (common.cuh).
//   *_brow     : rows of 1025..8192 floats in registers, one CTA per row
//                (block_rows.cuh).
//   longer rows: the bulk-copy pipeline of tma_rows.cu.
//   *_rowblock : any length and alignment, streaming two passes (rows whose
//                output sits on another 16-byte phase than the input).
#include "block_rows.cuh"
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

// MicroGPT CuBLASBackend::fused_softmax_ce_grad / pulsatrix logsumexp_rows.

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
lse_group(const float* __restrict__ x, float* __restrict__ lse, int64_t rows, int cols) {
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
                ld_chunk<VEC>(x + off + c * VEC, v[k]);
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
        if (!isinf(m)) {
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) s += exp_shifted(v[k][e], m);
        }
        s = group_sum<LANES>(s);
        if (live && g == 0) lse[row] = isinf(m) ? m : m + logf(s);
    }
}

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
ce_group(const float* __restrict__ x, const int32_t* __restrict__ targets, float* __restrict__ grad,
         float* __restrict__ row_loss, int64_t rows, int cols, float grad_scale) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        const int t = live ? __ldg(targets + row) : -1;
        const bool tvalid = t >= 0 && t < cols;
        float v[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk<VEC>(x + off + c * VEC, v[k]);
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
                for (int e = 0; e < VEC; ++e)
                    o[e] = grad_scale * (v[k][e] * inv - ((tvalid && c * VEC + e == t) ? 1.f : 0.f));
                st_chunk<VEC>(grad + off + c * VEC, o);
            }
        }
        if (live && g == 0) {
            const float lse = m + logf(s);
            row_loss[row] = tvalid ? lse - __ldg(x + off + t) : __int_as_float(0x7fc00000);
        }
    }
}

// ------------------------------------------------------ block-row kernels
// Rows of 1025..16384 floats, one CTA per row in registers (block_rows.cuh);
// the arithmetic of lse_group / ce_group with block reductions.

template <int NT, int NV, int VEC>
__device__ __forceinline__ float brow_load_max(const float* __restrict__ r, int nch, float (&v)[NV][VEC]) {
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = int(threadIdx.x) + k * NT;
        if (c < nch) {
            ld_chunk<VEC>(r + c * VEC, v[k]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
    }
    return m;
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
lse_brow(const float* __restrict__ x, float* __restrict__ lse, int64_t rows, int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        float v[NV][VEC];
        const float m = red.max(brow_load_max<NT, NV, VEC>(x + row * int64_t(cols), nch, v));
        float s = 0.f;
        if (!isinf(m)) {
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) s += exp_shifted(v[k][e], m);
        }
        s = red.sum(s);
        if (threadIdx.x == 0) lse[row] = isinf(m) ? m : m + logf(s);
    }
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
ce_brow(const float* __restrict__ x, const int32_t* __restrict__ targets, float* __restrict__ grad,
        float* __restrict__ row_loss, int64_t rows, int cols, float grad_scale) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        const int t = __ldg(targets + row);
        const bool tvalid = t >= 0 && t < cols;
        float v[NV][VEC];
        const float m = red.max(brow_load_max<NT, NV, VEC>(x + off, nch, v));
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
                for (int e = 0; e < VEC; ++e)
                    o[e] = grad_scale * (v[k][e] * inv - ((tvalid && c * VEC + e == t) ? 1.f : 0.f));
                st_chunk<VEC>(grad + off + c * VEC, o);
            }
        }
        if (threadIdx.x == 0) {
            const float l = m + logf(s);
            row_loss[row] = tvalid ? l - __ldg(x + off + t) : __int_as_float(0x7fc00000);
        }
    }
}

// ------------------------------------------------------------ streaming

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
lse_rowblock(const float* __restrict__ x, float* __restrict__ lse, int64_t rows, int64_t cols) {
    __shared__ float scratch[2 * kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * cols;
        MaxSum a{-INFINITY, 0.f};
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) a = ms_push(a, v[e]);
        }
        a = block_maxsum<kBlockThreads>(a, scratch);
        if (threadIdx.x == 0) lse[row] = isinf(a.m) ? a.m : a.m + logf(a.s);
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
ce_rowblock(const float* __restrict__ x, const int32_t* __restrict__ targets,
            float* __restrict__ grad, float* __restrict__ row_loss, int64_t rows, int64_t cols,
            float grad_scale) {
    __shared__ float scratch[2 * kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * cols;
        float* gr = grad + row * cols;
        MaxSum a{-INFINITY, 0.f};
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) a = ms_push(a, v[e]);
        }
        a = block_maxsum<kBlockThreads>(a, scratch);
        const int64_t t = __ldg(targets + row);
        const bool tvalid = t >= 0 && t < cols;
        const float inv = 1.0f / a.s;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                v[e] = grad_scale * (expf(v[e] - a.m) * inv - ((tvalid && c * VEC + e == t) ? 1.f : 0.f));
            st_chunk<VEC>(gr + c * VEC, v);
        }
        if (threadIdx.x == 0)
            row_loss[row] = tvalid ? (a.m + logf(a.s)) - __ldg(xr + t) : __int_as_float(0x7fc00000);
    }
}

// Mean of the row losses.  Launched as a programmatic dependent of the loss
// kernel: it waits here for that grid.  One block, fixed order: thread t adds
// rows t, t+1024, ... in order (eight loads in flight), warps combine with a
// fixed xor butterfly, then warp 0 combines the 32 warp sums the same way.
//
// The sum is carried as a double-word fp32 value hi + lo (about 48 significant
// bits), whose additions use only the fp32 pipes: a single block spends about
// 8 us on GB300's narrow fp64 pipe converting and adding 8192 losses in
// double, against about 1 us this way.  Error-free transformations:
//   TwoSum(a, b)   (Knuth): s = fl(a + b) and e with a + b = s + e exactly;
//   Fast2Sum(a, b) (Dekker, |a| >= |b|): the same with three operations;
// word + float and word + word follow the double-word additions of Joldes,
// Muller and Popescu (2017) ("DWPlusFP" and "AccurateDWPlusDW"), each with a
// relative error of order u^2, u = 2^-24.  A sum that is not finite in
// this form (an infinite or NaN loss, or fp32 overflow) is recomputed in double
// in the same fixed order, so such means are IEEE double sums as before.
struct DWord {
    float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bv = s - a;
    e = (a - (s - bv)) + (b - bv);
}

__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    e = b - (s - a);
}

__device__ __forceinline__ DWord dw_add(DWord x, float y) {
    float sh, sl, zh, zl;
    two_sum(x.hi, y, sh, sl);
    fast_two_sum(sh, x.lo + sl, zh, zl);
    return {zh, zl};
}

__device__ __forceinline__ DWord dw_add(DWord x, DWord y) {
    float sh, sl, th, tl, vh, vl, zh, zl;
    two_sum(x.hi, y.hi, sh, sl);
    two_sum(x.lo, y.lo, th, tl);
    fast_two_sum(sh, sl + th, vh, vl);
    fast_two_sum(vh, tl + vl, zh, zl);
    return {zh, zl};
}

__device__ __forceinline__ DWord dw_shfl_xor(DWord v, int o) {
    return {__shfl_xor_sync(kFullMask, v.hi, o), __shfl_xor_sync(kFullMask, v.lo, o)};
}

__global__ void __launch_bounds__(1024)
ce_mean(const float* row_loss, int64_t rows, double* __restrict__ mean) {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    __shared__ DWord part[32];
    __shared__ double dpart[32];
    __shared__ int redo;
    DWord s{0.f, 0.f};
    int64_t i = threadIdx.x;
    for (; i + 7 * 1024 < rows; i += 8 * 1024) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = row_loss[i + u * 1024];
#pragma unroll
        for (int u = 0; u < 8; ++u) s = dw_add(s, v[u]);
    }
    for (; i < rows; i += 1024) s = dw_add(s, row_loss[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = dw_add(s, dw_shfl_xor(s, o));
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        DWord t = part[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t = dw_add(t, dw_shfl_xor(t, o));
        if (threadIdx.x == 0) {
            const bool finite = isfinite(t.hi) && isfinite(t.lo);
            redo = finite ? 0 : 1;
            if (finite) *mean = (double(t.hi) + double(t.lo)) / double(rows);
        }
    }
    __syncthreads();
    if (!redo) return;  // block-uniform
    // Non-finite in fp32: the same fixed order in double.
    double d = 0.0;
    for (i = threadIdx.x; i < rows; i += 1024) d += double(row_loss[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(kFullMask, d, o);
    if ((threadIdx.x & 31) == 0) dpart[threadIdx.x >> 5] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < 32; ++w) t += dpart[w];
        *mean = t / double(rows);
    }
}

__global__ void fill_value(float* __restrict__ p, int64_t n, float v) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        p[i] = v;
}

}  // namespace

// ------------------------------------------------------------ launchers

// Longest rows of the block-row kernels before the TMA-streamed kernel takes
// over.  On GB300 at 16384 floats the TMA kernel is ahead (logsumexp 37.5
// against 45.7 us, cross-entropy 62.1 against 68.2 us on 2048 rows); at 8192
// and below the block-row kernels are (logsumexp 33.4 against 53.9 us on 4096
// rows, 31.4 against 166.6 us on 16384 x 2048).
constexpr int64_t kLseBrowMax = 8192;
constexpr int64_t kCeBrowMax = 8192;

cudaError_t launch_logsumexp(const float* x, float* lse, int64_t rows, int64_t cols, bool vec4,
                             cudaStream_t stream) {
    if (cols == 0) {
        const int64_t b = (rows + 255) / 256;
        fill_value<<<unsigned(b > 4096 ? 4096 : b), 256, 0, stream>>>(lse, rows, -INFINITY);
        note_launches(1);
        return cudaGetLastError();
    }
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        lse_group<G::LANES, G::NV, G::VEC>
            <<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(x, lse, rows, int(cols));
    });
    cudaError_t err = cudaSuccess;
    if (!done) {
        if (with_block_geometry(vec4, cols, kLseBrowMax, [&](auto geo) {
                using G = decltype(geo);
                lse_brow<G::NT, G::NV, G::VEC>
                    <<<block_row_grid(rows), G::NT, 0, stream>>>(x, lse, rows, int(cols));
            })) {
        } else if (launch_lse_tma(x, lse, rows, cols, stream, &err)) {
        } else if (vec4)
            lse_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, lse, rows, cols);
        else
            lse_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, lse, rows, cols);
    }
    note_launches(1);
    const cudaError_t last = cudaGetLastError();
    return err != cudaSuccess ? err : last;
}

cudaError_t launch_softmax_ce(const float* logits, const int32_t* targets, float* grad,
                              float* row_loss, double* mean_loss, int64_t rows, int64_t cols,
                              float grad_scale, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        ce_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            logits, targets, grad, row_loss, rows, int(cols), grad_scale);
    });
    cudaError_t err = cudaSuccess;
    if (!done) {
        if (with_block_geometry(vec4, cols, kCeBrowMax, [&](auto geo) {
                using G = decltype(geo);
                ce_brow<G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                    logits, targets, grad, row_loss, rows, int(cols), grad_scale);
            })) {
        } else if (launch_ce_tma(logits, targets, grad, row_loss, rows, cols, grad_scale, stream, &err)) {
        } else if (vec4)
            ce_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(logits, targets, grad,
                                                                         row_loss, rows, cols,
                                                                         grad_scale);
        else
            ce_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(logits, targets, grad,
                                                                         row_loss, rows, cols,
                                                                         grad_scale);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    note_launches(1);
    return launch_row_mean(row_loss, rows, mean_loss, stream);
}

cudaError_t launch_row_mean(const float* row_loss, int64_t rows, double* mean_loss, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1024);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, ce_mean, row_loss, rows, mean_loss);
    note_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace rowops
