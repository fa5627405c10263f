// rmsnorm.cu - RMSNorm forward/backward and column sums (pulsatrix
// rms_norm_forward, rms_norm_backward, column_sums).
//
//   forward   rms_i = sqrt(mean_j x_ij^2 + eps), out_ij = gamma_j x_ij / rms_i
//   backward  g' = g * gamma, dx = (g' - x * mean(g' x) / rms^2) / rms,
//             gamma_terms_ij = g_ij x_ij / rms_i   (per-row gamma contributions)
//   column sums  out_j = beta * out_j + sum_i in_ij
//
// Forward and backward are group kernels (geometry of common.cuh), block-row
// kernels for rows of 1025..16384 floats (block_rows.cuh) and a streaming
// fallback.  Column sums need no workspace: a cluster of 8 CTAs owns a
// tile of 32 columns and splits the rows into 8 consecutive ranges; inside a
// CTA warp w adds rows w, w+16, ... of its range in order, the 16 warps are
// combined in warp order through shared memory and the 8 CTAs in rank order
// through distributed shared memory.  The association is fixed, so results are
// deterministic (a blocked order, not one sequential pass over the rows).
#include "block_rows.cuh"
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

// Blocks of any whole number of warps up to 1024 threads, for the balanced
// launch (launch.h, balanced_groups).
template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(1024)
rms_fwd_group(const float* __restrict__ x, const float* __restrict__ gamma, float* __restrict__ out,
              float* __restrict__ row_rms, int64_t rows, int cols, float eps) {
    const int GPB = int(blockDim.x) / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
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
                for (int e = 0; e < VEC; ++e) v[k][e] = 0.f;
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss = fmaf(v[k][e], v[k][e], ss);
        ss = group_sum<LANES>(ss);
        const float rms = sqrtf(ss * inv_cols + eps);
        const float inv = 1.0f / rms;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float gm[VEC], o[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = gm[e] * (v[k][e] * inv);
                st_chunk<VEC>(out + off + c * VEC, o);
            }
        }
        if (live && g == 0) row_rms[row] = rms;
    }
}

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
rms_bwd_group(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ x,
              const float* __restrict__ row_rms, float* __restrict__ dx, float* __restrict__ terms,
              int64_t rows, int cols) {
    constexpr int GPB = kBlockThreads / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float a[NV][VEC], h[NV][VEC], gm[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk<VEC>(dy + off + c * VEC, a[k]);
                ld_chunk<VEC>(x + off + c * VEC, h[k]);
                ld_chunk<VEC>(gamma + c * VEC, gm[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = h[k][e] = gm[k][e] = 0.f;
            }
        }
        const float r = live ? __ldg(row_rms + row) : 1.f;
        const float inv = 1.0f / r;
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) s = fmaf(a[k][e] * gm[k][e], h[k][e], s);
        s = group_sum<LANES>(s) * inv_cols;
        const float c2 = s * inv * inv;  // mean(g' x) / r^2
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC], t[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    o[e] = (a[k][e] * gm[k][e] - h[k][e] * c2) * inv;
                    t[e] = a[k][e] * h[k][e] * inv;
                }
                st_chunk<VEC>(dx + off + c * VEC, o);
                st_chunk<VEC>(terms + off + c * VEC, t);
            }
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
rms_fwd_rowblock(const float* __restrict__ x, const float* __restrict__ gamma, float* __restrict__ out,
                 float* __restrict__ row_rms, int64_t rows, int64_t cols, float eps) {
    __shared__ float scratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        float ss = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(x + off + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss = fmaf(v[e], v[e], ss);
        }
        const float rms = sqrtf(block_sum<kBlockThreads>(ss, scratch) / float(cols) + eps);
        const float inv = 1.0f / rms;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC], gm[VEC];
            ld_chunk<VEC>(x + off + c * VEC, v);
            ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[e] = gm[e] * (v[e] * inv);
            st_chunk<VEC>(out + off + c * VEC, v);
        }
        if (threadIdx.x == 0) row_rms[row] = rms;
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
rms_bwd_rowblock(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ x,
                 const float* __restrict__ row_rms, float* __restrict__ dx, float* __restrict__ terms,
                 int64_t rows, int64_t cols) {
    __shared__ float scratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * cols;
        float s = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float a[VEC], h[VEC], gm[VEC];
            ld_chunk<VEC>(dy + off + c * VEC, a);
            ld_chunk<VEC>(x + off + c * VEC, h);
            ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
            for (int e = 0; e < VEC; ++e) s = fmaf(a[e] * gm[e], h[e], s);
        }
        s = block_sum<kBlockThreads>(s, scratch) / float(cols);
        const float inv = 1.0f / __ldg(row_rms + row);
        const float c2 = s * inv * inv;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float a[VEC], h[VEC], gm[VEC], o[VEC], t[VEC];
            ld_chunk<VEC>(dy + off + c * VEC, a);
            ld_chunk<VEC>(x + off + c * VEC, h);
            ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                o[e] = (a[e] * gm[e] - h[e] * c2) * inv;
                t[e] = a[e] * h[e] * inv;
            }
            st_chunk<VEC>(dx + off + c * VEC, o);
            st_chunk<VEC>(terms + off + c * VEC, t);
        }
    }
}

// ------------------------------------------------------ block-row kernels
// Rows of 1025..16384 floats, one CTA per row in registers (block_rows.cuh).

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
rms_fwd_brow(const float* __restrict__ x, const float* __restrict__ gamma, float* __restrict__ out,
             float* __restrict__ row_rms, int64_t rows, int cols, float eps) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float v[NV][VEC];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(x + off + c * VEC, v[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss = fmaf(v[k][e], v[k][e], ss);
        }
        const float rms = sqrtf(red.sum(ss) * inv_cols + eps);
        const float inv = 1.0f / rms;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float gm[VEC], o[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = gm[e] * (v[k][e] * inv);
                st_chunk<VEC>(out + off + c * VEC, o);
            }
        }
        if (threadIdx.x == 0) row_rms[row] = rms;
    }
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
rms_bwd_brow(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ x,
             const float* __restrict__ row_rms, float* __restrict__ dx, float* __restrict__ terms, int64_t rows,
             int cols) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        float a[NV][VEC], h[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(dy + off + c * VEC, a[k]);
                ld_chunk<VEC>(x + off + c * VEC, h[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = h[k][e] = 0.f;
            }
        }
        const float inv = 1.0f / __ldg(row_rms + row);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float gm[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s = fmaf(a[k][e] * gm[e], h[k][e], s);
            }
        }
        const float c2 = red.sum(s) * inv_cols * inv * inv;  // mean(g' x) / r^2
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float gm[VEC], o[VEC], t[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    o[e] = (a[k][e] * gm[e] - h[k][e] * c2) * inv;
                    t[e] = a[k][e] * h[k][e] * inv;
                }
                st_chunk<VEC>(dx + off + c * VEC, o);
                st_chunk<VEC>(terms + off + c * VEC, t);
            }
        }
    }
}

// ----------------------------------------------------------- column sums

constexpr int kColTile = 32;
constexpr int kColCluster = 8;
constexpr int kColWarps = 16;
constexpr int kColInFlight = 16;  // loads per thread in flight

__device__ __forceinline__ void csum_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void csum_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__global__ void __launch_bounds__(kColWarps * 32)
column_sums_cluster(const float* __restrict__ in, float* __restrict__ out, int64_t rows, int64_t cols,
                    float beta) {
    namespace cg = cooperative_groups;
    __shared__ float part[kColWarps][kColTile];
    __shared__ float cta_sum[kColTile];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t tile = blockIdx.x / kColCluster;
    const int64_t col = tile * kColTile + lane;
    const int64_t per = (rows + kColCluster - 1) / kColCluster;
    const int64_t r0 = rank * per;
    const int64_t r1 = r0 + per < rows ? r0 + per : rows;
    float s = 0.f;
    if (col < cols) {
        int64_t i = r0 + w;
        // kColInFlight independent loads in flight (a warp reads one 128-byte
        // row segment per load), added in row order
        for (; i + (kColInFlight - 1) * kColWarps < r1; i += kColInFlight * kColWarps) {
            float v[kColInFlight];
#pragma unroll
            for (int u = 0; u < kColInFlight; ++u) v[u] = __ldg(in + (i + u * kColWarps) * cols + col);
#pragma unroll
            for (int u = 0; u < kColInFlight; ++u) s += v[u];
        }
        for (; i < r1; i += kColWarps) s += __ldg(in + i * cols + col);
    }
    part[w][lane] = s;
    __syncthreads();
    if (w == 0) {
        float t = part[0][lane];
#pragma unroll
        for (int q = 1; q < kColWarps; ++q) t += part[q][lane];
        cta_sum[lane] = t;
    }
    csum_arrive();
    csum_wait();
    if (rank == 0 && w == 0 && col < cols) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < kColCluster; ++q) t += cluster.map_shared_rank(cta_sum, q)[lane];
        out[col] = (beta == 0.f ? 0.f : beta * out[col]) + t;
    }
    csum_arrive();
    csum_wait();  // keep cta_sum alive until rank 0 has read it
}

}  // namespace

cudaError_t launch_rmsnorm_fwd(const float* x, const float* gamma, float* out, float* row_rms, int64_t rows,
                               int64_t cols, float eps, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        const BalancedLaunch bl = balanced_groups(rows, G::LANES);
        if (bl.threads)
            rms_fwd_group<G::LANES, G::NV, G::VEC><<<bl.grid, bl.threads, 0, stream>>>(
                x, gamma, out, row_rms, rows, int(cols), eps);
        else
            rms_fwd_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
                x, gamma, out, row_rms, rows, int(cols), eps);
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                rms_fwd_brow<G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                    x, gamma, out, row_rms, rows, int(cols), eps);
            })) {
        } else if (vec4)
            rms_fwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, gamma, out, row_rms, rows, cols, eps);
        else
            rms_fwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, gamma, out, row_rms, rows, cols, eps);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bwd(const float* dy, const float* gamma, const float* x, const float* row_rms,
                               float* dx, float* terms, int64_t rows, int64_t cols, bool vec4,
                               cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        rms_bwd_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            dy, gamma, x, row_rms, dx, terms, rows, int(cols));
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                rms_bwd_brow<G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                    dy, gamma, x, row_rms, dx, terms, rows, int(cols));
            })) {
        } else if (vec4)
            rms_bwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(dy, gamma, x, row_rms, dx, terms,
                                                                              rows, cols);
        else
            rms_bwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(dy, gamma, x, row_rms, dx, terms,
                                                                              rows, cols);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_column_sums(const float* in, float* out, int64_t rows, int64_t cols, float beta,
                               cudaStream_t stream) {
    const int64_t tiles = (cols + kColTile - 1) / kColTile;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles * kColCluster));
    cfg.blockDim = dim3(kColWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kColCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, column_sums_cluster, in, out, rows, cols, beta);
    note_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace rowops
