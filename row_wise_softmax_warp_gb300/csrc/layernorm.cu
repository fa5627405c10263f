// layernorm.cu - LayerNorm forward (out, xhat, inv_std) and backward
// (dx, dgamma, dbeta) over the columns of a row-major matrix.
//
// Forward statistics are a two-pass mean/variance of the register-held row.
// The mean is accumulated around a shift (the row's first entry), so rows whose
// mean is large next to their spread (mean 5, std 0.1) keep full fp32 accuracy.
//
// Backward writes dx per row and the column sums dgamma_j = sum_i dy*xhat,
// dbeta_j = sum_i dy in two deterministic stages:
//   stage 1 writes one partial of the column sums per CTA (or cluster) to the
//     workspace: rows of 384..1024 floats on 16-byte boundaries take
//     ln_bwd_cols (column owners, the CTA's whole block of rows staged in
//     shared memory with cp.async) or, when the block does not fit,
//     ln_bwd_tma (ln_bwd_tma.cu: row blocks through the bulk-copy ring);
//     other rows of up to 1024 floats take ln_bwd_group (clusters of 8 CTAs:
//     groups accumulate their columns in registers, CTAs add their warps in
//     warp order through shared memory, the cluster adds its CTAs in rank
//     order through distributed shared memory); rows of 1025..8192 floats
//     take ln_bwd_brow (one CTA per row at a time, each thread keeping its
//     columns' partials in registers across the CTA's rows); longer rows take
//     ln_bwd_long (one 1024-thread CTA per SM, two passes over each row, each
//     thread's column partials in shared memory or, past 25600 floats, in
//     the CTA's workspace slot);
//   stage 2 (ln_params_reduce, a programmatic dependent of stage 1) adds the
//     partials per column in increasing order.
#include "block_rows.cuh"
#include "common.cuh"
#include "launch.h"

namespace rowops {
namespace {

constexpr int kLnClusterCtas = 8;

// -------------------------------------------------------------- forward
// pulsatrix HIPBackend::layer_norm_forward / TorchLean layer normalisation.

// Blocks of any whole number of warps up to 1024 threads, for the balanced
// launch (launch.h, balanced_groups).
template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(1024)
ln_fwd_group(const float* __restrict__ x, const float* __restrict__ gamma,
             const float* __restrict__ beta, float* __restrict__ out, float* __restrict__ xhat,
             float* __restrict__ inv_std, int64_t rows, int cols, float eps) {
    const int GPB = int(blockDim.x) / LANES;
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int lane = threadIdx.x & 31;
    const int leader = lane - g;  // lane of this group's first lane
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
        const float shift = __shfl_sync(kFullMask, v[0][0], leader);  // the row's first entry
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (g + k * LANES < nch)
#pragma unroll
                for (int e = 0; e < VEC; ++e) s += v[k][e] - shift;
        s = group_sum<LANES>(s);
        const float mean = shift + s * inv_cols;
        float q = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (g + k * LANES < nch)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    v[k][e] -= mean;
                    q = fmaf(v[k][e], v[k][e], q);
                }
        q = group_sum<LANES>(q);
        const float r = 1.0f / sqrtf(q * inv_cols + eps);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float gm[VEC], bt[VEC], h[VEC], o[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
                ld_chunk<VEC>(beta + c * VEC, bt);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    h[e] = v[k][e] * r;
                    o[e] = fmaf(gm[e], h[e], bt[e]);
                }
                st_chunk<VEC>(xhat + off + c * VEC, h);
                st_chunk<VEC>(out + off + c * VEC, o);
            }
        }
        if (live && g == 0) inv_std[row] = r;
    }
}

template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
ln_fwd_rowblock(const float* __restrict__ x, const float* __restrict__ gamma,
                const float* __restrict__ beta, float* __restrict__ out, float* __restrict__ xhat,
                float* __restrict__ inv_std, int64_t rows, int64_t cols, float eps) {
    __shared__ float scratch[kBlockThreads / 32];
    const int64_t nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * cols;
        const float shift = __ldg(xr);
        float s = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) s += v[e] - shift;
        }
        const float mean = shift + block_sum<kBlockThreads>(s, scratch) * inv_cols;
        float q = 0.f;
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float d = v[e] - mean;
                q = fmaf(d, d, q);
            }
        }
        const float r = 1.0f / sqrtf(block_sum<kBlockThreads>(q, scratch) * inv_cols + eps);
        for (int64_t c = threadIdx.x; c < nch; c += kBlockThreads) {
            float v[VEC], gm[VEC], bt[VEC], o[VEC];
            ld_chunk<VEC>(xr + c * VEC, v);
            ld_chunk<VEC>(gamma + c * VEC, gm);
            ld_chunk<VEC>(beta + c * VEC, bt);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[e] = (v[e] - mean) * r;
                o[e] = fmaf(gm[e], v[e], bt[e]);
            }
            st_chunk<VEC>(xhat + row * cols + c * VEC, v);
            st_chunk<VEC>(out + row * cols + c * VEC, o);
        }
        if (threadIdx.x == 0) inv_std[row] = r;
    }
}

// ------------------------------------------------------------- backward
// TorchLean layer-normalisation VJP / MicroGPT layer_norm_backward:
//   g' = dy*gamma, dx = r*(g' - mean(g') - xhat*mean(g'*xhat)),
//   dgamma_j = sum_i dy*xhat, dbeta_j = sum_i dy.

// Resident stage-1 CTAs per SM: shared memory holds (GPB + 1) x 2 x MAXC
// floats per CTA, so three CTAs of the 1024-float geometries fit and four of
// the others; the launch bounds give each geometry the registers of that
// residency.
constexpr int ln_bwd_blocks_per_sm(int maxc) { return maxc > 768 ? 3 : 4; }

// Geometry of the stage-1 grid, a pure function of rows, cols and the SM
// count: 8 rows per CTA, at most one wave of resident CTAs (and 1024), in
// whole clusters; CTAs walk more rows beyond that.
inline int64_t ln_bwd_ctas(int64_t rows, int64_t cols) {
    const int sms = sm_count();
    int64_t cap = int64_t(sms > 0 ? sms : 1) * ln_bwd_blocks_per_sm(cols > 768 ? 1024 : 768);
    cap = cap / kLnClusterCtas * kLnClusterCtas;
    if (cap > 1024) cap = 1024;
    if (cap < kLnClusterCtas) cap = kLnClusterCtas;
    int64_t b = (rows + 7) / 8;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return (b + kLnClusterCtas - 1) / kLnClusterCtas * kLnClusterCtas;
}
inline int64_t ln_bwd_partials(int64_t rows, int64_t cols) { return ln_bwd_ctas(rows, cols) / kLnClusterCtas; }

__device__ __forceinline__ void cl_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cl_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Dynamic shared memory: red[GPB groups][2][MAXC] (each group's column
// partials, dgamma then dbeta) then bpart[2][MAXC] (the CTA's), MAXC = the
// geometry's largest row.  With ln_bwd_blocks_per_sm(MAXC) blocks per SM the
// grid is a single wave.
template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads, ln_bwd_blocks_per_sm(LANES * NV * VEC))
ln_bwd_group(const float* __restrict__ dy, const float* __restrict__ gamma,
             const float* __restrict__ xhat, const float* __restrict__ inv_std,
             float* __restrict__ dx, float* __restrict__ ws, int64_t rows, int cols,
             int64_t rows_per_cta) {
    namespace cg = cooperative_groups;
    constexpr int MAXC = LANES * NV * VEC;
    constexpr int GPB = kBlockThreads / LANES;
    extern __shared__ __align__(16) float smem[];
    float* red = smem;
    float* bpart = smem + GPB * 2 * MAXC;
    // Let the dependent stage-2 kernel be scheduled now; it waits for this
    // grid's completion before reading the workspace.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    const int64_t r_begin = int64_t(blockIdx.x) * rows_per_cta;
    int64_t r_end = r_begin + rows_per_cta;
    if (r_end > rows) r_end = rows;

    float* pg = red + grp * 2 * MAXC;  // this group's dgamma partials
    float* pb = pg + MAXC;             // and dbeta partials (lanes own disjoint columns)
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int col = (g + k * LANES) * VEC + e;
            pg[col] = 0.f;
            pb[col] = 0.f;
        }

    for (int64_t base = r_begin; base < r_end; base += GPB) {  // block-uniform
        const int64_t row = base + grp;
        const bool live = row < r_end;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float a[NV][VEC], h[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                ld_chunk<VEC>(dy + off + c * VEC, a[k]);
                ld_chunk<VEC>(xhat + off + c * VEC, h[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = h[k][e] = 0.f;
            }
        }
        const float r = live ? __ldg(inv_std + row) : 0.f;
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (c < nch) {
                float gm[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int col = c * VEC + e;
                    pg[col] = fmaf(a[k][e], h[k][e], pg[col]);
                    pb[col] += a[k][e];
                    a[k][e] *= gm[e];  // g' = dy * gamma
                    s1 += a[k][e];
                    s2 = fmaf(a[k][e], h[k][e], s2);
                }
            }
        }
        s1 = group_sum<LANES>(s1) * inv_cols;
        s2 = group_sum<LANES>(s2) * inv_cols;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = g + k * LANES;
            if (live && c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = r * (a[k][e] - s1 - h[k][e] * s2);
                st_chunk<VEC>(dx + off + c * VEC, o);
            }
        }
    }
    __syncthreads();
    // Groups -> CTA partial, in group order.
    for (int i = threadIdx.x; i < 2 * MAXC; i += kBlockThreads) {
        float t = red[i];
        for (int q = 1; q < GPB; ++q) t += red[q * 2 * MAXC + i];
        bpart[i] = t;
    }
    // CTAs of the cluster -> cluster partial, rank order.  Rank q adds the
    // entries q*256 + tid (+ 8*256 ...) of all 8 CTAs.
    cg::cluster_group cluster = cg::this_cluster();
    cl_arrive();
    cl_wait();
    const int rank = int(cluster.block_rank());
    const int64_t cl_id = blockIdx.x / kLnClusterCtas;
    for (int i = rank * kBlockThreads + threadIdx.x; i < 2 * cols;
         i += kLnClusterCtas * kBlockThreads) {
        const int half = i >= cols ? 1 : 0;
        const int col = i - half * cols;
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < kLnClusterCtas; ++q)
            t += cluster.map_shared_rank(bpart, q)[half * MAXC + col];
        ws[cl_id * 2 * int64_t(cols) + i] = t;
    }
    cl_arrive();
    cl_wait();  // peers are done with this CTA's bpart
}

// Rows of more than 8192 floats: one 1024-thread CTA per SM walks a fixed
// block of rows in two passes per row (the second reads the row again from
// the L2, where one row per SM stays); each thread owns the same chunks of
// every row, so it adds its columns' partials of dgamma and dbeta without
// atomics, in shared memory when 2 x cols floats fit (SMEM) or else in the
// CTA's workspace slot, which ends up holding the CTA's partials either way.
constexpr int kLnLongThreads = 1024;
constexpr int64_t kLnLongSmemCols = 25600;  // 2 x cols floats in 200 KB

template <int VEC, bool SMEM>
__global__ void __launch_bounds__(kLnLongThreads, 1)
ln_bwd_long(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ xhat,
            const float* __restrict__ inv_std, float* __restrict__ dx, float* __restrict__ ws, int64_t rows,
            int cols, int64_t rows_per_cta) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    extern __shared__ __align__(16) float sp[];
    __shared__ float sc[4 * (kLnLongThreads / 32)];
    BlockReduce<kLnLongThreads> red(sc);
    constexpr int NT = kLnLongThreads;
    constexpr int U = VEC == 4 ? 2 : 8;  // 64 bytes of dy and xhat in flight per thread
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    float* wg = ws + int64_t(blockIdx.x) * 2 * cols;
    float* pg = SMEM ? sp : wg;
    float* pb = pg + cols;
    for (int c = threadIdx.x; c < nch; c += NT) {
        st_zero_chunk<VEC>(pg + c * VEC);
        st_zero_chunk<VEC>(pb + c * VEC);
    }
    const int64_t r_begin = int64_t(blockIdx.x) * rows_per_cta;
    int64_t r_end = r_begin + rows_per_cta;
    if (r_end > rows) r_end = rows;
    for (int64_t row = r_begin; row < r_end; ++row) {  // block-uniform
        const int64_t off = row * int64_t(cols);
        float s1 = 0.f, s2 = 0.f;
        for (int c0 = threadIdx.x; c0 < nch; c0 += U * NT) {
            float a[U][VEC], h[U][VEC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < nch) {
                    ld_chunk<VEC>(dy + off + c * VEC, a[u]);
                    ld_chunk<VEC>(xhat + off + c * VEC, h[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < nch) {
                    float gm[VEC];
                    ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float gp = a[u][e] * gm[e];  // g' = dy * gamma
                        s1 += gp;
                        s2 = fmaf(gp, h[u][e], s2);
                    }
                }
            }
        }
        red.sum2(s1, s2);
        s1 *= inv_cols;
        s2 *= inv_cols;
        const float r = __ldg(inv_std + row);
        for (int c0 = threadIdx.x; c0 < nch; c0 += U * NT) {
            float a[U][VEC], h[U][VEC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < nch) {
                    ld_chunk<VEC>(dy + off + c * VEC, a[u]);
                    ld_chunk<VEC>(xhat + off + c * VEC, h[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < nch) {
                    float gm[VEC], o[VEC], tg[VEC], tb[VEC];
                    ld_chunk<VEC>(gamma + c * VEC, gm);
                    ld_chunk_coherent<VEC>(pg + c * VEC, tg);
                    ld_chunk_coherent<VEC>(pb + c * VEC, tb);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        o[e] = r * (a[u][e] * gm[e] - s1 - h[u][e] * s2);
                        tg[e] = fmaf(a[u][e], h[u][e], tg[e]);
                        tb[e] += a[u][e];
                    }
                    st_chunk<VEC>(dx + off + c * VEC, o);
                    st_chunk<VEC>(pg + c * VEC, tg);
                    st_chunk<VEC>(pb + c * VEC, tb);
                }
            }
        }
    }
    if constexpr (SMEM) {
        for (int c = threadIdx.x; c < nch; c += NT) {
            float tg[VEC], tb[VEC];
            ld_chunk_coherent<VEC>(pg + c * VEC, tg);
            ld_chunk_coherent<VEC>(pb + c * VEC, tb);
            st_chunk<VEC>(wg + c * VEC, tg);
            st_chunk<VEC>(wg + cols + c * VEC, tb);
        }
    }
}

// ------------------------------------------------------ block-row kernels
// Rows of 1025..16384 floats (forward) or 1025..8192 floats (backward), one
// CTA per row in registers (block_rows.cuh); the arithmetic of the group
// kernels with block reductions.

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT)
ln_fwd_brow(const float* __restrict__ x, const float* __restrict__ gamma, const float* __restrict__ beta,
            float* __restrict__ out, float* __restrict__ xhat, float* __restrict__ inv_std, int64_t rows,
            int cols, float eps) {
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t off = row * int64_t(cols);
        const float shift = __ldg(x + off);  // the row's first entry
        float v[NV][VEC];
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(x + off + c * VEC, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s += v[k][e] - shift;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = 0.f;
            }
        }
        const float mean = shift + red.sum(s) * inv_cols;
        float q = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (int(threadIdx.x) + k * NT < nch)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    v[k][e] -= mean;
                    q = fmaf(v[k][e], v[k][e], q);
                }
        const float r = 1.0f / sqrtf(red.sum(q) * inv_cols + eps);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float gm[VEC], bt[VEC], h[VEC], o[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
                ld_chunk<VEC>(beta + c * VEC, bt);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    h[e] = v[k][e] * r;
                    o[e] = fmaf(gm[e], h[e], bt[e]);
                }
                st_chunk<VEC>(xhat + off + c * VEC, h);
                st_chunk<VEC>(out + off + c * VEC, o);
            }
        }
        if (threadIdx.x == 0) inv_std[row] = r;
    }
}

// Backward: the CTA walks a fixed block of rows; each thread keeps the
// column partials of dgamma and dbeta for its own columns in registers and
// writes them to the CTA's workspace slot at the end (stage 2,
// ln_params_reduce, adds the slots in order).  8 floats of the row per thread.
constexpr int64_t kLnBwdBrowMax = 8192;

inline int ln_bwd_brow_threads(int64_t cols) { return cols <= 2048 ? 256 : (cols <= 4096 ? 512 : 1024); }

template <typename F>
bool with_ln_bwd_brow_geometry(bool vec4, int64_t cols, F&& f) {
    if (cols <= 1024 || cols > kLnBwdBrowMax) return false;
    if (vec4) {
        if (cols <= 2048) f(BGeom<256, 2, 4>{});
        else if (cols <= 4096) f(BGeom<512, 2, 4>{});
        else f(BGeom<1024, 2, 4>{});
    } else {
        if (cols <= 2048) f(BGeom<256, 8, 1>{});
        else if (cols <= 4096) f(BGeom<512, 8, 1>{});
        else f(BGeom<1024, 8, 1>{});
    }
    return true;
}

template <int NT, int NV, int VEC>
__global__ void __launch_bounds__(NT, 1024 / NT)
ln_bwd_brow(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ xhat,
            const float* __restrict__ inv_std, float* __restrict__ dx, float* __restrict__ ws, int64_t rows,
            int cols, int64_t rows_per_cta) {
    // Let the dependent stage-2 kernel be scheduled now; it waits for this
    // grid's completion before reading the workspace.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    __shared__ float sc[4 * (NT / 32)];
    BlockReduce<NT> red(sc);
    const int nch = cols / VEC;
    const float inv_cols = 1.0f / float(cols);
    const int64_t r_begin = int64_t(blockIdx.x) * rows_per_cta;
    int64_t r_end = r_begin + rows_per_cta;
    if (r_end > rows) r_end = rows;
    float pg[NV][VEC], pb[NV][VEC];
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) pg[k][e] = pb[k][e] = 0.f;
    for (int64_t row = r_begin; row < r_end; ++row) {  // block-uniform
        const int64_t off = row * int64_t(cols);
        float a[NV][VEC], h[NV][VEC];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                ld_chunk<VEC>(dy + off + c * VEC, a[k]);
                ld_chunk<VEC>(xhat + off + c * VEC, h[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) a[k][e] = h[k][e] = 0.f;
            }
        }
        const float r = __ldg(inv_std + row);
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float gm[VEC];
                ld_chunk<VEC>(gamma + c * VEC, gm);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    pg[k][e] = fmaf(a[k][e], h[k][e], pg[k][e]);
                    pb[k][e] += a[k][e];
                    a[k][e] *= gm[e];  // g' = dy * gamma
                    s1 += a[k][e];
                    s2 = fmaf(a[k][e], h[k][e], s2);
                }
            }
        }
        red.sum2(s1, s2);
        s1 *= inv_cols;
        s2 *= inv_cols;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = int(threadIdx.x) + k * NT;
            if (c < nch) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = r * (a[k][e] - s1 - h[k][e] * s2);
                st_chunk<VEC>(dx + off + c * VEC, o);
            }
        }
    }
    float* wg = ws + int64_t(blockIdx.x) * 2 * cols;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = int(threadIdx.x) + k * NT;
        if (c < nch) {
            st_chunk<VEC>(wg + c * VEC, pg[k]);
            st_chunk<VEC>(wg + cols + c * VEC, pb[k]);
        }
    }
}

// Backward stage 1 with column owners (rows of 384..1024 floats on 16-byte
// boundaries whose CTA block fits in shared memory whole).  A CTA of up to
// 768 threads owns a contiguous block of rows, split into `sets` row sets of
// tp threads (tp = cols/4 rounded up to whole warps): thread (h, t) owns the
// float4 column chunk t of rows h, h + sets, ... of the block.  At the start
// every thread issues cp.async copies of exactly those chunks of dy and xhat
// (the whole block is requested at once, by all threads in parallel), in
// kLnColsPhases commit groups, and later reads only its own data, so it
// waits for its own copies and no other thread's.  Per phase:
//   pass A  adds the thread's dgamma/dbeta partials for its columns in
//           registers and reduces each row's sums of g' and g'*xhat over the
//           warp, one value per warp into shared memory (with two or more
//           rows a thread, one reduce-scatter of all the rows' sums,
//           ln_cols_pass_a: 6, 9 or 16 shuffles for 2, up to 4 or up to 8
//           rows, where per-row butterflies take 10 a row);
//   barrier of the set's warps only (a named barrier per set: the sets share
//           no rows, so one set's late copies do not hold up another's);
//   pass B  adds the warps' values of each row in warp order (once per row,
//           by the set's first warp behind a second set barrier, when the
//           phase gives a thread two or more rows) and writes dx; the writes
//           of a phase overlap the loads of the next.
// The column partials need no reduction across warps (each column chunk has
// one owner per set): the sets add theirs in set order (handed to set 0 as
// soon as their last pass A is done, where shared memory has room for them
// beside the rows) and the CTA writes one workspace slot; ln_params_reduce
// adds the slots in order.  (A single launch that finishes the column sums
// itself needs a rendezvous of all CTAs, which measured slower on GB300 than
// this programmatic-dependent second kernel.)
constexpr int kLnColsThreads = 768;
// Commit groups per thread (on GB300 at 4096 x 768, back to back: one 13.0 us,
// two 12.7, three 13.4; with the per-set barriers two 12.5-12.8, three 13.7,
// four 14.2).
constexpr int kLnColsPhases = 2;

// Barrier of one row set's tp threads (named barrier 1 + h; sets <= 8).
__device__ __forceinline__ void set_barrier(int h, int tp) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(1 + h), "r"(tp) : "memory");
}

// Named barrier on which sets 1.. hand their column partials to set 0: they
// arrive (without waiting) once their last pass A is done, set 0 waits, and
// adds them while the other sets still write dx (on GB300, back to back:
// 153 x 768 5.6 -> 5.5 us, 4096 x 384 9.0 -> 8.9; 4096 x 768 unchanged).
constexpr int kLnPartsBarrier = 15;
__device__ __forceinline__ void parts_arrive(int threads) {
    asm volatile("bar.arrive %0, %1;\n" ::"r"(kLnPartsBarrier), "r"(threads) : "memory");
}
__device__ __forceinline__ void parts_wait(int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(kLnPartsBarrier), "r"(threads) : "memory");
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Waits until at most n of this thread's commit groups are pending (n <= 3).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;\n" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;\n" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;\n" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 3;\n" ::: "memory"); break;
    }
}

// Pass A of ln_bwd_cols over 2..NR rows k0..k1-1 of this thread: the dgamma /
// dbeta partials of its columns, and the rows' 2*NR sums of g' and g'*xhat
// reduce-scattered over the warp.  Each round halves the values a lane holds
// (rounds at lane distances 16, 8, ... while values remain, then a butterfly
// over the rest), so every sum meets the same addition tree as a butterfly of
// its own at distances 16, 8, 4, 2, 1, bit for bit, in 2*NR - 1 + 4 - log2(NR)
// shuffles (6, 9, 16 for NR = 2, 4, 8) instead of 10 a row.  Lanes 32/(2*NR)*m .. hold value m (row m / 2,
// sum m % 2); the first of them stores it as the warp's value for the row.
template <int NR>
__device__ __forceinline__ void ln_cols_pass_a(const float4* sdy, const float4* sxh, float* red, float4 g,
                                               float4& pg, float4& pb, int h, int t, int tp, int sets, int wps,
                                               int wi, int lane, bool own, int k0, int k1) {
    float v[2 * NR];
#pragma unroll
    for (int i = 0; i < 2 * NR; ++i) v[i] = 0.f;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int k = k0 + i;
        if (own && k < k1) {
            const int j = h + k * sets;
            const float4 a = sdy[size_t(j) * tp + t], x = sxh[size_t(j) * tp + t];
            pg.x = fmaf(a.x, x.x, pg.x);
            pg.y = fmaf(a.y, x.y, pg.y);
            pg.z = fmaf(a.z, x.z, pg.z);
            pg.w = fmaf(a.w, x.w, pg.w);
            pb.x += a.x;
            pb.y += a.y;
            pb.z += a.z;
            pb.w += a.w;
            const float gx = a.x * g.x, gy = a.y * g.y, gz = a.z * g.z, gw = a.w * g.w;
            float s2 = 0.f;
            s2 = fmaf(gx, x.x, s2);
            s2 = fmaf(gy, x.y, s2);
            s2 = fmaf(gz, x.z, s2);
            s2 = fmaf(gw, x.w, s2);
            v[2 * i] = (gx + gy) + (gz + gw);
            v[2 * i + 1] = s2;
        }
    }
    int o = 16;
#pragma unroll
    for (int half = NR; half >= 1; half >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFullMask, send, o);
        }
    }
#pragma unroll
    for (; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(kFullMask, v[0], o);
    constexpr int kSpan = 32 / (2 * NR);  // lanes holding each value
    const int m = (lane / kSpan) & (2 * NR - 1);
    if (lane % kSpan == 0 && (m >> 1) < k1 - k0)
        red[(size_t(h + (k0 + (m >> 1)) * sets) * wps + wi) * 2 + (m & 1)] = v[0];
}

__global__ void __launch_bounds__(kLnColsThreads, 1)
ln_bwd_cols(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ xhat,
            const float* __restrict__ inv_std, float* __restrict__ dx, float* __restrict__ ws, int64_t rows,
            int cols, int64_t rows_per_cta, int sets, int tp, bool early) {
    // Let the dependent stage-2 kernel be scheduled now; it waits for this
    // grid's completion before reading the workspace.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    constexpr int P = kLnColsPhases;
    extern __shared__ __align__(16) float sm[];
    const int nc = cols >> 2;
    const int wps = tp >> 5;  // warps per set
    const int64_t r_begin = int64_t(blockIdx.x) * rows_per_cta;
    const int64_t r_end = r_begin + rows_per_cta < rows ? r_begin + rows_per_cta : rows;
    const int n_rows = r_end > r_begin ? int(r_end - r_begin) : 0;
    float4* sdy = reinterpret_cast<float4*>(sm);                              // [rows_per_cta][tp]
    float4* sxh = sdy + size_t(rows_per_cta) * tp;                             // [rows_per_cta][tp]
    float* red = reinterpret_cast<float*>(sxh + size_t(rows_per_cta) * tp);   // [rows_per_cta][wps][2]
    float* inv_s = red + size_t(rows_per_cta) * wps * 2;                       // [rows_per_cta]
    // with `early`, the sets' column partials get a region of their own
    float4* parts = reinterpret_cast<float4*>(                                  // [sets][2][tp]
        (reinterpret_cast<uintptr_t>(inv_s + rows_per_cta) + 15) & ~uintptr_t(15));
    const int h = int(threadIdx.x) / tp;
    const int t = int(threadIdx.x) % tp;
    const int lane = threadIdx.x & 31;
    const int wi = t >> 5;
    const bool own = t < nc;
    const int K = n_rows > h ? (n_rows - h + sets - 1) / sets : 0;  // rows of this thread's set
#pragma unroll
    for (int p = 0; p < P; ++p) {
        if (own)
            for (int k = p * K / P; k < (p + 1) * K / P; ++k) {
                const int j = h + k * sets;
                cp_async16(sdy + size_t(j) * tp + t, dy + (r_begin + j) * cols + 4 * t);
                cp_async16(sxh + size_t(j) * tp + t, xhat + (r_begin + j) * cols + 4 * t);
            }
        cp_async_commit();
    }
    for (int k = t; k < K; k += tp) inv_s[h + k * sets] = __ldg(inv_std + r_begin + h + k * sets);  // own set's rows
    const float4 g = own ? __ldg(reinterpret_cast<const float4*>(gamma) + t) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float inv_cols = 1.0f / float(cols);
    float4 pg = make_float4(0.f, 0.f, 0.f, 0.f), pb = pg;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        cp_async_wait_pending(P - 1 - p);  // this phase's rows have landed
        const int k0 = p * K / P, k1 = (p + 1) * K / P;
        if (k1 - k0 >= 2) {  // warp-uniform (a warp lies in one set)
            if (k1 - k0 == 2)
                ln_cols_pass_a<2>(sdy, sxh, red, g, pg, pb, h, t, tp, sets, wps, wi, lane, own, k0, k1);
            else if (k1 - k0 <= 4)
                ln_cols_pass_a<4>(sdy, sxh, red, g, pg, pb, h, t, tp, sets, wps, wi, lane, own, k0, k1);
            else
                ln_cols_pass_a<8>(sdy, sxh, red, g, pg, pb, h, t, tp, sets, wps, wi, lane, own, k0, k1);
        } else {  // one row or none: a butterfly per sum
            for (int k = k0; k < k1; ++k) {  // pass A
                const int j = h + k * sets;
                float s1 = 0.f, s2 = 0.f;
                if (own) {
                    const float4 a = sdy[size_t(j) * tp + t], x = sxh[size_t(j) * tp + t];
                    pg.x = fmaf(a.x, x.x, pg.x);
                    pg.y = fmaf(a.y, x.y, pg.y);
                    pg.z = fmaf(a.z, x.z, pg.z);
                    pg.w = fmaf(a.w, x.w, pg.w);
                    pb.x += a.x;
                    pb.y += a.y;
                    pb.z += a.z;
                    pb.w += a.w;
                    const float gx = a.x * g.x, gy = a.y * g.y, gz = a.z * g.z, gw = a.w * g.w;
                    s1 = (gx + gy) + (gz + gw);
                    s2 = fmaf(gx, x.x, s2);
                    s2 = fmaf(gy, x.y, s2);
                    s2 = fmaf(gz, x.z, s2);
                    s2 = fmaf(gw, x.w, s2);
                }
    #pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    s1 += __shfl_xor_sync(kFullMask, s1, o);
                    s2 += __shfl_xor_sync(kFullMask, s2, o);
                }
                if (lane == 0) {
                    red[(size_t(j) * wps + wi) * 2] = s1;
                    red[(size_t(j) * wps + wi) * 2 + 1] = s2;
                }
            }
        }
        if (early && p == P - 1 && h != 0) {  // this thread's column partials are final
            parts[(size_t(h) * 2) * tp + t] = pg;
            parts[(size_t(h) * 2 + 1) * tp + t] = pb;
            parts_arrive(int(blockDim.x));
        }
        set_barrier(h, tp);  // the set's warps' row sums (and, the first time, inv_std) are in shared memory
        // With two or more rows a thread in the phase (the same for the whole
        // set), the set's first warp adds the warps' sums of each row (lane
        // l: row k0 + l) in warp order into the row's first slot, once,
        // instead of every owner adding them (4096 x 768 on GB300, back to
        // back: 12.9 -> 12.3 us); with one row the extra barrier costs more.
        const bool once = k1 - k0 >= 2;
        if (once) {
            if (wi == 0 && lane < k1 - k0) {
                const int j = h + (k0 + lane) * sets;
                float s1 = 0.f, s2 = 0.f;
                for (int w = 0; w < wps; ++w) {
                    s1 += red[(size_t(j) * wps + w) * 2];
                    s2 += red[(size_t(j) * wps + w) * 2 + 1];
                }
                red[size_t(j) * wps * 2] = s1 * inv_cols;
                red[size_t(j) * wps * 2 + 1] = s2 * inv_cols;
            }
            set_barrier(h, tp);
        }
        for (int k = k0; k < k1; ++k) {  // pass B
            const int j = h + k * sets;
            float s1, s2;
            if (once) {
                const float2 u = reinterpret_cast<const float2*>(red)[size_t(j) * wps];
                s1 = u.x;
                s2 = u.y;
            } else {
                s1 = 0.f;
                s2 = 0.f;
                for (int w = 0; w < wps; ++w) {
                    s1 += red[(size_t(j) * wps + w) * 2];
                    s2 += red[(size_t(j) * wps + w) * 2 + 1];
                }
                s1 *= inv_cols;
                s2 *= inv_cols;
            }
            if (own) {
                const float r = inv_s[j];
                const float4 a = sdy[size_t(j) * tp + t], x = sxh[size_t(j) * tp + t];
                float4 o;
                o.x = r * (a.x * g.x - s1 - x.x * s2);
                o.y = r * (a.y * g.y - s1 - x.y * s2);
                o.z = r * (a.z * g.z - s1 - x.z * s2);
                o.w = r * (a.w * g.w - s1 - x.w * s2);
                reinterpret_cast<float4*>(dx + (r_begin + j) * cols)[t] = o;
            }
        }
    }
    float4* cr = parts;
    if (early) {
        if (h != 0) return;
        parts_wait(int(blockDim.x));  // every other set has stored its partials
    } else {
        __syncthreads();  // the staged rows are no longer read: the space holds the sets' partials
        cr = sdy;         // [sets][2][tp]
        cr[(size_t(h) * 2) * tp + t] = pg;
        cr[(size_t(h) * 2 + 1) * tp + t] = pb;
        __syncthreads();
    }
    if (h == 0 && own) {
        for (int q = 1; q < sets; ++q) {
            const float4 u = cr[(size_t(q) * 2) * tp + t], v = cr[(size_t(q) * 2 + 1) * tp + t];
            pg.x += u.x;
            pg.y += u.y;
            pg.z += u.z;
            pg.w += u.w;
            pb.x += v.x;
            pb.y += v.y;
            pb.z += v.z;
            pb.w += v.w;
        }
        float4* slot = reinterpret_cast<float4*>(ws + int64_t(blockIdx.x) * 2 * cols);
        slot[t] = pg;
        slot[nc + t] = pb;
    }
}

// Launch shape of ln_bwd_cols with at most max_ctas CTAs (0: one per SM):
// grid, rows per CTA, row sets, threads per set and dynamic shared memory;
// grid = 0 when the shape is not taken (the block does not fit).
struct LnColsPlan {
    int64_t grid = 0, per_cta = 0;
    int sets = 0, tp = 0;
    bool early = false;  // column partials handed over in their own region (see ln_bwd_cols)
    size_t smem = 0;
};

LnColsPlan ln_cols_plan(int64_t rows, int64_t cols, int64_t max_ctas) {
    LnColsPlan pl;
    if (cols < 384 || cols > 1024 || cols % 4 != 0 || rows <= 0) return pl;
    const int sms = sm_count();
    if (sms <= 0) return pl;
    int64_t g = rows < sms ? rows : sms;
    if (max_ctas > 0 && g > max_ctas) g = max_ctas;
    if (g <= 0) return pl;
    const int64_t per_cta = (rows + g - 1) / g;
    g = (rows + per_cta - 1) / per_cta;
    const int tp = int((cols / 4 + 31) / 32 * 32);
    const int sets = kLnColsThreads / tp;
    const int64_t per_set = (per_cta + sets - 1) / sets;
    if ((per_set + kLnColsPhases - 1) / kLnColsPhases > 8) return pl;  // pass A holds 8 rows
    const size_t rows_bytes = size_t(per_cta) * (size_t(2) * tp * 16 + size_t(tp / 32) * 2 * 4 + 4);
    const size_t parts_bytes = size_t(sets) * 2 * tp * 16;  // the sets' column partials at the end
    // the partials in a region of their own when it fits, else in the rows' space at the end
    const size_t smem_early = (rows_bytes + 15) / 16 * 16 + parts_bytes;
    const bool early = smem_early <= 226 * 1024;
    const size_t smem = early ? smem_early : (rows_bytes > parts_bytes ? rows_bytes : parts_bytes);
    if (smem > 226 * 1024) return pl;
    pl.grid = g;
    pl.per_cta = per_cta;
    pl.sets = sets;
    pl.tp = tp;
    pl.smem = smem;
    pl.early = early;
    return pl;
}

// Stage 2: out[i] = sum_p ws[p][i] for i in [0, 2*cols).  A block covers 32
// outputs with 8 warps: warp j adds partials j, j+8, j+16, ... in order (loads
// coalesced across the 32 outputs), then thread i adds the 8 warp sums in warp
// order; the association is fixed, so results are deterministic.  Launched as a
// programmatic dependent of stage 1: it waits here for stage 1's writes.
__global__ void __launch_bounds__(kBlockThreads)
ln_params_reduce(const float* ws, int64_t partials, int64_t cols,
                 float* __restrict__ dgamma, float* __restrict__ dbeta) {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    __shared__ float part[kBlockThreads / 32][32];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t i = int64_t(blockIdx.x) * 32 + lane;
    const int64_t stride = 2 * cols;
    float t = 0.f;
    if (i < stride) {
        // Batches of B loads in flight (one L2 round trip per batch for up to
        // 8 * B partials), added in partial order; a missing partial adds +0.
        constexpr int B = 24;
        for (int64_t p0 = w; p0 < partials; p0 += 8 * B) {
            float v[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int64_t p = p0 + 8 * b;
                v[b] = p < partials ? ws[p * stride + i] : 0.f;
            }
#pragma unroll
            for (int b = 0; b < B; ++b) t += v[b];
        }
    }
    part[w][lane] = t;
    __syncthreads();
    if (w == 0 && i < stride) {
        float r = part[0][lane];
#pragma unroll
        for (int q = 1; q < kBlockThreads / 32; ++q) r += part[q][lane];
        if (i < cols)
            dgamma[i] = r;
        else
            dbeta[i - cols] = r;
    }
}

}  // namespace

// ------------------------------------------------------------ launchers

cudaError_t launch_layernorm_fwd(const float* x, const float* gamma, const float* beta,
                                 float* out, float* xhat, float* inv_std, int64_t rows,
                                 int64_t cols, float eps, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        const BalancedLaunch bl = balanced_groups(rows, G::LANES);
        if (bl.threads)
            ln_fwd_group<G::LANES, G::NV, G::VEC><<<bl.grid, bl.threads, 0, stream>>>(
                x, gamma, beta, out, xhat, inv_std, rows, int(cols), eps);
        else
            ln_fwd_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
                x, gamma, beta, out, xhat, inv_std, rows, int(cols), eps);
    });
    if (!done) {
        if (with_block_geometry(vec4, cols, kBlockRowMax, [&](auto geo) {
                using G = decltype(geo);
                ln_fwd_brow<G::NT, G::NV, G::VEC><<<block_row_grid(rows), G::NT, 0, stream>>>(
                    x, gamma, beta, out, xhat, inv_std, rows, int(cols), eps);
            })) {
        } else if (vec4)
            ln_fwd_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, gamma, beta, out, xhat,
                                                                             inv_std, rows, cols, eps);
        else
            ln_fwd_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, gamma, beta, out, xhat,
                                                                             inv_std, rows, cols, eps);
    }
    note_launches(1);
    return cudaGetLastError();
}

// Column partials of the two-kernel backward: one per cluster of the group
// kernel (rows of up to 1024 floats that the fused kernel does not take),
// one per resident CTA of the block-row kernel (1024 threads per SM), one per
// CTA of the long-row kernel.
int64_t ln_bwd_slots(int64_t rows, int64_t cols) {
    if (cols > 1024) {
        const int sms = sm_count();
        const int64_t per_sm = cols <= kLnBwdBrowMax ? 1024 / ln_bwd_brow_threads(cols) : 1;
        const int64_t p = int64_t(sms > 0 ? sms : 1) * per_sm;
        return rows < p ? rows : p;
    }
    return ln_bwd_partials(rows, cols);
}

// Stage-1 partials for rows of up to 1024 floats: the larger of the lane-group
// kernel's cluster count and the column-owner / ring kernels' CTA count, so
// the size does not depend on alignment.  With a byte budget the CTA count is
// capped to fit it.
int64_t ln_bwd_cap(int64_t cols, size_t budget) {
    return budget ? int64_t(budget / (size_t(8) * size_t(cols))) : 0;
}

size_t layernorm_bwd_workspace(int64_t rows, int64_t cols, size_t budget) {
    if (rows <= 0 || cols <= 0) return 0;
    int64_t slots = ln_bwd_slots(rows, cols);
    if (cols <= 1024) {
        // the column-owner kernel runs up to one CTA per SM; the ring kernel
        // no more than that
        const int sms = sm_count();
        int64_t c = rows < sms ? rows : int64_t(sms);
        const int64_t cap = ln_bwd_cap(cols, budget);
        if (cap > 0 && c > cap) c = cap;
        if (c > slots) slots = c;
    }
    return size_t(slots) * 2 * size_t(cols) * sizeof(float);
}

cudaError_t launch_layernorm_bwd(const float* dy, const float* gamma, const float* xhat,
                                 const float* inv_std, float* dx, float* dgamma, float* dbeta,
                                 int64_t rows, int64_t cols, float* ws, bool vec4,
                                 cudaStream_t stream, size_t budget) {
    cudaError_t err = cudaSuccess;
    int64_t partials = ln_bwd_slots(rows, cols);
    bool done = false;
    const int64_t cap = ln_bwd_cap(cols, budget);
    if (vec4) {
        const LnColsPlan pl = ln_cols_plan(rows, cols, cap);
        if (pl.grid > 0) {
            err = cudaFuncSetAttribute(ln_bwd_cols, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
            if (err != cudaSuccess) return err;
            ln_bwd_cols<<<unsigned(pl.grid), pl.sets * pl.tp, pl.smem, stream>>>(
                dy, gamma, xhat, inv_std, dx, ws, rows, int(cols), pl.per_cta, pl.sets, pl.tp, pl.early);
            partials = pl.grid;
            done = true;
        } else if (launch_ln_bwd_tma(dy, gamma, xhat, inv_std, dx, ws, rows, cols, cap, stream, &err)) {
            partials = ln_bwd_tma_ctas(rows, cols, cap);
            done = true;
        }
    }
    if (!done) done = with_ln_bwd_brow_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        const int64_t per_cta = (rows + partials - 1) / partials;
        ln_bwd_brow<G::NT, G::NV, G::VEC><<<unsigned(partials), G::NT, 0, stream>>>(
            dy, gamma, xhat, inv_std, dx, ws, rows, int(cols), per_cta);
    });
    if (!done) done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        constexpr int MAXC = G::LANES * G::NV * G::VEC;
        constexpr int GPB = kBlockThreads / G::LANES;
        const size_t smem = size_t(GPB + 1) * 2 * MAXC * sizeof(float);
        auto kern = ln_bwd_group<G::LANES, G::NV, G::VEC>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return;
        partials = ln_bwd_partials(rows, cols);
        const int64_t ctas = partials * kLnClusterCtas;
        const int64_t per_cta = (rows + ctas - 1) / ctas;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(ctas));
        cfg.blockDim = dim3(kBlockThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kLnClusterCtas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, kern, dy, gamma, xhat, inv_std, dx, ws, rows, int(cols),
                                 per_cta);
    });
    if (!done) {
        const int64_t per_cta = (rows + partials - 1) / partials;
        const bool in_smem = cols <= kLnLongSmemCols;
        const size_t smem = in_smem ? size_t(2) * size_t(cols) * sizeof(float) : 0;
        auto launch = [&](auto kern) {
            if (smem > 0) {
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
                if (err != cudaSuccess) return;
            }
            kern<<<unsigned(partials), kLnLongThreads, smem, stream>>>(dy, gamma, xhat, inv_std, dx, ws, rows,
                                                                       int(cols), per_cta);
        };
        if (vec4) {
            if (in_smem) launch(ln_bwd_long<4, true>);
            else launch(ln_bwd_long<4, false>);
        } else {
            if (in_smem) launch(ln_bwd_long<1, true>);
            else launch(ln_bwd_long<1, false>);
        }
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int64_t nb = (2 * cols + 31) / 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(nb));
    cfg.blockDim = dim3(kBlockThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, ln_params_reduce, static_cast<const float*>(ws), partials, cols,
                             dgamma, dbeta);
    note_launches(2);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace rowops

// ------------------------------------------------ allocation-free variant
// LayerNorm backward for callers that cannot hand the library a workspace
// (see rowops_layernorm_bwd_noalloc in include/rowops.h).  Its workspace is a
// fixed array in device memory that the library owns for the life of the
// process on every GPU that loads it.

#include <mutex>

#include "rowops.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_ln_bwd_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
float* g_scratch_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device.  Host code only
// holds a host-side stand-in under the array's name, so the real address is
// asked for once per device, with that device current.
int scratch_for_current_device(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
        return ROWOPS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ln_bwd_scratch) != cudaSuccess || p == nullptr)
            return ROWOPS_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return ROWOPS_OK;
}

}  // namespace

extern "C" size_t rowops_layernorm_bwd_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int rowops_layernorm_bwd_noalloc(const float* dy, const float* gamma, const float* xhat,
                                            const float* inv_std, float* dx, float* dgamma,
                                            float* dbeta, int64_t rows, int64_t cols,
                                            rowops_stream stream) {
    // The argument rules of rowops_layernorm_bwd, in its order; then the size
    // check against the array; the array's address is looked up last.
    bool vec4 = false;
    if (int e = rowops::layernorm_bwd_checks(dy, gamma, xhat, inv_std, dx, dgamma, dbeta, rows, cols, &vec4))
        return e;
    if (rows == 0) return ROWOPS_OK;
    if (rowops::layernorm_bwd_workspace(rows, cols, kNoAllocScratchBytes) > kNoAllocScratchBytes)
        return ROWOPS_ERR_WORKSPACE;
    float* ws = nullptr;
    if (int e = scratch_for_current_device(&ws)) return e;
    const cudaError_t err = rowops::launch_layernorm_bwd(dy, gamma, xhat, inv_std, dx, dgamma, dbeta, rows, cols,
                                                         ws, vec4, reinterpret_cast<cudaStream_t>(stream),
                                                         kNoAllocScratchBytes);
    return err == cudaSuccess ? ROWOPS_OK : ROWOPS_ERR_CUDA;
}
