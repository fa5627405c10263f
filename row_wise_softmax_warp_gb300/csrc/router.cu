// router.cu - the fused MoE router (hard-masked softmax and the top-k kept
// mask of its output in one pass) and pulsatrix top_k_rows (the k largest or
// smallest values of each row in rank order, with their columns).
//
// router_group: a lane group holds a row (geometry of common.cuh), computes
// P = masked softmax exactly as masked_group does, stores it, and runs the
// kept-mask selection (kept_core.cuh) on the same fp32 registers, so the mask
// equals rowops_topk_kept applied to the stored P, bit for bit, while P is
// never read back from HBM (13 bytes per element instead of 9 + 8).
//
// top_k_rows: the order is a strict total order on (key, column) with key the
// order-preserving uint32 of the value, NaN mapped above +inf and -0 onto +0.
// k <= 2 takes a tournament of each lane's (or, on rows of more than 1024
// floats, each thread's) entries and butterfly merges of the best pairs; on
// rows of up to 1024 floats larger k takes candidates or k rounds that each
// pick the best remaining key (max for largest, min for smallest) and the
// lowest column holding it; longer rows with larger k the select kernel.
#include "common.cuh"
#include "kept_core.cuh"
#include "launch.h"


namespace rowops {
namespace {

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
router_group(const float* x, const uint8_t* __restrict__ mask, float* p, float* __restrict__ kept,
             int64_t rows, int cols, int k) {
    constexpr int GPB = kBlockThreads / LANES;
    __shared__ KeptScratch kscratch[kBlockThreads / 32];  // the candidate path's, one per warp
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int nch = cols / VEC;
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += int64_t(gridDim.x) * GPB) {
        const int64_t row = base + grp;
        const bool live = row < rows;
        const int64_t off = (live ? row : 0) * int64_t(cols);
        float v[NV][VEC];
        bool al[NV][VEC], valid[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk) {
            const int c = g + kk * LANES;
            if (live && c < nch) {
                ld_chunk_coherent<VEC>(x + off + c * VEC, v[kk]);  // p may be x
                ld_mask<VEC>(mask + off + c * VEC, al[kk]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) al[kk][e] = false;
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) valid[kk][e] = live && c < nch;
        }
        // Hard-masked softmax (the arithmetic of masked_group).
        float m = -INFINITY;
        int n_allowed = 0;
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (al[kk][e]) {
                    m = fmaxf(m, v[kk][e]);
                    ++n_allowed;
                }
        m = group_max<LANES>(m);
        n_allowed = group_sum_int<LANES>(n_allowed);
        float s = 0.f;
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[kk][e] = al[kk][e] ? exp_shifted(v[kk][e], m) : 0.f;
                s += v[kk][e];
            }
        s = group_sum<LANES>(s);
        const float inv = n_allowed > 0 ? 1.0f / s : 0.f;
        float probe = 0.f;  // probabilities sum to at most 1; NaN makes the sum NaN
#pragma unroll
        for (int kk = 0; kk < NV; ++kk) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[kk][e] = al[kk][e] ? v[kk][e] * inv : 0.f;  // the stored probabilities
                probe += v[kk][e];
            }
            const int c = g + kk * LANES;
            if (live && c < nch) st_chunk<VEC>(p + off + c * VEC, v[kk]);
        }
        // Top-k kept mask of those probabilities.
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

// ------------------------------------------------------------ top_k_rows

__device__ __forceinline__ uint32_t rank_key(float x) {
    return isnan(x) ? 0xffffffffu : ordered_key(x);
}

template <int LANES>
__device__ __forceinline__ uint32_t group_max_u32(uint32_t v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

template <int LANES>
__device__ __forceinline__ uint32_t group_min_u32(uint32_t v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

// top_k_rows for 3 <= k <= LANES (groups of 8 or more lanes): the entries
// whose selection key (rank key, complemented for smallest-first) reaches tau,
// the k-th largest of the group's lane maxima, include the top k (each lane's
// maximum is an entry of the row, so at least k reach it, and every entry
// ranked above one that reaches it reaches it too).  When every row of the
// warp has at most 32 such candidates they are ranked among themselves by
// counting (larger key first, then lower column) and the first k written;
// otherwise nothing is touched and false is returned (warp-uniform).
template <int LANES, int NV, int VEC>
__device__ __forceinline__ bool topk_by_candidates(const uint32_t (&sel)[NV][VEC], const bool (&avail)[NV][VEC],
                                                   const float (&v)[NV][VEC], int k, bool live, float* vr,
                                                   float* ir, KeptScratch* ks) {
    const int g = threadIdx.x % LANES;
    const int leader = (threadIdx.x & 31) - g;
    const int gi = (threadIdx.x & 31) / LANES;
    uint32_t lm = 0u;  // a lane without entries counts as key 0, which every key reaches
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (avail[kk][e]) lm = max(lm, sel[kk][e]);
    uint32_t s = lm;  // the group's lane maxima in descending order
#pragma unroll
    for (int kk = 2; kk <= LANES; kk <<= 1)
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(kFullMask, s, j);
            const bool lower = (g & j) == 0;
            const bool desc = (g & kk) == 0;
            s = (lower == desc) ? max(s, o) : min(s, o);
        }
    const uint32_t tau = __shfl_sync(kFullMask, s, leader + k - 1);
    int cnt = 0;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e) cnt += (avail[kk][e] && sel[kk][e] >= tau) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, o, LANES);
        if (g >= o) incl += y;
    }
    const int total = __shfl_sync(kFullMask, incl, leader + LANES - 1);
    if (__any_sync(kFullMask, total > 32)) return false;
    unsigned* sk = ks->bits[gi];
    int* sc = ks->c[gi];
    float* sv = ks->v[gi];
    __syncwarp();  // the warp's previous use of the scratch is over
    int slot = incl - cnt;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (avail[kk][e] && sel[kk][e] >= tau) {
                sk[slot] = sel[kk][e];
                sc[slot] = (g + kk * LANES) * VEC + e;
                sv[slot] = v[kk][e];
                ++slot;
            }
    __syncwarp();
    for (int i = g; i < total; i += LANES) {
        const uint32_t ki = sk[i];
        const int ci = sc[i];
        int rank = 0;
        for (int q = 0; q < total; ++q) rank += (sk[q] > ki || (sk[q] == ki && sc[q] < ci)) ? 1 : 0;
        if (live && rank < k) {
            vr[rank] = sv[i];
            ir[rank] = float(ci);
        }
    }
    return true;
}

template <int LANES, int NV, int VEC>
__global__ void __launch_bounds__(kBlockThreads)
top_k_rows_group(const float* __restrict__ x, float* __restrict__ values, float* __restrict__ indices,
                 int64_t rows, int cols, int k, int largest) {
    constexpr int GPB = kBlockThreads / LANES;
    __shared__ KeptScratch kscratch[kBlockThreads / 32];  // the candidate path's, one per warp
    const int g = threadIdx.x % LANES;
    const int grp = threadIdx.x / LANES;
    const int leader = (threadIdx.x & 31) - g;
    const int nch = cols / VEC;
    const int64_t stride = int64_t(gridDim.x) * GPB;
    float nv[NV][VEC];
    kept_load_row<LANES, NV, VEC>(x, int64_t(blockIdx.x) * GPB + grp, rows, cols, nv);
    for (int64_t base = int64_t(blockIdx.x) * GPB; base < rows; base += stride) {  // block-uniform
        float v[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[kk][e] = nv[kk][e];
        if (base + stride < rows) kept_load_row<LANES, NV, VEC>(x, base + stride + grp, rows, cols, nv);
        const int64_t row = base + grp;
        const bool live = row < rows;
        uint32_t key[NV][VEC];
        bool avail[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk) {
            const int c = g + kk * LANES;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                key[kk][e] = rank_key(v[kk][e]);
                avail[kk][e] = live && c < nch;
            }
        }
        if (k <= 2) {
            // Without NaN or infinities in the warp's rows (a finite sum), the
            // key order is the float order (-0 == +0) and the tournament runs
            // on the values themselves, negated for smallest-first; the
            // winners' values come back by negating again, bit for bit.
            float probe = 0.f;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) probe += v[kk][e];
            if (!__any_sync(kFullMask, !(fabsf(probe) <= 3.402823466e38f))) {  // warp-uniform
                const float sgn = largest ? 1.f : -1.f;
                constexpr int E = NV * VEC;
                float xs[E];
                int cs[E];
#pragma unroll
                for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) cs[kk * VEC + e] = (g + kk * LANES) * VEC + e;
                kept_detail::Top2<float> t;
                if (cols == LANES * E) {  // every entry in the row (warp-uniform; rows past the last are not stored)
#pragma unroll
                    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) xs[kk * VEC + e] = sgn * v[kk][e];
                    t = kept_detail::group_top2<LANES, E, float>(xs, cs, -INFINITY);
                } else {
#pragma unroll
                    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) xs[kk * VEC + e] = avail[kk][e] ? sgn * v[kk][e] : -INFINITY;
                    t = kept_detail::group_top2<LANES, E, float>(xs, cs, -INFINITY);
                }
                if (live && g == 0) {
                    values[row * int64_t(k)] = sgn * t.v1;
                    indices[row * int64_t(k)] = float(t.c1);
                    if (k == 2) {
                        values[row * int64_t(k) + 1] = sgn * t.v2;
                        indices[row * int64_t(k) + 1] = float(t.c2);
                    }
                }
                continue;
            }
            // The group's best two (key, column) pairs in the order "larger
            // key first, then lower column" (keys complemented for
            // smallest-first): a tournament over each lane's entries in column
            // order, then a butterfly (kept_core.cuh).  An entry outside the
            // row counts as key 0 at its own column, above every column of
            // the row, so it loses every tie and, as k <= cols, is not picked.
            const uint32_t flip = largest ? 0u : 0xffffffffu;
            constexpr int E = NV * VEC;
            uint32_t ks[E];
            int cs[E];
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    ks[kk * VEC + e] = avail[kk][e] ? key[kk][e] ^ flip : 0u;
                    cs[kk * VEC + e] = (g + kk * LANES) * VEC + e;
                }
            const kept_detail::Top2<uint32_t> t = kept_detail::group_top2<LANES, E, uint32_t>(ks, cs, 0u);
            const int i1 = t.c1, i2 = t.c2;
            // The lanes holding the two columns pass their values to the group.
            float v1 = 0.f, v2 = 0.f;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int c = (g + kk * LANES) * VEC + e;
                    if (c == i1) v1 = v[kk][e];
                    if (c == i2) v2 = v[kk][e];
                }
            v1 = __shfl_sync(kFullMask, v1, leader + (i1 / VEC) % LANES);
            v2 = __shfl_sync(kFullMask, v2, leader + (k == 2 ? (i2 / VEC) % LANES : 0));
            if (live && g == 0) {
                values[row * int64_t(k)] = v1;
                indices[row * int64_t(k)] = float(i1);
                if (k == 2) {
                    values[row * int64_t(k) + 1] = v2;
                    indices[row * int64_t(k) + 1] = float(i2);
                }
            }
            continue;
        }
        if constexpr (LANES >= 8) {
            if (k <= LANES) {  // block-uniform
                uint32_t sel[NV][VEC];
                const uint32_t flip = largest ? 0u : 0xffffffffu;
#pragma unroll
                for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) sel[kk][e] = key[kk][e] ^ flip;
                if (topk_by_candidates<LANES, NV, VEC>(sel, avail, v, k, live, values + row * int64_t(k),
                                                       indices + row * int64_t(k), &kscratch[threadIdx.x >> 5]))
                    continue;
            }
        }
        for (int r = 0; r < k; ++r) {
            uint32_t best = largest ? 0u : 0xffffffffu;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (avail[kk][e]) best = largest ? max(best, key[kk][e]) : min(best, key[kk][e]);
            best = largest ? group_max_u32<LANES>(best) : group_min_u32<LANES>(best);
            int pick = INT_MAX;
            float val = 0.f;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int col = (g + kk * LANES) * VEC + e;
                    if (avail[kk][e] && key[kk][e] == best && col < pick) {
                        pick = col;
                        val = v[kk][e];
                    }
                }
            const int gpick = group_min_int<LANES>(pick);
            // The lane that holds the picked column passes its value to lane 0.
            const int owner = (gpick / VEC) % LANES;
            val = __shfl_sync(kFullMask, val, leader + owner);
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if ((g + kk * LANES) * VEC + e == gpick) avail[kk][e] = false;
            if (live && g == 0) {
                values[row * int64_t(k) + r] = val;
                indices[row * int64_t(k) + r] = float(gpick);
            }
        }
    }
}

// Any length and alignment: one block per row, k rounds of block reductions
// over the row re-read from global memory (L1/L2); round r takes the best entry
// ranked strictly after round r-1's pick.
template <int VEC>
__global__ void __launch_bounds__(kBlockThreads)
top_k_rows_rowblock(const float* __restrict__ x, float* __restrict__ values, float* __restrict__ indices,
                    int64_t rows, int cols, int k, int largest) {
    __shared__ uint32_t red[kBlockThreads / 32];
    __shared__ int redi[kBlockThreads / 32];
    const int nch = cols / VEC;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * int64_t(cols);
        float* vr = values + row * int64_t(k);
        float* ir = indices + row * int64_t(k);
        // The previous pick bounds the next: (key, column) strictly after it.
        uint32_t prev_key = 0;
        int prev_col = -1;
        for (int r = 0; r < k; ++r) {
            uint32_t best = largest ? 0u : 0xffffffffu;
            int best_col = INT_MAX;
            for (int c = threadIdx.x; c < nch; c += kBlockThreads) {
                float t[VEC];
                ld_chunk<VEC>(xr + c * VEC, t);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const uint32_t kx = rank_key(t[e]);
                    const int col = c * VEC + e;
                    bool after;  // strictly after the previous pick in rank order
                    if (r == 0)
                        after = true;
                    else if (largest)
                        after = kx < prev_key || (kx == prev_key && col > prev_col);
                    else
                        after = kx > prev_key || (kx == prev_key && col > prev_col);
                    const bool better = largest ? (kx > best || (kx == best && col < best_col))
                                                : (kx < best || (kx == best && col < best_col));
                    if (after && better) {
                        best = kx;
                        best_col = col;
                    }
                }
            }
            // block argbest: (key, column) in rank order
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint32_t ok = __shfl_xor_sync(kFullMask, best, o);
                const int oc = __shfl_xor_sync(kFullMask, best_col, o);
                const bool take = largest ? (ok > best || (ok == best && oc < best_col))
                                          : (ok < best || (ok == best && oc < best_col));
                if (take) {
                    best = ok;
                    best_col = oc;
                }
            }
            if (lane == 0) {
                red[w] = best;
                redi[w] = best_col;
            }
            __syncthreads();
            uint32_t bk = red[0];
            int bc = redi[0];
            for (int q = 1; q < kBlockThreads / 32; ++q) {
                const bool take = largest ? (red[q] > bk || (red[q] == bk && redi[q] < bc))
                                          : (red[q] < bk || (red[q] == bk && redi[q] < bc));
                if (take) {
                    bk = red[q];
                    bc = redi[q];
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                vr[r] = __ldg(xr + bc);
                ir[r] = float(bc);
            }
            prev_key = bk;
            prev_col = bc;
        }
    }
}

// Rows of more than 1024 floats with k <= 2: one pass.  One CTA per row
// (rows blockIdx.x, + gridDim.x, ...); each thread keeps the best two of its
// chunks (chunks c = tid, tid + NT, ...: a tournament inside each float4
// chunk, then an ordered merge into the running pair, whose columns are all
// lower), then a butterfly over the warp and one over the warps' pairs in
// shared memory.  Without NaN or infinity in the row (a finite sum of its
// values, block-wide) the ranking runs on the values themselves, negated for
// smallest-first; otherwise the row is ranked again, from the L2, on the rank
// keys (NaN above every number), and the winners' values re-read.
template <class T, int VEC>
__device__ __forceinline__ kept_detail::Top2<T> top2_chunk(const T (&v)[VEC], int col0, T lowest) {
    int cs[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) cs[e] = col0 + e;
    return kept_detail::top2_range<VEC, T>(v, cs, 0, lowest);
}

// The block's best two of each thread's pair t (every thread calls it;
// shared arrays of NT/32 pairs); returns it in every thread.
template <int NT, class T>
__device__ __forceinline__ kept_detail::Top2<T> block_top2(kept_detail::Top2<T> t, T lowest, T* sv, int* sc) {
    using kept_detail::Top2;
    constexpr int W = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const Top2<T> u{__shfl_xor_sync(kFullMask, t.v1, o), __shfl_xor_sync(kFullMask, t.v2, o),
                        __shfl_xor_sync(kFullMask, t.c1, o), __shfl_xor_sync(kFullMask, t.c2, o)};
        t = kept_detail::top2_merge<false>(t, u);
    }
    __syncthreads();  // the previous use of the shared pairs is over
    if (lane == 0) {
        sv[2 * wid] = t.v1;
        sv[2 * wid + 1] = t.v2;
        sc[2 * wid] = t.c1;
        sc[2 * wid + 1] = t.c2;
    }
    __syncthreads();
    t = lane < W ? Top2<T>{sv[2 * lane], sv[2 * lane + 1], sc[2 * lane], sc[2 * lane + 1]}
                 : Top2<T>{lowest, lowest, INT_MAX, INT_MAX};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const Top2<T> u{__shfl_xor_sync(kFullMask, t.v1, o), __shfl_xor_sync(kFullMask, t.v2, o),
                        __shfl_xor_sync(kFullMask, t.c1, o), __shfl_xor_sync(kFullMask, t.c2, o)};
        t = kept_detail::top2_merge<false>(t, u);
    }
    return t;
}

template <int NT, int VEC>
__global__ void __launch_bounds__(NT)
top_k_rows_top2(const float* __restrict__ x, float* __restrict__ values, float* __restrict__ indices,
                int64_t rows, int cols, int k, int largest) {
    using kept_detail::Top2;
    constexpr int U = 4;  // chunks in flight per thread
    __shared__ float fv[2 * (NT / 32)];
    __shared__ uint32_t kv[2 * (NT / 32)];
    __shared__ int cv[2 * (NT / 32)];
    const int tid = threadIdx.x;
    const float sgn = largest ? 1.f : -1.f;
    const uint32_t flip = largest ? 0u : 0xffffffffu;
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * int64_t(cols);
        Top2<float> t{-INFINITY, -INFINITY, INT_MAX, INT_MAX};  // no entry yet
        bool first = true;
        float probe = 0.f;
        for (int c0 = 0; c0 < nch; c0 += U * NT) {  // block-uniform
            float v[U][VEC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < nch) ld_chunk<VEC>(xr + c * VEC, v[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < nch) {
                    float xs[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        probe += v[u][e];
                        xs[e] = sgn * v[u][e];
                    }
                    const Top2<float> ct = top2_chunk<float, VEC>(xs, c * VEC, -INFINITY);
                    // a whole float4 chunk fills both places, so the running
                    // pair is always complete and the merge can be ordered;
                    // single entries merge under the full rule
                    if constexpr (VEC >= 2) t = first ? ct : kept_detail::top2_merge<true>(t, ct);
                    else t = first ? ct : kept_detail::top2_merge<false>(t, ct);
                    first = false;
                }
            }
        }
        float* vr = values + row * int64_t(k);
        float* ir = indices + row * int64_t(k);
        if (!__syncthreads_or(!(fabsf(probe) <= 3.402823466e38f))) {  // block-uniform
            t = block_top2<NT, float>(t, -INFINITY, fv, cv);
            if (tid == 0) {
                vr[0] = sgn * t.v1;
                ir[0] = float(t.c1);
                if (k == 2) {
                    vr[1] = sgn * t.v2;
                    ir[1] = float(t.c2);
                }
            }
            continue;
        }
        // NaN or infinity in the row: rank keys, the row again from the L2
        Top2<uint32_t> tk{0u, 0u, INT_MAX, INT_MAX};
        first = true;
        for (int c0 = 0; c0 < nch; c0 += U * NT) {
            float v[U][VEC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < nch) ld_chunk<VEC>(xr + c * VEC, v[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < nch) {
                    uint32_t ks[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) ks[e] = rank_key(v[u][e]) ^ flip;
                    const Top2<uint32_t> ct = top2_chunk<uint32_t, VEC>(ks, c * VEC, 0u);
                    if constexpr (VEC >= 2) tk = first ? ct : kept_detail::top2_merge<true>(tk, ct);
                    else tk = first ? ct : kept_detail::top2_merge<false>(tk, ct);
                    first = false;
                }
            }
        }
        tk = block_top2<NT, uint32_t>(tk, 0u, kv, cv);
        if (tid == 0) {
            vr[0] = xr[tk.c1];
            ir[0] = float(tk.c1);
            if (k == 2) {
                vr[1] = xr[tk.c2];
                ir[1] = float(tk.c2);
            }
        }
    }
}

// Rows of more than 1024 floats with 2 <= k <= kSelectMaxK.  One CTA per row
// (rows blockIdx.x, + gridDim.x, ...; NT = 256 threads and 4 CTAs per SM for
// rows of up to 8192 floats, 512 threads and 2 CTAs per SM beyond, so that
// other CTAs' loads overlap a CTA's selection work).  An entry's order is that
// of the 64-bit composite (key << 32) | (0xffffffff - column), key = rank key
// complemented for smallest-first: larger key first, then lower column.
//   pass 1   read the row from HBM and take each thread's largest key; each
//            is an entry of the row, so at least k entries reach tau, the
//            smallest over warps of each warp's ceil(k/W)-th largest thread
//            maximum (W warps), and the top k are among the entries at or
//            above tau;
//   pass 2   read the row again (from the L2, where it still is) and collect
//            those candidates in shared memory; when there are at most
//            kSelectMaxCand of them (for logits, a few times k), sort them
//            (bitonic) and write the first k.
// Otherwise (large k, or many entries tied at tau) a radix select over the
// row, again from the L2, finds the k-th largest key T: four passes each
// histogram one byte of the keys whose higher bytes match the prefix found so
// far; then the entries above T and the lowest columns equal to T (in column
// order: a block scan per tile of the row) are collected and sorted.
// Values are re-read from the row for the output, keeping their bits.
constexpr int kSelectMaxK = 1024;
constexpr int kSelectMaxCand = 2048;
constexpr int kSelectUnroll = 4;

template <int NT>
struct SelectSmem {
    uint64_t cand[kSelectMaxCand];  // composites: candidates, or the collected k
    uint32_t hist[256];
    uint32_t wtau[NT / 32];
    int scan[NT / 32];
    int count;
    uint32_t prefix;
    int need;
};

__device__ __forceinline__ uint32_t select_key(float v, uint32_t flip) { return rank_key(v) ^ flip; }

__device__ __forceinline__ uint64_t composite(uint32_t key, int col) {
    return (uint64_t(key) << 32) | uint32_t(0xffffffffu - uint32_t(col));
}

// Adds this warp's `in` lanes to hist[bin], one atomic per distinct bin.  Every
// lane of the warp calls it.
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, bool in, uint32_t bin, int lane) {
    unsigned todo = __ballot_sync(kFullMask, in);
    while (todo) {
        const int leader = __ffs(todo) - 1;
        const uint32_t lb = __shfl_sync(kFullMask, bin, leader);
        const unsigned same = __ballot_sync(kFullMask, in && bin == lb);
        if (lane == leader) atomicAdd(&hist[lb], uint32_t(__popc(same)));
        todo &= ~same;
    }
}

// Sorts s[0, n) into descending order with the whole block (n a power of two;
// s complete on entry, sorted and visible to every thread on return).
__device__ void block_bitonic_desc(uint64_t* s, int n) {
    for (int kk = 2; kk <= n; kk <<= 1)
        for (int j = kk >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t a = s[i], b = s[l];
                    const bool desc = (i & kk) == 0;
                    if (desc ? (a < b) : (a > b)) {
                        s[i] = b;
                        s[l] = a;
                    }
                }
            }
            __syncthreads();
        }
}

// Pads s[n0, pow2) with 0 (below every entry), sorts, and writes the first k.
__device__ void sort_and_write(uint64_t* s, int n0, int k, const float* __restrict__ xr, float* vr, float* ir) {
    int n = 2;
    while (n < n0) n <<= 1;
    for (int i = n0 + int(threadIdx.x); i < n; i += blockDim.x) s[i] = 0;
    __syncthreads();
    block_bitonic_desc(s, n);
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
        const int col = int(0xffffffffu - uint32_t(s[i]));
        vr[i] = __ldg(xr + col);
        ir[i] = float(col);
    }
    __syncthreads();  // shared memory is rebuilt for the next row
}

template <int NT, int VEC>
__global__ void __launch_bounds__(NT, 1024 / NT)
top_k_rows_select(const float* __restrict__ x, float* __restrict__ values, float* __restrict__ indices,
                  int64_t rows, int cols, int k, int largest) {
    constexpr int W = NT / 32;
    __shared__ SelectSmem<NT> sm;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t flip = largest ? 0u : 0xffffffffu;
    const int nch = cols / VEC;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * int64_t(cols);
        float* vr = values + row * int64_t(k);
        float* ir = indices + row * int64_t(k);
        // pass 1: each thread's largest key
        uint32_t tmax = 0;
        bool has = false;
        for (int c0 = 0; c0 < nch; c0 += kSelectUnroll * NT) {  // block-uniform
            float t[kSelectUnroll][VEC];
#pragma unroll
            for (int u = 0; u < kSelectUnroll; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < nch) ld_chunk<VEC>(xr + c * VEC, t[u]);
            }
#pragma unroll
            for (int u = 0; u < kSelectUnroll; ++u)
                if (c0 + u * NT + tid < nch) {
                    has = true;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) tmax = max(tmax, select_key(t[u][e], flip));
                }
        }
        // tau: each warp's m-th largest maximum (m = ceil(k/W); a thread
        // without entries counts as key 0, which every key reaches; m > 32
        // gives no bound), then the smallest over warps
        {
            uint32_t v = has ? tmax : 0u;
#pragma unroll
            for (int kk = 2; kk <= 32; kk <<= 1)  // warp bitonic sort, descending by lane
#pragma unroll
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    const uint32_t o = __shfl_xor_sync(kFullMask, v, j);
                    const bool lower = (lane & j) == 0;
                    const bool desc = (lane & kk) == 0;
                    v = (lower == desc) ? max(v, o) : min(v, o);
                }
            const int m = (k + W - 1) / W;
            const uint32_t wt = m <= 32 ? __shfl_sync(kFullMask, v, m - 1) : 0u;
            if (lane == 0) sm.wtau[wid] = wt;
            if (tid == 0) sm.count = 0;
        }
        __syncthreads();
        uint32_t tau = sm.wtau[0];
        for (int w = 1; w < W; ++w) tau = min(tau, sm.wtau[w]);
        // pass 2: the candidates (warp-aggregated slots)
        for (int c0 = 0; c0 < nch; c0 += kSelectUnroll * NT) {  // block-uniform
            float t[kSelectUnroll][VEC];
#pragma unroll
            for (int u = 0; u < kSelectUnroll; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < nch) ld_chunk<VEC>(xr + c * VEC, t[u]);
            }
#pragma unroll
            for (int u = 0; u < kSelectUnroll; ++u) {
                const int c = c0 + u * NT + tid;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const uint32_t kx = c < nch ? select_key(t[u][e], flip) : 0u;
                    const bool cand = c < nch && kx >= tau;
                    const unsigned bal = __ballot_sync(kFullMask, cand);
                    if (bal == 0) continue;  // warp-uniform
                    int base = 0;
                    if (lane == 0) base = atomicAdd(&sm.count, __popc(bal));
                    base = __shfl_sync(kFullMask, base, 0);
                    const int slot = base + __popc(bal & ((1u << lane) - 1u));
                    if (cand && slot < kSelectMaxCand) sm.cand[slot] = composite(kx, c * VEC + e);
                }
            }
        }
        __syncthreads();
        const int ncand = sm.count;
        if (ncand <= kSelectMaxCand) {  // block-uniform
            sort_and_write(sm.cand, ncand, k, xr, vr, ir);
            continue;
        }
        // radix select of the k-th largest key, over the row in the L2
        uint32_t prefix = 0, pmask = 0;
        int kr = k;  // entries still to find at or below the current prefix
        for (int shift = 24; shift >= 0; shift -= 8) {
            if (tid < 256) sm.hist[tid] = 0;
            __syncthreads();
            for (int c0 = 0; c0 < nch; c0 += NT) {  // block-uniform
                const int c = c0 + tid;
                float t[VEC];
                if (c < nch) ld_chunk<VEC>(xr + c * VEC, t);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const uint32_t kx = c < nch ? select_key(t[e], flip) : 0u;
                    const bool in = c < nch && (kx & pmask) == prefix;
                    warp_hist_add(sm.hist, in, (kx >> shift) & 255u, lane);
                }
            }
            __syncthreads();
            if (wid == 0) {
                // bins from the top: lane l covers bins 255-8l .. 248-8l
                uint32_t cnt[8], part = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    cnt[q] = sm.hist[255 - 8 * lane - q];
                    part += cnt[q];
                }
                uint32_t incl = part;  // inclusive scan over lanes (top bins first)
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t excl = incl - part;
                const unsigned hit = __ballot_sync(kFullMask, excl < uint32_t(kr) && uint32_t(kr) <= incl);
                if (lane == __ffs(hit) - 1) {
                    uint32_t above = excl;
                    int b = 255 - 8 * lane;
                    for (int q = 0; q < 8; ++q, --b) {
                        if (above + cnt[q] >= uint32_t(kr)) break;
                        above += cnt[q];
                    }
                    sm.prefix = prefix | (uint32_t(b) << shift);
                    sm.need = kr - int(above);
                }
            }
            __syncthreads();
            prefix = sm.prefix;
            kr = sm.need;
            pmask |= 255u << shift;
        }
        // collect: entries above T, and the kr lowest columns equal to T; a
        // tile of the row is NT consecutive chunks, one per thread, so thread
        // order is column order within a tile
        const uint32_t T = prefix;
        if (tid == 0) sm.count = 0;
        int taken_eq = 0;  // entries equal to T taken in earlier tiles
        __syncthreads();
        for (int c0 = 0; c0 < nch; c0 += NT) {  // block-uniform
            const int c = c0 + tid;
            float t[VEC];
            uint32_t kx[VEC];
            int eq = 0;
            if (c < nch) {
                ld_chunk<VEC>(xr + c * VEC, t);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    kx[e] = select_key(t[e], flip);
                    eq += kx[e] == T ? 1 : 0;
                }
            }
            int incl = eq;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sm.scan[wid] = incl;
            __syncthreads();
            int wbase = 0, tile_eq = 0;
            for (int w = 0; w < W; ++w) {
                const int v = sm.scan[w];
                if (w < wid) wbase += v;
                tile_eq += v;
            }
            int r = taken_eq + wbase + incl - eq;  // rank among equal entries of this thread's first
            if (c < nch) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    bool take = kx[e] > T;
                    if (kx[e] == T) take = r++ < kr;
                    if (take) sm.cand[atomicAdd(&sm.count, 1)] = composite(kx[e], c * VEC + e);
                }
            }
            taken_eq += tile_eq;
            __syncthreads();  // sm.scan is rewritten by the next tile
        }
        sort_and_write(sm.cand, k, k, xr, vr, ir);
    }
}

}  // namespace

cudaError_t launch_router(const float* x, const uint8_t* mask, float* p, float* kept, int64_t rows,
                          int64_t cols, int64_t k, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        router_group<G::LANES, G::NV, G::VEC><<<group_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            x, mask, p, kept, rows, int(cols), int(k));
    });
    if (done) {
        note_launches(1);
        return cudaGetLastError();
    }
    // Rows longer than a warp holds: the two ops one after the other.
    cudaError_t err = launch_masked_softmax(x, mask, p, rows, cols, vec4, stream);
    if (err != cudaSuccess) return err;
    return launch_topk_kept(p, kept, rows, cols, k, vec4, stream);
}

cudaError_t launch_top_k_rows(const float* x, float* values, float* indices, int64_t rows, int64_t cols,
                              int64_t k, bool largest, bool vec4, cudaStream_t stream) {
    const bool done = with_geometry(vec4, cols, [&](auto geo) {
        using G = decltype(geo);
        top_k_rows_group<G::LANES, G::NV, G::VEC><<<stream_grid(rows, G::LANES), kBlockThreads, 0, stream>>>(
            x, values, indices, rows, int(cols), int(k), largest ? 1 : 0);
    });
    cudaError_t err = cudaSuccess;
    const int sms = sm_count();
    if (!done && k <= 2 && sms > 0) {
        // as many CTAs of 256 threads as are resident (on GB300, 2048 x 50304,
        // k = 2, back to back: 256 threads 69.6 us, 128 71.9, 512 82.4, 1024
        // 101.6; the two-pass select took 183)
        auto launch = [&](auto kern) {
            int per_sm = 0;
            constexpr int nt = 256;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nt, 0) != cudaSuccess || per_sm < 1)
                per_sm = 1;
            const int64_t cap = int64_t(sms) * per_sm;
            kern<<<unsigned(rows < cap ? rows : cap), nt, 0, stream>>>(x, values, indices, rows, int(cols),
                                                                        int(k), largest ? 1 : 0);
        };
        if (vec4) launch(top_k_rows_top2<256, 4>);
        else launch(top_k_rows_top2<256, 1>);
    } else if (!done && k >= 2 && k <= kSelectMaxK && sms > 0) {
        auto launch = [&](auto kern, int nt, int per_sm) {
            const int64_t cap = int64_t(sms) * per_sm;
            const unsigned grid = unsigned(rows < cap ? rows : cap);
            kern<<<grid, nt, 0, stream>>>(x, values, indices, rows, int(cols), int(k), largest ? 1 : 0);
        };
        if (cols <= 8192) {  // 4 CTAs of 256 threads per SM
            if (vec4) launch(top_k_rows_select<256, 4>, 256, 4);
            else launch(top_k_rows_select<256, 1>, 256, 4);
        } else {  // 2 CTAs of 512 threads per SM: 61 MB of 50304-float rows stay in the L2
            if (vec4) launch(top_k_rows_select<512, 4>, 512, 2);
            else launch(top_k_rows_select<512, 1>, 512, 2);
        }
    } else if (!done) {
        if (vec4)
            top_k_rows_rowblock<4><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, values, indices, rows,
                                                                                 int(cols), int(k), largest);
        else
            top_k_rows_rowblock<1><<<row_grid(rows), kBlockThreads, 0, stream>>>(x, values, indices, rows,
                                                                                 int(cols), int(k), largest);
    }
    note_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace rowops
