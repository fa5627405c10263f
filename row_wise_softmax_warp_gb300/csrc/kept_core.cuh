// kept_core.cuh - the kept-mask selection for a row held by a lane group
// (geometry of common.cuh), shared by the kept-mask kernel and the fused router.
//
// Without NaN, "beats" (TorchLean Spec.MoE.kept: j beats i when x_j > x_i, or
// when neither is larger and j < i) is a strict total order: larger value first,
// and among equal values (-0 == +0 included) the lower column.  The entries
// beating i are then exactly those ranked above it, so kept_i = [rank_i < k],
// found exactly without counting:
//   k <= 2      each lane's best two (value, column) pairs by a branch-free
//               tournament over its entries in column order, then a
//               butterfly merge of the pairs across the group;
//   k <= LANES  (groups of 8 or more lanes, with per-warp shared scratch)
//               candidates: each lane's largest value is an entry of the row,
//               so at least k entries reach tau, the k-th largest of the
//               group's lane maxima, and every entry ranked above an entry
//               that reaches tau reaches it too.  When at most 32 entries of
//               each row of the warp reach tau, they are ranked among
//               themselves by counting; otherwise the rounds below run;
//   k <= 8      k rounds of "best remaining entry": a group max of the
//               remaining floats, then a group min of the columns holding that
//               value (the index tie-break);
//   cols-k <= 8 the same from the bottom (min value, highest column): the
//               cols-k entries found are the ones dropped;
//   otherwise   a bitwise radix select of the k-th largest 64-bit key
//               (order-preserving value bits << 32 | cols-1-column).
// A NaN is neither larger nor smaller than anything, which makes the relation
// intransitive; a warp that meets a NaN in any of its rows counts beats
// literally, O(cols) comparisons per entry.  Either way the result equals the
// literal compare-and-count bit for bit.
#pragma once

#include <climits>

#include "common.cuh"

namespace rowops {
// Per-warp shared-memory scratch of the candidate path: for each group of the
// warp (at most 4: groups of 8 or more lanes) 32 candidate slots and the kept
// bits of a row of up to 1024 columns.
struct KeptScratch {
    float v[4][32];
    int c[4][32];
    unsigned bits[4][32];
};

namespace kept_detail {

constexpr int kMaxRounds = 8;

// (xv, xc) comes before (yv, yc) in the rule's order (no NaN): larger value,
// or equal value (-0 == +0) and lower column.
__device__ __forceinline__ bool beats(float xv, int xc, float yv, int yc) {
    return xv > yv || (xv == yv && xc < yc);
}

// The best two entries of a set, (v1, c1) ahead of (v2, c2): larger key, or
// equal keys and the lower column.  T is float (no NaN: -0 == +0 ties) or an
// order-preserving uint32 key.
template <class T>
struct Top2 {
    T v1, v2;
    int c1, c2;
};

template <class T>
__device__ __forceinline__ bool ahead(T av, int ac, T bv, int bc) {
    return av > bv || (av == bv && ac < bc);
}

// Top2 of two entries, a's column below b's.
template <class T>
__device__ __forceinline__ Top2<T> top2_pair(T av, int ac, T bv, int bc) {
    const bool t = av >= bv;  // equal keys: the lower column, a
    return Top2<T>{t ? av : bv, t ? bv : av, t ? ac : bc, t ? bc : ac};
}

// Top2 of the union of two disjoint sets; with `ordered` every column of a is
// below every column of b, so equal keys go to a without comparing columns.
template <bool ordered, class T>
__device__ __forceinline__ Top2<T> top2_merge(const Top2<T>& a, const Top2<T>& b) {
    const bool t = ordered ? a.v1 >= b.v1 : !ahead(b.v1, b.c1, a.v1, a.c1);
    // the runner-up is the better of the winner's second and the loser's first
    const T av = t ? a.v2 : a.v1, bv = t ? b.v1 : b.v2;
    const int ac = t ? a.c2 : a.c1, bc = t ? b.c1 : b.c2;
    const bool u = ordered ? av >= bv : !ahead(bv, bc, av, ac);
    return Top2<T>{t ? a.v1 : b.v1, u ? av : bv, t ? a.c1 : b.c1, u ? ac : bc};
}

// Top2 of entries [lo, lo + N) of a lane's list (columns increasing along
// it): a tournament of adjacent blocks, so every merge is an ordered one.
// `lowest` is a key no entry is below: the empty runner-up place of a single
// entry.  The left block takes the larger half, so a single entry is only
// ever a right block, where a tie with the empty place goes to the real entry
// on the left.
template <int N, class T>
__device__ __forceinline__ Top2<T> top2_range(const T* x, const int* c, int lo, T lowest) {
    if constexpr (N == 1) {
        return Top2<T>{x[lo], lowest, c[lo], INT_MAX};
    } else if constexpr (N == 2) {
        return top2_pair(x[lo], c[lo], x[lo + 1], c[lo + 1]);
    } else {
        return top2_merge<true>(top2_range<N - N / 2>(x, c, lo, lowest),
                                top2_range<N / 2>(x, c, lo + N - N / 2, lowest));
    }
}

// The group's best two: each lane's by the tournament over its E entries in
// column order, then a butterfly merging the lanes' pairs (disjoint at every
// round) under the full rule, where an empty place (column INT_MAX) loses
// every tie; every lane of the group ends with the result.
template <int LANES, int E, class T>
__device__ __forceinline__ Top2<T> group_top2(const T (&x)[E], const int (&c)[E], T lowest) {
    Top2<T> t = top2_range<E>(x, c, 0, lowest);
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) {
        const Top2<T> u{__shfl_xor_sync(kFullMask, t.v1, o), __shfl_xor_sync(kFullMask, t.v2, o),
                        __shfl_xor_sync(kFullMask, t.c1, o), __shfl_xor_sync(kFullMask, t.c2, o)};
        t = top2_merge<false>(t, u);
    }
    return t;
}

__device__ __forceinline__ uint64_t make_key(float x, int col, int cols) {
    return (uint64_t(ordered_key(x)) << 32) | uint32_t(cols - 1 - col);
}

// Number of low-word bits that can be nonzero: cols - 1 < 2^lb.
__device__ __forceinline__ int low_bits(int cols) { return cols <= 1 ? 0 : 32 - __clz(cols - 1); }

// The candidate path (see the file comment).  Returns false, touching nothing,
// when a row of the warp has more than 32 candidates; warp-uniform.
template <int LANES, int NV, int VEC>
__device__ __forceinline__ bool kept_by_candidates(const float (&v)[NV][VEC], const bool (&valid)[NV][VEC],
                                                   int k, bool (&keep)[NV][VEC], KeptScratch* ks) {
    const int g = threadIdx.x % LANES;
    const int leader = (threadIdx.x & 31) - g;
    const int gi = (threadIdx.x & 31) / LANES;
    float lm = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (valid[kk][e]) lm = fmaxf(lm, v[kk][e]);
    // the group's lane maxima in descending order (bitonic network over g)
    float s = lm;
#pragma unroll
    for (int kk = 2; kk <= LANES; kk <<= 1)
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
            const float o = __shfl_xor_sync(kFullMask, s, j);
            const bool lower = (g & j) == 0;
            const bool desc = (g & kk) == 0;
            s = (lower == desc) ? fmaxf(s, o) : fminf(s, o);
        }
    const float tau = __shfl_sync(kFullMask, s, leader + k - 1);
    int cnt = 0;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e) cnt += (valid[kk][e] && v[kk][e] >= tau) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, o, LANES);
        if (g >= o) incl += y;
    }
    const int total = __shfl_sync(kFullMask, incl, leader + LANES - 1);
    if (__any_sync(kFullMask, total > 32)) return false;
    float* sv = ks->v[gi];
    int* sc = ks->c[gi];
    unsigned* sb = ks->bits[gi];
    __syncwarp();  // the warp's previous use of the scratch is over
    for (int w = g; w < 32; w += LANES) sb[w] = 0u;
    int slot = incl - cnt;
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (valid[kk][e] && v[kk][e] >= tau) {
                sv[slot] = v[kk][e];
                sc[slot] = (g + kk * LANES) * VEC + e;
                ++slot;
            }
    __syncwarp();
    for (int i = g; i < total; i += LANES) {
        const float vi = sv[i];
        const int ci = sc[i];
        int rank = 0;
        for (int q = 0; q < total; ++q) rank += beats(sv[q], sc[q], vi, ci) ? 1 : 0;
        if (rank < k) atomicOr(&sb[ci >> 5], 1u << (ci & 31));
    }
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int col = (g + kk * LANES) * VEC + e;
            keep[kk][e] = valid[kk][e] && ((sb[col >> 5] >> (col & 31)) & 1u) != 0u;
        }
    return true;
}

}  // namespace kept_detail

// k <= 2 on a row that fills every lane's entries, with no NaN in the warp's
// rows: the row's best two by group_top2, then zeros over the whole row and
// 1.0 at the one or two winning columns, each stored by the lane that wrote
// that column's chunk (in that order, so the 1.0 lands last): the same mask as
// kept_select, without a comparison per entry.  kr is the row's mask, written
// only when `live`.  Every lane of the warp must call it.
template <int LANES, int NV, int VEC>
__device__ __forceinline__ void kept_store_top2_full(const float (&v)[NV][VEC], int k, bool live, float* kr) {
    const int g = threadIdx.x % LANES;
    constexpr int E = NV * VEC;
    float xs[E];
    int cs[E];
#pragma unroll
    for (int kk = 0; kk < NV; ++kk)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            xs[kk * VEC + e] = v[kk][e];
            cs[kk * VEC + e] = (g + kk * LANES) * VEC + e;
        }
    const kept_detail::Top2<float> t = kept_detail::group_top2<LANES, E, float>(xs, cs, -INFINITY);
    if (live) {
#pragma unroll
        for (int kk = 0; kk < NV; ++kk) st_zero_chunk<VEC>(kr + (g + kk * LANES) * VEC);
        if ((t.c1 / VEC) % LANES == g) kr[t.c1] = 1.f;
        if (k == 2 && (t.c2 / VEC) % LANES == g) kr[t.c2] = 1.f;
    }
}

// Loads row `row` into a group's registers (zeros outside the row or past the
// last row); read-only input.
template <int LANES, int NV, int VEC>
__device__ __forceinline__ void kept_load_row(const float* __restrict__ x, int64_t row, int64_t rows, int cols,
                                              float (&v)[NV][VEC]) {
    const int g = threadIdx.x % LANES;
    const int nch = cols / VEC;
    const bool live = row < rows;
    const int64_t off = (live ? row : 0) * int64_t(cols);
#pragma unroll
    for (int kk = 0; kk < NV; ++kk) {
        const int c = g + kk * LANES;
        if (live && c < nch) {
            ld_chunk<VEC>(x + off + c * VEC, v[kk]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[kk][e] = 0.f;
        }
    }
}

// Sets keep[kk][e] for this lane's entries of the row its group holds.  `valid`
// marks entries inside the row; any_nan must be warp-uniform (true when any
// group of the warp has a NaN in its row).  Every lane of the warp must call it.
template <int LANES, int NV, int VEC>
__device__ __forceinline__ void kept_select(const float (&v)[NV][VEC], const bool (&valid)[NV][VEC],
                                            bool any_nan, int cols, int k, bool (&keep)[NV][VEC],
                                            KeptScratch* ks = nullptr) {
    using namespace kept_detail;
    const int g = threadIdx.x % LANES;
    const int leader = (threadIdx.x & 31) - g;
    const int lb = low_bits(cols);
    if (any_nan) {
        // A NaN makes "beats" intransitive: count beats literally (warp-uniform branch).
        int cnt[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) cnt[kk][e] = 0;
#pragma unroll
        for (int ko = 0; ko < NV; ++ko)
#pragma unroll
            for (int eo = 0; eo < VEC; ++eo)
                for (int o = 0; o < LANES; ++o) {
                    const float xj = __shfl_sync(kFullMask, v[ko][eo], leader + o);
                    const int j = (o + ko * LANES) * VEC + eo;
                    if (j < cols) {
#pragma unroll
                        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                            for (int e = 0; e < VEC; ++e) {
                                const int i = (g + kk * LANES) * VEC + e;
                                const float xi = v[kk][e];
                                const bool larger = xj > xi;
                                const bool neither = !(xj > xi) && !(xi > xj);
                                cnt[kk][e] += (larger || (neither && j < i)) ? 1 : 0;
                            }
                    }
                }
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) keep[kk][e] = cnt[kk][e] < k;
    } else if (k <= 2) {
        // Top two: each lane's best two by a tournament over its entries in
        // column order (an entry outside the row counts as -inf at its own
        // column, which is above every column of the row, so it loses every
        // tie); then a butterfly merges the lanes' pairs under the full rule,
        // and every lane ends with the row's best two.  A row has at least
        // k entries, so no entry outside it is picked.
        // (When the row fills every lane's entries, no entry lies outside it
        // and the substitution is skipped: a row past the last one is not
        // stored.)
        constexpr int E = NV * VEC;
        float xs[E];
        int cs[E];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) cs[kk * VEC + e] = (g + kk * LANES) * VEC + e;
        Top2<float> t;
        if (cols == LANES * E) {  // warp-uniform
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) xs[kk * VEC + e] = v[kk][e];
            t = group_top2<LANES, E, float>(xs, cs, -INFINITY);
        } else {
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) xs[kk * VEC + e] = valid[kk][e] ? v[kk][e] : -INFINITY;
            t = group_top2<LANES, E, float>(xs, cs, -INFINITY);
        }
        const int i1 = t.c1, i2 = k == 1 ? -1 : t.c2;
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int c = (g + kk * LANES) * VEC + e;
                keep[kk][e] = c == i1 || c == i2;
            }
    } else if (LANES >= 8 && k <= LANES && ks != nullptr && cols <= 1024 &&
               kept_by_candidates<LANES, NV, VEC>(v, valid, k, keep, ks)) {
        // ranked among the candidates
    } else if (k <= kMaxRounds || cols - k <= kMaxRounds) {
        // Rounds of "best remaining entry".  Without NaN, float comparison is
        // the order of the rule (-0 == +0 ties, broken by column): from the
        // top, the largest value and the lowest column holding it; from the
        // bottom, the smallest value and the highest column holding it.
        const bool top = k <= kMaxRounds;
        const int rounds = top ? k : cols - k;
        bool taken[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) taken[kk][e] = false;
        for (int r = 0; r < rounds; ++r) {
            float best = top ? -INFINITY : INFINITY;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (valid[kk][e] && !taken[kk][e])
                        best = top ? fmaxf(best, v[kk][e]) : fminf(best, v[kk][e]);
            best = top ? group_max<LANES>(best) : group_min<LANES>(best);
            int pick = top ? INT_MAX : -1;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int col = (g + kk * LANES) * VEC + e;
                    if (valid[kk][e] && !taken[kk][e] && v[kk][e] == best)
                        pick = top ? min(pick, col) : max(pick, col);
                }
            pick = top ? group_min_int<LANES>(pick) : group_max_int<LANES>(pick);
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) taken[kk][e] |= ((g + kk * LANES) * VEC + e) == pick;
        }
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) keep[kk][e] = top ? taken[kk][e] : !taken[kk][e];
    } else {
        // Radix select of the k-th largest 64-bit key (value, cols-1-col).
        uint64_t key[NV][VEC];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) key[kk][e] = make_key(v[kk][e], (g + kk * LANES) * VEC + e, cols);
        uint64_t t = 0;
        for (int b = 63; b >= 0; --b) {
            if (b < 32 && b >= lb) continue;  // low-word bits that are always 0
            const uint64_t cand = t | (uint64_t(1) << b);
            int n = 0;
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int e = 0; e < VEC; ++e) n += (valid[kk][e] && key[kk][e] >= cand) ? 1 : 0;
            if (group_sum_int<LANES>(n) >= k) t = cand;
        }
#pragma unroll
        for (int kk = 0; kk < NV; ++kk)
#pragma unroll
            for (int e = 0; e < VEC; ++e) keep[kk][e] = key[kk][e] >= t;
    }
}

}  // namespace rowops
