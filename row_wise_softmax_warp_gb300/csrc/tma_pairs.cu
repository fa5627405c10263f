// tma_pairs.cu - long rows with two inputs, streamed through the bulk-copy
// ring (pipeline.cuh) as chunk pairs, twice per row: weighted-logits and
// fixed-teacher cross-entropy (tma_rows2) and the softmax backward
// (tma_softmax_bwd).  The second pass reads the rows again from the L2.
#include "launch.h"
#include "pipeline.cuh"

namespace rowops {
namespace {

// Two-input kernel (tma_rows2): chunks of at most 12288 floats.
constexpr int64_t kMaxChunk2 = 12288;

// ----------------------------------------------- two-input rows, two passes
// Producer of the two-input kernels (one lane): the chunk pairs (x_k, w_k) of
// each of the CTA's rows, twice (pass 0 with the evict-normal L2 policy, pass 1
// evict-first), into consecutive ring slots.
__device__ void produce_pairs(const float* x, const float* w, int64_t rows, int cols, int chunk, int nslot,
                              float* buf, uint64_t* full, uint64_t* empty, volatile int* abort_flag) {
    const uint64_t keep = policy_evict_normal(), drop = policy_evict_first();
    uint64_t n = 0;
    bool ok = true;
    for (int64_t row = blockIdx.x; ok && row < rows; row += gridDim.x) {
        int head, body;
        row_split(x + row * int64_t(cols), cols, head, body);
        const float* src[2] = {x + row * int64_t(cols) + head, w + row * int64_t(cols) + head};
        const int nch = (body + chunk - 1) / chunk;
        for (int pass = 0; ok && pass < 2; ++pass)
            for (int k = 0; ok && k < nch; ++k)
                for (int in = 0; in < 2; ++in, ++n) {
                    const int s = int(n % nslot);
                    const uint64_t use = n / nslot;
                    if (use > 0 && !mbar_wait(&empty[s], uint32_t((use - 1) & 1), abort_flag)) {
                        raise_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    const int cnt = min(chunk, body - k * chunk);
                    mbar_arrive_expect_tx(&full[s], uint32_t(cnt) * 4u);
                    bulk_load_hint(buf + size_t(s) * chunk, src[in] + size_t(k) * chunk, uint32_t(cnt) * 4u,
                                   &full[s], pass == 0 ? keep : drop);
                }
    }
    if (!ok) {
        // Let the copies already issued land before the CTA's shared memory goes away.
        const uint64_t first = n > uint64_t(nslot) ? n - nslot : 0;
        for (uint64_t j = first; j < n; ++j) {
            volatile int never = 0;
            mbar_wait(&full[j % nslot], uint32_t((j / nslot) & 1), &never);
        }
    }
}

// Weighted-logits and fixed-teacher cross-entropy on long rows: x (logits or
// student) and w (weights or teacher logits) stream through the ring as
// chunk pairs (x_k, w_k), twice per row: pass 0 folds the running (max, sum)
// of x and of the teacher (or the weight sum), pass 1 forms the loss and the
// gradient.  A CTA has one row pair in flight, so on 152 SMs the second pass
// reads rows that the first pass brought into the L2 a moment earlier: HBM sees
// one read of each input element and one write of each gradient element.
// Rows are split at their first 16-byte boundary as above; x and w share
// their alignment modulo 16 bytes (checked by the launcher); a gradient on
// another 16-byte phase is written with scalar stores.  The kernel choice does
// not depend on the gradient, so the row losses are the same bits with and
// without it.
template <bool TEACHER>
__global__ void __launch_bounds__(kTmaThreads, 1)
tma_rows2(const float* x, const float* w, float* grad, float* __restrict__ row_loss, int64_t rows, int cols,
          int chunk, int nslot, float grad_scale, bool grad_vec) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* buf = reinterpret_cast<float*>(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + size_t(nslot) * chunk * sizeof(float));
    uint64_t* empty = full + nslot;
    __shared__ uint64_t red_bar[2];
    __shared__ float red[2][kConsumerWarps][4];
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // The mean-loss kernel may be scheduled now; it waits for this grid.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    if (tid == 0) {
        for (int s = 0; s < nslot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(&red_bar[0], kConsumerWarps);
        mbar_init(&red_bar[1], kConsumerWarps);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) produce_pairs(x, w, rows, cols, chunk, nslot, buf, full, empty, &abort_flag);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ct = tid - 32;
    const int cw = warp - 1;
    uint64_t n = 0;    // slot uses consumed
    uint32_t rv = 0;   // rendezvous so far
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * int64_t(cols);
        const float* wr = w + row * int64_t(cols);
        int head, body;
        row_split(xr, cols, head, body);
        const int nch = (body + chunk - 1) / chunk;
        int ej = -1;  // head (warp 0) and tail (warp 1) lanes, as in tma_rows
        if (ct < head) ej = ct;
        else if (ct >= 32 && ct - 32 < cols - head - body) ej = head + body + (ct - 32);
        const float xe = ej >= 0 ? __ldg(xr + ej) : -INFINITY;
        const float we = ej >= 0 ? __ldg(wr + ej) : (TEACHER ? -INFINITY : 0.f);
        // pass 0: (max, sum) of x; teacher (max, sum) or the weight sum
        float ma = -INFINITY, sa = 0.f, mb = -INFINITY, sb = 0.f;
        if (ej >= 0) {
            push1(ma, sa, xe);
            if constexpr (TEACHER) push1(mb, sb, we); else sb += we;
        }
        for (int k = 0; k < nch; ++k, n += 2) {
            if (!wait_use(full, nslot, n, &abort_flag) || !wait_use(full, nslot, n + 1, &abort_flag)) return;
            const int cnt4 = min(chunk, body - k * chunk) >> 2;
            const float4* ca = reinterpret_cast<const float4*>(buf + size_t(n % nslot) * chunk);
            const float4* cb = reinterpret_cast<const float4*>(buf + size_t((n + 1) % nslot) * chunk);
            for (int i = ct; i < cnt4; i += kConsumers) {
                push4(ma, sa, ca[i]);
                const float4 b = cb[i];
                if constexpr (TEACHER) push4(mb, sb, b); else sb += (b.x + b.y) + (b.z + b.w);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[n % nslot]);
                mbar_arrive(&empty[(n + 1) % nslot]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            merge2(ma, sa, __shfl_xor_sync(kFullMask, ma, o), __shfl_xor_sync(kFullMask, sa, o));
            if constexpr (TEACHER)
                merge2(mb, sb, __shfl_xor_sync(kFullMask, mb, o), __shfl_xor_sync(kFullMask, sb, o));
            else
                sb += __shfl_xor_sync(kFullMask, sb, o);
        }
        float all[kConsumerWarps][4];
        const float mine[4] = {ma, sa, mb, sb};
        if (!rendezvous4(red, red_bar, cw, lane, rv, mine, all, &abort_flag)) return;
        float MA = all[0][0], SA = all[0][1], MB = all[0][2], SB = all[0][3];
        for (int q = 1; q < kConsumerWarps; ++q) {
            merge2(MA, SA, all[q][0], all[q][1]);
            if constexpr (TEACHER) merge2(MB, SB, all[q][2], all[q][3]); else SB += all[q][3];
        }
        const float lse = MA + logf(SA);
        const float inv_sa = 1.0f / SA;
        const float qs = TEACHER ? 1.0f / SB : 1.f;
        // pass 1: loss and gradient
        float loss = 0.f;
        float* dst = grad != nullptr ? grad + row * int64_t(cols) : nullptr;
        auto element = [&](float a, float b, float& o) {
            const float q = TEACHER ? ex2((b - MB) * kLog2e) * qs : b;
            loss = fmaf(q, lse - a, loss);
            const float p = ex2((a - MA) * kLog2e) * inv_sa;
            o = TEACHER ? grad_scale * (p - q) : grad_scale * (p * SB - q);
        };
        if (ej >= 0) {
            float o;
            element(xe, we, o);
            if (dst != nullptr) dst[ej] = o;
        }
        for (int k = 0; k < nch; ++k, n += 2) {
            if (!wait_use(full, nslot, n, &abort_flag) || !wait_use(full, nslot, n + 1, &abort_flag)) return;
            const int cnt4 = min(chunk, body - k * chunk) >> 2;
            const float4* ca = reinterpret_cast<const float4*>(buf + size_t(n % nslot) * chunk);
            const float4* cb = reinterpret_cast<const float4*>(buf + size_t((n + 1) % nslot) * chunk);
            float* dk = dst != nullptr ? dst + head + size_t(k) * chunk : nullptr;
            for (int i = ct; i < cnt4; i += kConsumers) {
                const float4 a = ca[i], b = cb[i];
                float4 o;
                element(a.x, b.x, o.x);
                element(a.y, b.y, o.y);
                element(a.z, b.z, o.z);
                element(a.w, b.w, o.w);
                if (dk != nullptr) {
                    if (grad_vec) {
                        __stcs(reinterpret_cast<float4*>(dk) + i, o);  // evict first
                    } else {  // grad on another 16-byte phase than x: four stores
                        __stcs(dk + 4 * i, o.x);
                        __stcs(dk + 4 * i + 1, o.y);
                        __stcs(dk + 4 * i + 2, o.z);
                        __stcs(dk + 4 * i + 3, o.w);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[n % nslot]);
                mbar_arrive(&empty[(n + 1) % nslot]);
            }
        }
        loss = group_sum<32>(loss);
        const float mine2[4] = {loss, 0.f, 0.f, 0.f};
        if (!rendezvous4(red, red_bar, cw, lane, rv, mine2, all, &abort_flag)) return;
        if (ct == 0) {
            float l = all[0][0];
            for (int q = 1; q < kConsumerWarps; ++q) l += all[q][0];
            row_loss[row] = l;
        }
    }
}

// Softmax backward on rows longer than the block-row kernels hold (MicroGPT
// softmax_backward: dx = y * (dy - sum_k y_k dy_k)): the (y, dy) chunk pairs
// stream through the ring twice, as in tma_rows2; pass 0 folds the row's dot
// product, the 16 warps add theirs in warp order, and pass 1 writes dx
// (evict-first, so the L2 keeps the rows waiting for their second pass).
// y and dy share their alignment modulo 16 bytes; dx on another phase is
// written with scalar stores.
__global__ void __launch_bounds__(kTmaThreads, 1)
tma_softmax_bwd(const float* y, const float* dy, float* dx, int64_t rows, int cols, int chunk, int nslot,
                bool dx_vec) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* buf = reinterpret_cast<float*>(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + size_t(nslot) * chunk * sizeof(float));
    uint64_t* empty = full + nslot;
    __shared__ uint64_t red_bar[2];
    __shared__ float red[2][kConsumerWarps][4];
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < nslot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(&red_bar[0], kConsumerWarps);
        mbar_init(&red_bar[1], kConsumerWarps);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) produce_pairs(y, dy, rows, cols, chunk, nslot, buf, full, empty, &abort_flag);
        return;
    }

    const int ct = tid - 32;
    const int cw = warp - 1;
    uint64_t n = 0;   // slot uses consumed
    uint32_t rv = 0;  // rendezvous so far
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* yr = y + row * int64_t(cols);
        const float* dr = dy + row * int64_t(cols);
        int head, body;
        row_split(yr, cols, head, body);
        const int nch = (body + chunk - 1) / chunk;
        int ej = -1;  // head (warp 0) and tail (warp 1) lanes, as in tma_rows
        if (ct < head) ej = ct;
        else if (ct >= 32 && ct - 32 < cols - head - body) ej = head + body + (ct - 32);
        const float ye = ej >= 0 ? __ldg(yr + ej) : 0.f;
        const float de = ej >= 0 ? __ldg(dr + ej) : 0.f;
        float dot = ye * de;
        for (int k = 0; k < nch; ++k, n += 2) {
            if (!wait_use(full, nslot, n, &abort_flag) || !wait_use(full, nslot, n + 1, &abort_flag)) return;
            const int cnt4 = min(chunk, body - k * chunk) >> 2;
            const float4* ca = reinterpret_cast<const float4*>(buf + size_t(n % nslot) * chunk);
            const float4* cb = reinterpret_cast<const float4*>(buf + size_t((n + 1) % nslot) * chunk);
            for (int i = ct; i < cnt4; i += kConsumers) {
                const float4 a = ca[i], b = cb[i];
                dot = fmaf(a.x, b.x, dot);
                dot = fmaf(a.y, b.y, dot);
                dot = fmaf(a.z, b.z, dot);
                dot = fmaf(a.w, b.w, dot);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[n % nslot]);
                mbar_arrive(&empty[(n + 1) % nslot]);
            }
        }
        dot = group_sum<32>(dot);
        float all[kConsumerWarps][4];
        const float mine[4] = {dot, 0.f, 0.f, 0.f};
        if (!rendezvous4(red, red_bar, cw, lane, rv, mine, all, &abort_flag)) return;
        float c = all[0][0];
        for (int q = 1; q < kConsumerWarps; ++q) c += all[q][0];
        float* dst = dx + row * int64_t(cols);
        if (ej >= 0) dst[ej] = ye * (de - c);
        for (int k = 0; k < nch; ++k, n += 2) {
            if (!wait_use(full, nslot, n, &abort_flag) || !wait_use(full, nslot, n + 1, &abort_flag)) return;
            const int cnt4 = min(chunk, body - k * chunk) >> 2;
            const float4* ca = reinterpret_cast<const float4*>(buf + size_t(n % nslot) * chunk);
            const float4* cb = reinterpret_cast<const float4*>(buf + size_t((n + 1) % nslot) * chunk);
            float* dk = dst + head + size_t(k) * chunk;
            for (int i = ct; i < cnt4; i += kConsumers) {
                const float4 a = ca[i], b = cb[i];
                float4 o;
                o.x = a.x * (b.x - c);
                o.y = a.y * (b.y - c);
                o.z = a.z * (b.z - c);
                o.w = a.w * (b.w - c);
                if (dx_vec) {
                    __stcs(reinterpret_cast<float4*>(dk) + i, o);
                } else {
                    __stcs(dk + 4 * i, o.x);
                    __stcs(dk + 4 * i + 1, o.y);
                    __stcs(dk + 4 * i + 2, o.z);
                    __stcs(dk + 4 * i + 3, o.w);
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[n % nslot]);
                mbar_arrive(&empty[(n + 1) % nslot]);
            }
        }
    }
}

// Two-input rows (tma_rows2): a ring of whole chunk pairs in ~192 KB.
constexpr size_t kRingBytes2 = 192 * 1024;

// Ring of the two-input kernels for rows of `cols` floats: chunk (floats),
// slots and dynamic shared memory; false when the rows do not suit them.
bool pair_ring(int64_t cols, int* chunk, int* nslot, size_t* smem) {
    if (cols < 1024 || cols > INT32_MAX / 2) return false;
    const int64_t per_row = (cols + kMaxChunk2 - 1) / kMaxChunk2;
    *chunk = int(((cols + per_row - 1) / per_row + 3) / 4 * 4);
    int64_t fit = int64_t(kRingBytes2) / (int64_t(*chunk) * 4);
    if (fit > kMaxSlots) fit = kMaxSlots;
    if (fit < 2) return false;
    *nslot = int(fit);
    *smem = size_t(*nslot) * *chunk * sizeof(float) + 2 * size_t(*nslot) * sizeof(uint64_t);
    return *smem <= kMaxDynSmem;
}

template <bool TEACHER>
bool launch_tma2(const float* x, const float* w, float* grad, float* row_loss, int64_t rows, int64_t cols,
                 float grad_scale, cudaStream_t stream, cudaError_t* err) {
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
    if ((xa & 3) != 0 || (reinterpret_cast<uintptr_t>(w) & 15) != (xa & 15)) return false;
    const bool grad_vec = grad != nullptr && (reinterpret_cast<uintptr_t>(grad) & 15) == (xa & 15);
    int chunk = 0, nslot = 0;
    size_t smem = 0;
    if (!pair_ring(cols, &chunk, &nslot, &smem)) return false;
    const int sms = sm_count();
    if (sms <= 0) return false;
    auto kern = tma_rows2<TEACHER>;
    *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (*err != cudaSuccess) return true;
    const int64_t grid = rows < sms ? rows : sms;
    kern<<<unsigned(grid), kTmaThreads, smem, stream>>>(x, w, grad, row_loss, rows, int(cols), chunk, nslot,
                                                        grad_scale, grad_vec);
    *err = cudaGetLastError();
    return true;
}

}  // namespace

bool launch_soft_ce_tma(const float* x, const float* w, float* grad, float* row_loss, int64_t rows, int64_t cols,
                        float grad_scale, cudaStream_t stream, cudaError_t* err) {
    return launch_tma2<false>(x, w, grad, row_loss, rows, cols, grad_scale, stream, err);
}

bool launch_teacher_ce_tma(const float* s, const float* t, float* grad, float* row_loss, int64_t rows,
                           int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err) {
    return launch_tma2<true>(s, t, grad, row_loss, rows, cols, grad_scale, stream, err);
}

bool launch_softmax_bwd_tma(const float* y, const float* dy, float* dx, int64_t rows, int64_t cols,
                            cudaStream_t stream, cudaError_t* err) {
    const uintptr_t ya = reinterpret_cast<uintptr_t>(y);
    if ((ya & 3) != 0 || (reinterpret_cast<uintptr_t>(dy) & 15) != (ya & 15)) return false;
    const bool dx_vec = (reinterpret_cast<uintptr_t>(dx) & 15) == (ya & 15);
    int chunk = 0, nslot = 0;
    size_t smem = 0;
    if (!pair_ring(cols, &chunk, &nslot, &smem)) return false;
    const int sms = sm_count();
    if (sms <= 0) return false;
    *err = cudaFuncSetAttribute(tma_softmax_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (*err != cudaSuccess) return true;
    const int64_t grid = rows < sms ? rows : sms;
    tma_softmax_bwd<<<unsigned(grid), kTmaThreads, smem, stream>>>(y, dy, dx, rows, int(cols), chunk, nslot,
                                                                   dx_vec);
    *err = cudaGetLastError();
    return true;
}

uint32_t pipeline_timeouts_pairs() { return read_pipeline_timeouts(); }

}  // namespace rowops
