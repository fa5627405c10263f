// tma_rows.cu - long rows (logsumexp, softmax cross-entropy, softmax forward,
// weighted-logits and fixed-teacher cross-entropy) streamed through shared
// memory by the Tensor Memory Accelerator's bulk copies.
//
// One persistent CTA per SM walks rows blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 0 is the producer: one lane issues bulk copies (cp.async.bulk, global ->
// shared, completion counted on an mbarrier) of row chunks into a ring of
// `nslot` slots.  Warps 1..16 are consumers:
//   phase A  waits for each chunk and folds it into a running (max, sum exp);
//            the 16 warps then merge their pairs in warp order (an mbarrier
//            rendezvous, double-buffered by row parity);
//   phase B  (cross-entropy, softmax) re-reads the chunks, still resident in
//            shared memory, writes the gradient / probabilities straight to
//            global memory and releases each slot to the producer.
// For logsumexp a slot is released right after phase A, so the ring streams
// continuously; for cross-entropy and softmax the ring holds the whole row
// (nslot * chunk >= cols), and the next row's chunks are loaded as soon as the
// current row's gradient has been written from them.  HBM sees exactly one read
// of every input element and one write of every output element.
//
// Further kernels reuse the pipeline with two passes over each row, the
// second reading the row again from the L2: tma_rows_2pass (cross-entropy and
// softmax rows too long to stay resident, each row split over a cluster of two
// CTAs), tma_rows2 (weighted-logits and fixed-teacher cross-entropy, whose two
// input rows stream as chunk pairs) and tma_softmax_bwd (softmax backward on
// long rows, (y, dy) chunk pairs).  ln_bwd_tma streams blocks of whole rows for
// the LayerNorm backward.
//
// Rows need not start on a 16-byte boundary (cols % 4 != 0, or an offset
// base): the row's first boundary splits off a head of h < 4 floats, the body
// (a multiple of 4 floats) goes through the bulk copies, and the tail of
// t < 4 floats after it is read with plain loads by consumer lanes, which also
// write the head and tail outputs.  The output row must have the same
// alignment modulo 16 bytes as the input row, so that the body's stores stay
// 128-bit.
//
// exp(x - m) is evaluated as 2^((x - m)*log2(e)) with the ex2.approx
// instruction.
//
// Every wait is bounded: a wait that runs out (which only a bug could cause)
// raises an abort flag that all waits of the CTA watch, counts one timeout in
// g_pipeline_timeouts and makes every thread leave; the producer first waits,
// again bounded, for the copies it has in flight.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "rowops.h"

namespace rowops {

__device__ unsigned int g_pipeline_timeouts;

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;
constexpr int kMaxSlots = 16;
constexpr uint32_t kSuspendNs = 100000;  // per try_wait
constexpr uint32_t kWaitPolls = 1u << 15;  // with the hint: a few seconds at most

enum class RowOp { kLse, kCe, kSoftmax };

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Tests the phase; a thread whose phase is not complete yet is suspended by the
// hardware until it completes or kSuspendNs passes, so waiting warps do not
// spin and steal issue slots from the producer.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity; false on timeout or abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < kWaitPolls; ++i) {
        if (mbar_test(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    return false;
}

__device__ __forceinline__ void bulk_load(float* dst, const float* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The same copy with an L2 eviction priority (a policy from createpolicy).
__device__ __forceinline__ void bulk_load_hint(float* dst, const float* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;\n" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policies for the two-pass kernels: the second pass and the outputs are
// marked evict-first, so the L2 keeps the first pass's lines for the second
// pass (on GB300, 1024 x 152064 CE: 277 -> 253 us; re-read bytes from 100% to
// 29% of the row; evict-last for the first pass measured the same as normal).
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}

__device__ __forceinline__ float ex2(float x) { return ex2_approx(x); }

// Running (max, sum 2^((x - max) log2 e)) over a float4.
__device__ __forceinline__ void push4(float& m, float& s, const float4 v) {
    const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mx > m) {
        s *= ex2((m - mx) * kLog2e);  // m = -inf gives 0
        m = mx;
    }
    s += ex2((v.x - m) * kLog2e) + ex2((v.y - m) * kLog2e) + ex2((v.z - m) * kLog2e) +
         ex2((v.w - m) * kLog2e);
}

// Running (max, sum) over one value (head and tail floats of a row).
__device__ __forceinline__ void push1(float& m, float& s, const float v) {
    if (v > m) {
        s *= ex2((m - v) * kLog2e);
        m = v;
    }
    s += ex2((v - m) * kLog2e);
}

// Split of a row at its first 16-byte boundary: `head` floats before it
// (0..3), then `body` floats (a multiple of 4) for the bulk copies; the
// remaining cols - head - body (0..3) floats are the tail.  `src` is 4-byte
// aligned (checked by the launcher).
__device__ __forceinline__ void row_split(const float* src, int cols, int& head, int& body) {
    const int mis = int((reinterpret_cast<uintptr_t>(src) >> 2) & 3);
    head = (4 - mis) & 3;
    if (head > cols) head = cols;
    body = (cols - head) & ~3;
}

__device__ __forceinline__ void merge2(float& m, float& s, float m2, float s2) {
    const float mm = fmaxf(m, m2);
    if (mm == -INFINITY) return;
    s = s * ex2((m - mm) * kLog2e) + s2 * ex2((m2 - mm) * kLog2e);
    m = mm;
}

__device__ void raise_abort(volatile int* abort_flag) {
    if (!*abort_flag) {
        *abort_flag = 1;
        atomicAdd(&g_pipeline_timeouts, 1u);
    }
}

template <RowOp OP>
__global__ void __launch_bounds__(kTmaThreads, 1)
tma_rows(const float* x, float* out, const int32_t* __restrict__ targets, float* __restrict__ aux,
         int64_t rows, int cols, int chunk, int nslot, float grad_scale) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* buf = reinterpret_cast<float*>(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + size_t(nslot) * chunk * sizeof(float));
    uint64_t* empty = full + nslot;
    __shared__ uint64_t red_bar[2];
    __shared__ float red[2][kConsumerWarps][2];
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if constexpr (OP == RowOp::kCe) {
        // The mean-loss kernel may be scheduled now; it waits for this grid.
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    }

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
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        uint64_t n = 0;
        bool ok = true;
        for (int64_t row = blockIdx.x; ok && row < rows; row += gridDim.x) {
            const float* src = x + row * int64_t(cols);
            int head, body;
            row_split(src, cols, head, body);
            src += head;
            const int nch = (body + chunk - 1) / chunk;
            for (int k = 0; k < nch; ++k, ++n) {
                const int s = int(n % nslot);
                const uint64_t use = n / nslot;
                if (use > 0 && !mbar_wait(&empty[s], uint32_t((use - 1) & 1), &abort_flag)) {
                    raise_abort(&abort_flag);
                    ok = false;
                    break;
                }
                const int cnt = min(chunk, body - k * chunk);
                mbar_arrive_expect_tx(&full[s], uint32_t(cnt) * 4u);
                bulk_load(buf + size_t(s) * chunk, src + size_t(k) * chunk, uint32_t(cnt) * 4u, &full[s]);
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
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ct = tid - 32;
    const int cw = warp - 1;
    uint64_t n = 0;
    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const float* src = x + row * int64_t(cols);
        int head, body;
        row_split(src, cols, head, body);
        const int nch = (body + chunk - 1) / chunk;
        // Lanes 0..head-1 of consumer warp 0 own the head floats, lanes
        // 0..tail-1 of consumer warp 1 the tail floats; `ej` is the column.
        int ej = -1;
        if (ct < head) ej = ct;
        else if (ct >= 32 && ct - 32 < cols - head - body) ej = head + body + (ct - 32);
        const float xe = ej >= 0 ? src[ej] : -INFINITY;  // coherent: softmax may run in place
        float m = -INFINITY, s = 0.f;
        if (ej >= 0) push1(m, s, xe);
        for (int k = 0; k < nch; ++k) {
            const uint64_t q = n + k;
            const int slot = int(q % nslot);
            if (!mbar_wait(&full[slot], uint32_t((q / nslot) & 1), &abort_flag)) {
                raise_abort(&abort_flag);
                return;
            }
            const int cnt4 = min(chunk, body - k * chunk) >> 2;
            const float4* c4 = reinterpret_cast<const float4*>(buf + size_t(slot) * chunk);
            for (int i = ct; i < cnt4; i += kConsumers) push4(m, s, c4[i]);
            if constexpr (OP == RowOp::kLse) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
        }
        // (max, sum) of the row: warp butterfly, then the 16 warps in order.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            merge2(m, s, __shfl_xor_sync(kFullMask, m, o), __shfl_xor_sync(kFullMask, s, o));
        const int par = it & 1;
        if (lane == 0) {
            red[par][cw][0] = m;
            red[par][cw][1] = s;
            mbar_arrive(&red_bar[par]);
        }
        if (!mbar_wait(&red_bar[par], uint32_t((it >> 1) & 1), &abort_flag)) {
            raise_abort(&abort_flag);
            return;
        }
        float M = red[par][0][0], S = red[par][0][1];
        for (int w = 1; w < kConsumerWarps; ++w) merge2(M, S, red[par][w][0], red[par][w][1]);
        const float lse = isinf(M) ? M : M + logf(S);

        if constexpr (OP == RowOp::kLse) {
            if (ct == 0) out[row] = lse;
        } else {
            const float inv = 1.0f / S;
            int t = -1;
            if constexpr (OP == RowOp::kCe) {
                t = __ldg(targets + row);
                if (ct == 0) {
                    float loss = __int_as_float(0x7fc00000);
                    if (t >= 0 && t < cols) {
                        const int tb = t - head;  // position in the body
                        if (tb >= 0 && tb < body) {
                            const uint64_t qt = n + tb / chunk;
                            loss = lse - buf[size_t(qt % nslot) * chunk + tb % chunk];
                        } else {
                            loss = lse - __ldg(src + t);
                        }
                    }
                    aux[row] = loss;
                }
            }
            float* dst = out + row * int64_t(cols);
            if (ej >= 0) {
                float p = ex2((xe - M) * kLog2e) * inv;
                if constexpr (OP == RowOp::kCe) p = grad_scale * (p - (ej == t ? 1.f : 0.f));
                dst[ej] = p;
            }
            dst += head;
            for (int k = 0; k < nch; ++k) {
                const int slot = int((n + k) % nslot);
                const int cnt4 = min(chunk, body - k * chunk) >> 2;
                const float4* c4 = reinterpret_cast<const float4*>(buf + size_t(slot) * chunk);
                float4* d4 = reinterpret_cast<float4*>(dst + size_t(k) * chunk);
                for (int i = ct; i < cnt4; i += kConsumers) {
                    const float4 v = c4[i];
                    float4 p;
                    p.x = ex2((v.x - M) * kLog2e) * inv;
                    p.y = ex2((v.y - M) * kLog2e) * inv;
                    p.z = ex2((v.z - M) * kLog2e) * inv;
                    p.w = ex2((v.w - M) * kLog2e) * inv;
                    if constexpr (OP == RowOp::kCe) {
                        const int j = head + k * chunk + 4 * i;
                        p.x = grad_scale * (p.x - (j == t ? 1.f : 0.f));
                        p.y = grad_scale * (p.y - (j + 1 == t ? 1.f : 0.f));
                        p.z = grad_scale * (p.z - (j + 2 == t ? 1.f : 0.f));
                        p.w = grad_scale * (p.w - (j + 3 == t ? 1.f : 0.f));
                    }
                    d4[i] = p;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
        }
        n += nch;
    }
}

// Bounded wait for slot use q of the ring; false (after raising the abort) on
// timeout or abort.
__device__ __forceinline__ bool wait_use(uint64_t* full, int nslot, uint64_t q, volatile int* abort_flag) {
    if (mbar_wait(&full[int(q % nslot)], uint32_t((q / nslot) & 1), abort_flag)) return true;
    raise_abort(abort_flag);
    return false;
}

// The consumer warps exchange 4 floats each through `red` (double-buffered by
// the rendezvous count rv); every warp gets all of them in `all`.
__device__ __forceinline__ bool rendezvous4(float (*red)[kConsumerWarps][4], uint64_t* red_bar, int cw, int lane,
                                           uint32_t& rv, const float (&mine)[4], float (&all)[kConsumerWarps][4],
                                           volatile int* abort_flag) {
    const int par = int(rv & 1);
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) red[par][cw][i] = mine[i];
        mbar_arrive(&red_bar[par]);
    }
    if (!mbar_wait(&red_bar[par], (rv >> 1) & 1, abort_flag)) {
        raise_abort(abort_flag);
        return false;
    }
    ++rv;
    for (int q = 0; q < kConsumerWarps; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i) all[q][i] = red[par][q][i];
    return true;
}

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

// ------------------------------------------------- one input, two passes
// Cluster helpers for the split two-pass kernel.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster (not warp-aligned).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
// Bounded wait on a barrier that another CTA of the cluster arrives on; the
// acquire makes that CTA's writes before its arrival visible.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < kWaitPolls; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
            : "memory");
        if (ok) return true;
        if (*abort_flag) return false;
    }
    return false;
}

// Cross-entropy and softmax forward on rows longer than the ring can hold
// whole: the row streams through the ring twice, pass 0 folding (max, sum)
// and pass 1 writing the gradient or probabilities; pass 1 reads from the L2
// what pass 0 brought in.  With SPLIT = 2 a cluster of two CTAs (on two SMs)
// shares each row: rank 0 takes the head and the first half of the body,
// rank 1 the rest and the tail; after pass 0 each CTA stores its (max, sum)
// into the other's shared memory and arrives on the other's barrier, and both
// merge the two pairs in rank order (the same bits in both).  A row then holds
// half as much of the L2 between its passes, so with one row per SM in flight
// the second pass finds more of it there.  Every wait is bounded; every thread
// of the cluster meets at a final cluster barrier, so neither CTA leaves while
// the other may still write into its shared memory.  Softmax may run in
// place: every chunk of pass 1 is copied into shared memory before the
// consumers overwrite it in global memory, and pass 0 of the row is over (in
// both CTAs) before pass 1 writes anything.
template <RowOp OP, int SPLIT>
__global__ void __launch_bounds__(kTmaThreads, 1)
tma_rows_2pass(const float* x, float* out, const int32_t* __restrict__ targets, float* __restrict__ aux,
               int64_t rows, int cols, int chunk, int nslot, float grad_scale) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* buf = reinterpret_cast<float*>(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + size_t(nslot) * chunk * sizeof(float));
    uint64_t* empty = full + nslot;
    __shared__ uint64_t red_bar[2];
    __shared__ float red[2][kConsumerWarps][4];
    __shared__ volatile int abort_flag;
    __shared__ uint64_t xbar[2];                // SPLIT: the other CTA's (max, sum) has arrived
    __shared__ __align__(8) float xch[2][2];    // and is here (double-buffered by row parity)

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if constexpr (OP == RowOp::kCe) {
        // The mean-loss kernel may be scheduled now; it waits for this grid.
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    }
    const int rank = SPLIT > 1 ? int(cluster_rank()) : 0;
    const int64_t unit = blockIdx.x / SPLIT;     // rows unit, unit + units, ...
    const int64_t units = gridDim.x / SPLIT;
    if (tid == 0) {
        for (int s = 0; s < nslot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(&red_bar[0], kConsumerWarps);
        mbar_init(&red_bar[1], kConsumerWarps);
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    if constexpr (SPLIT > 1) cluster_sync_all();  // the other CTA's barriers are ready

    // This CTA's part of a row: body floats [lo, hi) (multiples of 4), the
    // head (rank 0) and the tail (last rank).
    auto part = [&](int body, int& lo, int& hi) {
        const int half = ((body / SPLIT) + 3) & ~3;
        lo = rank == 0 ? 0 : (half < body ? half : body);
        hi = rank == SPLIT - 1 ? body : (half < body ? half : body);
    };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t keep = policy_evict_normal(), drop = policy_evict_first();
            uint64_t n = 0;
            bool ok = true;
            for (int64_t row = unit; ok && row < rows; row += units) {
                int head, body, lo, hi;
                row_split(x + row * int64_t(cols), cols, head, body);
                part(body, lo, hi);
                const float* src = x + row * int64_t(cols) + head + lo;
                const int len = hi - lo;
                const int nch = (len + chunk - 1) / chunk;
                for (int pass = 0; ok && pass < 2; ++pass)
                    for (int k = 0; k < nch; ++k, ++n) {
                        const uint64_t policy = pass == 0 ? keep : drop;
                        const int s = int(n % nslot);
                        const uint64_t use = n / nslot;
                        if (use > 0 && !mbar_wait(&empty[s], uint32_t((use - 1) & 1), &abort_flag)) {
                            raise_abort(&abort_flag);
                            ok = false;
                            break;
                        }
                        const int cnt = min(chunk, len - k * chunk);
                        mbar_arrive_expect_tx(&full[s], uint32_t(cnt) * 4u);
                        bulk_load_hint(buf + size_t(s) * chunk, src + size_t(k) * chunk, uint32_t(cnt) * 4u,
                                       &full[s], policy);
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
    } else {
        // ------------------------------------------------------ consumers
        const int ct = tid - 32;
        const int cw = warp - 1;
        uint64_t n = 0;   // slot uses consumed
        uint32_t rv = 0;  // rendezvous so far
        uint32_t it = 0;  // rows of this CTA so far (exchange parity)
        for (int64_t row = unit; row < rows; row += units, ++it) {
            const float* xr = x + row * int64_t(cols);
            int head, body, lo, hi;
            row_split(xr, cols, head, body);
            part(body, lo, hi);
            const int len = hi - lo;
            const int nch = (len + chunk - 1) / chunk;
            int ej = -1;  // head (warp 0 of rank 0) and tail (warp 1 of the last rank) lanes
            if (rank == 0 && ct < head) ej = ct;
            else if (rank == SPLIT - 1 && ct >= 32 && ct - 32 < cols - head - body) ej = head + body + (ct - 32);
            const float xe = ej >= 0 ? xr[ej] : -INFINITY;  // coherent: softmax may run in place
            float m = -INFINITY, s = 0.f;
            if (ej >= 0) push1(m, s, xe);
            bool ok = true;
            for (int k = 0; k < nch; ++k, ++n) {
                if (!wait_use(full, nslot, n, &abort_flag)) {
                    ok = false;
                    break;
                }
                const int cnt4 = min(chunk, len - k * chunk) >> 2;
                const float4* c4 = reinterpret_cast<const float4*>(buf + size_t(n % nslot) * chunk);
                for (int i = ct; i < cnt4; i += kConsumers) push4(m, s, c4[i]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[n % nslot]);
            }
            if (!ok) break;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                merge2(m, s, __shfl_xor_sync(kFullMask, m, o), __shfl_xor_sync(kFullMask, s, o));
            float all[kConsumerWarps][4];
            const float mine[4] = {m, s, 0.f, 0.f};
            if (!rendezvous4(red, red_bar, cw, lane, rv, mine, all, &abort_flag)) break;
            float M = all[0][0], S = all[0][1];
            for (int q = 1; q < kConsumerWarps; ++q) merge2(M, S, all[q][0], all[q][1]);
            if constexpr (SPLIT > 1) {
                const int par = int(it & 1);
                if (ct == 0) {
                    const uint32_t other = uint32_t(rank ^ 1);
                    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(map_to_rank(&xch[par][0], other)),
                                 "f"(M), "f"(S)
                                 : "memory");
                    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(
                                     map_to_rank(&xbar[par], other))
                                 : "memory");
                }
                if (!mbar_wait_cluster(&xbar[par], (it >> 1) & 1, &abort_flag)) {
                    raise_abort(&abort_flag);
                    break;
                }
                const float Mo = xch[par][0], So = xch[par][1];
                if (rank == 0) {
                    merge2(M, S, Mo, So);
                } else {
                    float M0 = Mo, S0 = So;
                    merge2(M0, S0, M, S);
                    M = M0;
                    S = S0;
                }
            }
            const float inv = 1.0f / S;
            int t = -1;
            if constexpr (OP == RowOp::kCe) {
                t = __ldg(targets + row);
                if (rank == 0 && ct == 0) {
                    const float lse = isinf(M) ? M : M + logf(S);
                    aux[row] = (t >= 0 && t < cols) ? lse - __ldg(xr + t) : __int_as_float(0x7fc00000);
                }
            }
            float* dst = out + row * int64_t(cols);
            if (ej >= 0) {
                float p = ex2((xe - M) * kLog2e) * inv;
                if constexpr (OP == RowOp::kCe) p = grad_scale * (p - (ej == t ? 1.f : 0.f));
                dst[ej] = p;
            }
            for (int k = 0; k < nch; ++k, ++n) {
                if (!wait_use(full, nslot, n, &abort_flag)) {
                    ok = false;
                    break;
                }
                const int cnt4 = min(chunk, len - k * chunk) >> 2;
                const float4* c4 = reinterpret_cast<const float4*>(buf + size_t(n % nslot) * chunk);
                float4* d4 = reinterpret_cast<float4*>(dst + head + lo + size_t(k) * chunk);
                for (int i = ct; i < cnt4; i += kConsumers) {
                    const float4 v = c4[i];
                    float4 p;
                    p.x = ex2((v.x - M) * kLog2e) * inv;
                    p.y = ex2((v.y - M) * kLog2e) * inv;
                    p.z = ex2((v.z - M) * kLog2e) * inv;
                    p.w = ex2((v.w - M) * kLog2e) * inv;
                    if constexpr (OP == RowOp::kCe) {
                        const int j = head + lo + k * chunk + 4 * i;
                        p.x = grad_scale * (p.x - (j == t ? 1.f : 0.f));
                        p.y = grad_scale * (p.y - (j + 1 == t ? 1.f : 0.f));
                        p.z = grad_scale * (p.z - (j + 2 == t ? 1.f : 0.f));
                        p.w = grad_scale * (p.w - (j + 3 == t ? 1.f : 0.f));
                    }
                    __stcs(&d4[i], p);  // written once, not read again: evict first
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[n % nslot]);
            }
            if (!ok) break;
        }
    }
    if constexpr (SPLIT > 1) cluster_sync_all();  // no CTA leaves while the other may still write to it
}

constexpr int64_t kMaxChunk = 16384;       // floats per bulk copy, at most
constexpr size_t kRingBytes = 200 * 1024;   // target ring size (whole rows resident)
// Streaming ring (logsumexp).  On GB300, 8192 x 50304: 3 slots of 12576 floats
// (147 KB) ran at 0.98 of the HBM copy rate, 4 slots (one row, 196 KB) at 0.89.
constexpr size_t kStreamRingBytes = 160 * 1024;
constexpr size_t kMaxDynSmem = 226 * 1024;  // 227 KB per block, less room for static shared memory
// Two-pass rows (see launch_tma).  On GB300, CE on 1024 x 152064 with the
// row split over two CTAs: 48 KB chunks in four slots 239 us, 64 KB in three
// 242 us, 64 KB in two (a 160 KB ring) 251 us, 32 KB in six 267 us.
constexpr int64_t kMaxChunk2p = 12288;
constexpr size_t kRing2p = 200 * 1024;
// Two-input kernel (tma_rows2): chunks of at most 12288 floats.
constexpr int64_t kMaxChunk2 = 12288;

template <RowOp OP>
bool launch_tma(const float* x, float* out, const int32_t* targets, float* aux, int64_t rows,
                int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err) {
    // Long rows only; 4-byte aligned buffers; for the ops that write rows, the
    // output row has the input row's alignment modulo 16 bytes.
    if (cols < 1024 || cols > INT32_MAX / 2) return false;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
    if ((xa & 3) != 0) return false;
    if (OP != RowOp::kLse && ((reinterpret_cast<uintptr_t>(out) & 15) != (xa & 15))) return false;
    // A row is cut into equal chunks of at most kMaxChunk floats: every chunk
    // costs the pipeline a fixed ~0.5 us per SM, so chunks are kept large (on
    // GB300, 16 KB chunks left logsumexp at 0.70 of the HBM copy rate, 48-64 KB
    // chunks reach 0.95).  The ring holds as many chunks as fit in ~200 KB; for
    // cross-entropy and softmax it holds a whole row when one fits (about 56K
// floats), and longer rows take the two-pass kernel.
    const int64_t per_row = (cols + kMaxChunk - 1) / kMaxChunk;
    const int chunk = int(((cols + per_row - 1) / per_row + 3) / 4 * 4);
    int64_t fit = int64_t(OP == RowOp::kLse ? kStreamRingBytes : kRingBytes) / (int64_t(chunk) * 4);
    if (fit > 8) fit = 8;
    if constexpr (OP == RowOp::kLse) {
        if (fit < 2) fit = 2;
    } else {
        if (fit < per_row) fit = per_row;  // whole row resident
    }
    int nslot = int(fit);
    size_t smem = size_t(nslot) * chunk * sizeof(float) + 2 * size_t(nslot) * sizeof(uint64_t);
    const int sms = sm_count();
    if (sms <= 0) return false;
    const int64_t grid = rows < sms ? rows : sms;
    if (smem <= kMaxDynSmem && nslot <= kMaxSlots) {
        auto kern = tma_rows<OP>;
        *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (*err != cudaSuccess) return true;
        kern<<<unsigned(grid), kTmaThreads, smem, stream>>>(x, out, targets, aux, rows, int(cols), chunk, nslot,
                                                             grad_scale);
        *err = cudaGetLastError();
        return true;
    }
    if constexpr (OP == RowOp::kLse) {
        return false;
    } else {
        // The row does not fit in shared memory: stream it twice (the second
        // pass reads the L2), each CTA of a cluster taking half of it, in
        // chunks of at most kMaxChunk2p floats through a ring of about kRing2p.
        const int64_t half = (cols + 1) / 2;
        const int64_t per_half = (half + kMaxChunk2p - 1) / kMaxChunk2p;
        const int chunk2 = int(((half + per_half - 1) / per_half + 3) / 4 * 4);
        fit = int64_t(kRing2p) / (int64_t(chunk2) * 4);
        if (fit > 8) fit = 8;
        if (fit < 2) fit = 2;
        nslot = int(fit);
        const int chunk = chunk2;
        smem = size_t(nslot) * chunk * sizeof(float) + 2 * size_t(nslot) * sizeof(uint64_t);
        if (smem > kMaxDynSmem) return false;
        // Two CTAs per row in clusters of two, as many clusters as can be
        // resident at once (one CTA per SM); one CTA per row if the device
        // cannot place them.
        auto kern2 = tma_rows_2pass<OP, 2>;
        *err = cudaFuncSetAttribute(kern2, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (*err != cudaSuccess) return true;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kTmaThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // Resident clusters for this shared-memory size, asked once per device
        // and size (which also keeps the query out of stream captures after
        // the first call, so captured and eager calls pick the same kernel).
        int clusters = 0;
        {
            static std::mutex mu;
            static int64_t keys[16][2];
            static int counts[16];
            static int used = 0;
            int dev = -1;
            (void)cudaGetDevice(&dev);
            std::lock_guard<std::mutex> lock(mu);
            int i = 0;
            while (i < used && !(keys[i][0] == dev && keys[i][1] == int64_t(smem))) ++i;
            if (i < used) {
                clusters = counts[i];
            } else {
                if (cudaOccupancyMaxActiveClusters(&clusters, kern2, &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();  // not fatal: fall back to one CTA per row
                    clusters = 0;
                }
                if (used < 16) {
                    keys[used][0] = dev;
                    keys[used][1] = int64_t(smem);
                    counts[used] = clusters;
                    ++used;
                }
            }
        }
        if (clusters > 0) {
            const int64_t nclu = rows < clusters ? rows : clusters;
            cfg.gridDim = dim3(unsigned(2 * nclu));
            *err = cudaLaunchKernelEx(&cfg, kern2, x, out, targets, aux, rows, int(cols), chunk, nslot,
                                      grad_scale);
            if (*err == cudaSuccess) *err = cudaGetLastError();
            return true;
        }
        auto kern = tma_rows_2pass<OP, 1>;
        *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (*err != cudaSuccess) return true;
        kern<<<unsigned(grid), kTmaThreads, smem, stream>>>(x, out, targets, aux, rows, int(cols), chunk, nslot,
                                                             grad_scale);
        *err = cudaGetLastError();
        return true;
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

// ------------------------------------------ LayerNorm backward, row blocks
// TorchLean layer-normalisation VJP / MicroGPT layer_norm_backward on rows of
// 384..1024 floats on 16-byte boundaries:
//   g' = dy*gamma, dx = r*(g' - mean(g') - xhat*mean(g'*xhat)),
//   dgamma_j = sum_i dy*xhat, dbeta_j = sum_i dy.
// One persistent CTA per SM owns a contiguous block of rows.  The producer
// copies `slot_rows` rows of dy and of xhat at a time (two bulk copies per
// slot: the rows of a block are contiguous) into the ring.  Consumer warp w
// processes the CTA's rows w, w + 16, ...; lane l owns the float4 chunks l,
// l + 32, ... of every row, so it adds its columns' dgamma and dbeta partials
// in registers across all of its rows.  A warp waits only for the slots that
// hold its rows and releases each after its last row there; slot_rows is a
// power of two and nslot a multiple of the period 16 / slot_rows (below 16
// rows), so the slots warp w touches are w / slot_rows + j * period and it
// waits on every use of each of them, in order: a parity wait never meets a
// phase two uses old.  (Making every warp visit every slot instead measured
// slower on GB300: 4096 x 768, 22.1 us against 18.1.)  A row is swept twice in shared memory (the sums of g' and
// g'*xhat, then dx), and dx goes straight to global memory.  When the rows are
// done, the 16 warps add their partials in warp order through shared memory
// (the ring, free by then) and the CTA writes its partial to workspace slot
// blockIdx.x; ln_params_reduce adds the slots in order.  HBM sees one read of
// dy and xhat and one write of dx.
constexpr int kLnTmaMaxNV = 8;                 // float4 chunks per lane: 1024 floats
constexpr size_t kLnTmaSlotBytes = 48 * 1024;  // rows of dy and xhat per slot, at most
constexpr size_t kLnTmaRingBytes = 200 * 1024;

template <int NV>
__global__ void __launch_bounds__(kTmaThreads, 1)
ln_bwd_tma(const float* __restrict__ dy, const float* __restrict__ gamma, const float* __restrict__ xhat,
           const float* __restrict__ inv_std, float* __restrict__ dx, float* __restrict__ ws, int64_t rows,
           int cols, int64_t rows_per_cta, int slot_rows, int nslot) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const size_t slot_floats = size_t(2) * slot_rows * cols;
    float* ring = reinterpret_cast<float*>(smem_raw);
    float* gs = ring + size_t(nslot) * slot_floats;  // gamma
    uint64_t* full = reinterpret_cast<uint64_t*>(gs + cols);  // cols % 4 == 0: 16-byte aligned
    uint64_t* empty = full + nslot;
    __shared__ volatile int abort_flag;

    // The dependent stage-2 kernel may be scheduled now; it waits for this grid.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t r_begin = int64_t(blockIdx.x) * rows_per_cta;
    const int64_t r_end = r_begin + rows_per_cta < rows ? r_begin + rows_per_cta : rows;
    const int64_t n_rows = r_end > r_begin ? r_end - r_begin : 0;
    const int64_t n_slots = (n_rows + slot_rows - 1) / slot_rows;
    if (tid == 0) {
        // The warps owning a full slot's rows (min(slot_rows, 16) of them)
        // each release it once.
        const uint32_t owners = uint32_t(slot_rows < kConsumerWarps ? slot_rows : kConsumerWarps);
        for (int q = 0; q < nslot; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], owners);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        int64_t k = 0;
        bool ok = true;
        for (; k < n_slots; ++k) {
            const int q = int(k % nslot);
            const int64_t use = k / nslot;
            if (use > 0 && !mbar_wait(&empty[q], uint32_t((use - 1) & 1), &abort_flag)) {
                raise_abort(&abort_flag);
                ok = false;
                break;
            }
            const int64_t r0 = r_begin + k * slot_rows;
            const int64_t nr = r_end - r0 < slot_rows ? r_end - r0 : slot_rows;
            const uint32_t bytes = uint32_t(nr) * uint32_t(cols) * 4u;
            float* dst = ring + size_t(q) * slot_floats;
            mbar_arrive_expect_tx(&full[q], 2u * bytes);
            bulk_load(dst, dy + r0 * cols, bytes, &full[q]);
            bulk_load(dst + size_t(slot_rows) * cols, xhat + r0 * cols, bytes, &full[q]);
        }
        if (!ok) {
            // Let the copies already issued land before the CTA's shared memory goes away.
            for (int64_t j = k > nslot ? k - nslot : 0; j < k; ++j) {
                volatile int never = 0;
                mbar_wait(&full[j % nslot], uint32_t((j / nslot) & 1), &never);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // gamma into shared memory while the first copies are in flight.
    const int ct = tid - 32;
    for (int i = ct; i < cols; i += kConsumers) gs[i] = __ldg(gamma + i);
    asm volatile("bar.sync 1, %0;\n" ::"r"(kConsumers) : "memory");
    const int cw = warp - 1;
    const int nc = cols >> 2;
    const float inv_cols = 1.0f / float(cols);
    const float4* g4 = reinterpret_cast<const float4*>(gs);
    float4 pg[NV], pb[NV];  // this lane's columns: dgamma and dbeta partials
#pragma unroll
    for (int u = 0; u < NV; ++u) pg[u] = pb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    int64_t waited = -1;  // the last slot this warp has waited for
    for (int64_t i = cw; i < n_rows; i += kConsumerWarps) {
        const int64_t k = i / slot_rows;
        const int q = int(k % nslot);
        if (k != waited) {
            if (!mbar_wait(&full[q], uint32_t((k / nslot) & 1), &abort_flag)) {
                raise_abort(&abort_flag);
                break;
            }
            waited = k;
        }
        {
            const int64_t row = r_begin + i;
            const float r = __ldg(inv_std + row);
            const size_t j = size_t(i - k * slot_rows);
            const float4* d4 = reinterpret_cast<const float4*>(ring + size_t(q) * slot_floats + j * cols);
            const float4* h4 =
                reinterpret_cast<const float4*>(ring + size_t(q) * slot_floats + (slot_rows + j) * cols);
            float s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int c = lane + 32 * u;
                if (c < nc) {
                    const float4 a = d4[c], h = h4[c], g = g4[c];
                    pg[u].x = fmaf(a.x, h.x, pg[u].x);
                    pg[u].y = fmaf(a.y, h.y, pg[u].y);
                    pg[u].z = fmaf(a.z, h.z, pg[u].z);
                    pg[u].w = fmaf(a.w, h.w, pg[u].w);
                    pb[u].x += a.x;
                    pb[u].y += a.y;
                    pb[u].z += a.z;
                    pb[u].w += a.w;
                    const float gx = a.x * g.x, gy = a.y * g.y, gz = a.z * g.z, gw = a.w * g.w;
                    s1 += (gx + gy) + (gz + gw);
                    s2 = fmaf(gx, h.x, s2);
                    s2 = fmaf(gy, h.y, s2);
                    s2 = fmaf(gz, h.z, s2);
                    s2 = fmaf(gw, h.w, s2);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s1 += __shfl_xor_sync(kFullMask, s1, o);
                s2 += __shfl_xor_sync(kFullMask, s2, o);
            }
            s1 *= inv_cols;
            s2 *= inv_cols;
            float4* o4 = reinterpret_cast<float4*>(dx + row * cols);
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int c = lane + 32 * u;
                if (c < nc) {
                    const float4 a = d4[c], h = h4[c], g = g4[c];
                    float4 o;
                    o.x = r * (a.x * g.x - s1 - h.x * s2);
                    o.y = r * (a.y * g.y - s1 - h.y * s2);
                    o.z = r * (a.z * g.z - s1 - h.z * s2);
                    o.w = r * (a.w * g.w - s1 - h.w * s2);
                    o4[c] = o;
                }
            }
        }
        __syncwarp();
        // The warp's last row in this slot releases it.
        if (lane == 0 && (i + kConsumerWarps) / slot_rows != k) mbar_arrive(&empty[q]);
    }
    // Warps -> CTA partial, in warp order, through the ring (every copy has
    // landed: each was waited for by the warps owning its rows).
    asm volatile("bar.sync 1, %0;\n" ::"r"(kConsumers) : "memory");
    float* red = ring;  // [16 warps][2][cols]
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = lane + 32 * u;
        if (c < nc) {
            reinterpret_cast<float4*>(red + size_t(cw) * 2 * cols)[c] = pg[u];
            reinterpret_cast<float4*>(red + (size_t(cw) * 2 + 1) * cols)[c] = pb[u];
        }
    }
    asm volatile("bar.sync 1, %0;\n" ::"r"(kConsumers) : "memory");
    for (int e = ct; e < 2 * cols; e += kConsumers) {
        float t = red[e];
        for (int w = 1; w < kConsumerWarps; ++w) t += red[size_t(w) * 2 * cols + e];
        ws[int64_t(blockIdx.x) * 2 * cols + e] = t;
    }
}
}  // namespace


bool launch_lse_tma(const float* x, float* lse, int64_t rows, int64_t cols, cudaStream_t stream,
                    cudaError_t* err) {
    return launch_tma<RowOp::kLse>(x, lse, nullptr, nullptr, rows, cols, 1.f, stream, err);
}

bool launch_ce_tma(const float* x, const int32_t* targets, float* grad, float* row_loss, int64_t rows,
                   int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err) {
    return launch_tma<RowOp::kCe>(x, grad, targets, row_loss, rows, cols, grad_scale, stream, err);
}

bool launch_soft_ce_tma(const float* x, const float* w, float* grad, float* row_loss, int64_t rows, int64_t cols,
                        float grad_scale, cudaStream_t stream, cudaError_t* err) {
    return launch_tma2<false>(x, w, grad, row_loss, rows, cols, grad_scale, stream, err);
}

bool launch_teacher_ce_tma(const float* s, const float* t, float* grad, float* row_loss, int64_t rows,
                           int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err) {
    return launch_tma2<true>(s, t, grad, row_loss, rows, cols, grad_scale, stream, err);
}

bool launch_softmax_tma(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t stream,
                        cudaError_t* err) {
    return launch_tma<RowOp::kSoftmax>(x, y, nullptr, nullptr, rows, cols, 1.f, stream, err);
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

int64_t ln_bwd_tma_ctas(int64_t rows, int64_t cols) {
    // Below 384 floats the lane-group kernel is faster (on GB300, 65536 x 256:
    // 45.7 us against 50.8; 16384 x 512: 35.5 against 32.4).
    if (cols < 384 || cols > 128 * kLnTmaMaxNV || rows <= 0) return 0;
    const int sms = sm_count();
    if (sms <= 0) return 0;
    // At most 2^17 / cols CTAs: the partials (8 * cols bytes each) of any row
    // count then stay within 1 MiB.
    int64_t g = rows < sms ? rows : sms;
    const int64_t cap = (int64_t(1) << 17) / cols;
    return g < cap ? g : cap;
}

bool launch_ln_bwd_tma(const float* dy, const float* gamma, const float* xhat, const float* inv_std, float* dx,
                       float* ws, int64_t rows, int64_t cols, cudaStream_t stream, cudaError_t* err) {
    const int64_t grid = ln_bwd_tma_ctas(rows, cols);
    if (grid <= 0 || cols % 4 != 0) return false;
    // slot_rows: a power of two; nslot: a multiple of 16 / slot_rows (see the kernel).
    int64_t slot_rows = 64;
    while (slot_rows > 1 && size_t(slot_rows) * 8 * size_t(cols) > kLnTmaSlotBytes) slot_rows >>= 1;
    const size_t slot_bytes = size_t(slot_rows) * 8 * size_t(cols);
    int64_t nslot = int64_t(kLnTmaRingBytes / slot_bytes);
    if (nslot > kMaxSlots) nslot = kMaxSlots;
    const int64_t period = slot_rows < kConsumerWarps ? kConsumerWarps / slot_rows : 1;
    nslot -= nslot % period;
    // The ring also holds the 16 warps' partials at the end.
    if (nslot < 2 || size_t(nslot) * slot_bytes < size_t(kConsumerWarps) * 8 * size_t(cols)) return false;
    const size_t smem = size_t(nslot) * slot_bytes + size_t(cols) * sizeof(float) + 2 * size_t(nslot) * sizeof(uint64_t);
    if (smem > kMaxDynSmem) return false;
    const int64_t per_cta = (rows + grid - 1) / grid;
    auto launch = [&](auto kern) {
        *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (*err != cudaSuccess) return;
        kern<<<unsigned(grid), kTmaThreads, smem, stream>>>(dy, gamma, xhat, inv_std, dx, ws, rows, int(cols),
                                                            per_cta, int(slot_rows), int(nslot));
        *err = cudaGetLastError();
    };
    switch ((cols + 127) / 128) {
        case 3: launch(ln_bwd_tma<3>); break;
        case 4: launch(ln_bwd_tma<4>); break;
        case 5: launch(ln_bwd_tma<5>); break;
        case 6: launch(ln_bwd_tma<6>); break;
        case 7: launch(ln_bwd_tma<7>); break;
        default: launch(ln_bwd_tma<8>); break;
    }
    return true;
}

}  // namespace rowops

extern "C" uint32_t rowops_pipeline_timeouts(void) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, rowops::g_pipeline_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    return v;
}
