// tma_rows.cu - long rows (logsumexp, softmax cross-entropy, softmax forward)
// streamed through shared memory by the Tensor Memory Accelerator.
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

constexpr int64_t kMaxChunk = 16384;       // floats per bulk copy, at most
constexpr size_t kRingBytes = 200 * 1024;   // target ring size (whole rows resident)
// Streaming ring (logsumexp).  On GB300, 8192 x 50304: 3 slots of 12576 floats
// (147 KB) ran at 0.98 of the HBM copy rate, 4 slots (one row, 196 KB) at 0.89.
constexpr size_t kStreamRingBytes = 160 * 1024;
constexpr size_t kMaxDynSmem = 226 * 1024;  // 227 KB per block, less room for static shared memory

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
    // cross-entropy and softmax it must hold a whole row.
    const int64_t per_row = (cols + kMaxChunk - 1) / kMaxChunk;
    const int chunk = int(((cols + per_row - 1) / per_row + 3) / 4 * 4);
    int64_t fit = int64_t(OP == RowOp::kLse ? kStreamRingBytes : kRingBytes) / (int64_t(chunk) * 4);
    if (fit > 8) fit = 8;
    if constexpr (OP == RowOp::kLse) {
        if (fit < 2) fit = 2;
    } else {
        if (fit < per_row) fit = per_row;  // whole row resident
    }
    const int nslot = int(fit);
    const size_t smem = size_t(nslot) * chunk * sizeof(float) + 2 * size_t(nslot) * sizeof(uint64_t);
    if (smem > kMaxDynSmem || nslot > kMaxSlots) return false;
    const int sms = sm_count();
    if (sms <= 0) return false;
    auto kern = tma_rows<OP>;
    *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (*err != cudaSuccess) return true;
    const int64_t grid = rows < sms ? rows : sms;
    kern<<<unsigned(grid), kTmaThreads, smem, stream>>>(x, out, targets, aux, rows, int(cols), chunk, nslot,
                                                         grad_scale);
    *err = cudaGetLastError();
    return true;
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

bool launch_softmax_tma(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t stream,
                        cudaError_t* err) {
    return launch_tma<RowOp::kSoftmax>(x, y, nullptr, nullptr, rows, cols, 1.f, stream, err);
}

}  // namespace rowops

extern "C" uint32_t rowops_pipeline_timeouts(void) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, rowops::g_pipeline_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    return v;
}
