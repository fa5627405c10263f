// tma_rows.cu - long rows with one input (logsumexp, softmax cross-entropy,
// softmax forward) streamed through shared memory by the Tensor Memory
// Accelerator's bulk copies, in the ring of pipeline.cuh.
//
// One persistent CTA per SM walks rows blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 0 is the producer: one lane issues bulk copies of row chunks into a
// ring of `nslot` slots.  Warps 1..16 are consumers:
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
// Cross-entropy and softmax rows too long to stay resident take tma_rows_2pass:
// two passes over each row (the second reading the L2), each row split over a
// cluster of two CTAs.  The two-input kernels are in tma_pairs.cu, the
// LayerNorm backward's row blocks in ln_bwd_tma.cu.
//
// Rows need not start on a 16-byte boundary (cols % 4 != 0, or an offset
// base): the row's first boundary splits off a head of h < 4 floats, the body
// (a multiple of 4 floats) goes through the bulk copies, and the tail of
// t < 4 floats after it is read with plain loads by consumer lanes, which also
// write the head and tail outputs.  An output row with the input row's
// alignment modulo 16 bytes takes 128-bit stores; one on another phase takes
// scalar stores (the same kernels, built for either).
//
// exp(x - m) is evaluated as 2^((x - m)*log2(e)) with the ex2.approx
// instruction.
#include <mutex>

#include "launch.h"
#include "pipeline.cuh"
#include "rowops.h"

namespace rowops {
namespace {

enum class RowOp { kLse, kCe, kSoftmax };

// Output float4 i of a chunk whose first float is dk: one 128-bit store when
// the output row shares the input row's 16-byte phase (VEC), else four.
template <bool VEC>
__device__ __forceinline__ void store4(float* dk, int i, const float4 p) {
    if constexpr (VEC) {
        reinterpret_cast<float4*>(dk)[i] = p;
    } else {
        dk[4 * i] = p.x;
        dk[4 * i + 1] = p.y;
        dk[4 * i + 2] = p.z;
        dk[4 * i + 3] = p.w;
    }
}
// The same with streaming (evict-first) stores.
template <bool VEC>
__device__ __forceinline__ void store4_cs(float* dk, int i, const float4 p) {
    if constexpr (VEC) {
        __stcs(reinterpret_cast<float4*>(dk) + i, p);
    } else {
        __stcs(dk + 4 * i, p.x);
        __stcs(dk + 4 * i + 1, p.y);
        __stcs(dk + 4 * i + 2, p.z);
        __stcs(dk + 4 * i + 3, p.w);
    }
}

template <RowOp OP, bool OUT_VEC>
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
                float* dk = dst + size_t(k) * chunk;
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
                    store4<OUT_VEC>(dk, i, p);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
        }
        n += nch;
    }
}

// ------------------------------------------------- one input, two passes
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
template <RowOp OP, int SPLIT, bool OUT_VEC>
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
                float* dk = dst + head + lo + size_t(k) * chunk;
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
                    store4_cs<OUT_VEC>(dk, i, p);  // written once, not read again: evict first
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
// Two-pass rows (see launch_tma).  On GB300, CE on 1024 x 152064 with the
// row split over two CTAs: 48 KB chunks in four slots 239 us, 64 KB in three
// 242 us, 64 KB in two (a 160 KB ring) 251 us, 32 KB in six 267 us.
constexpr int64_t kMaxChunk2p = 12288;
constexpr size_t kRing2p = 200 * 1024;

// OUT_VEC: the output rows share the input rows' 16-byte phase (128-bit
// stores); otherwise the kernels write them with scalar stores.
template <RowOp OP, bool OUT_VEC>
bool launch_tma_v(const float* x, float* out, const int32_t* targets, float* aux, int64_t rows,
                  int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err) {
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
        auto kern = tma_rows<OP, OUT_VEC>;
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
        auto kern2 = tma_rows_2pass<OP, 2, OUT_VEC>;
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
        auto kern = tma_rows_2pass<OP, 1, OUT_VEC>;
        *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (*err != cudaSuccess) return true;
        kern<<<unsigned(grid), kTmaThreads, smem, stream>>>(x, out, targets, aux, rows, int(cols), chunk, nslot,
                                                             grad_scale);
        *err = cudaGetLastError();
        return true;
    }
}

// Long rows only, 4-byte aligned buffers.
template <RowOp OP>
bool launch_tma(const float* x, float* out, const int32_t* targets, float* aux, int64_t rows,
                int64_t cols, float grad_scale, cudaStream_t stream, cudaError_t* err) {
    if (cols < 1024 || cols > INT32_MAX / 2) return false;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
    if ((xa & 3) != 0) return false;
    if constexpr (OP == RowOp::kLse) {
        return launch_tma_v<OP, true>(x, out, targets, aux, rows, cols, grad_scale, stream, err);
    } else {
        if ((reinterpret_cast<uintptr_t>(out) & 15) == (xa & 15))
            return launch_tma_v<OP, true>(x, out, targets, aux, rows, cols, grad_scale, stream, err);
        return launch_tma_v<OP, false>(x, out, targets, aux, rows, cols, grad_scale, stream, err);
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

bool launch_softmax_tma(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t stream,
                        cudaError_t* err) {
    return launch_tma<RowOp::kSoftmax>(x, y, nullptr, nullptr, rows, cols, 1.f, stream, err);
}

uint32_t pipeline_timeouts_rows() { return read_pipeline_timeouts(); }

}  // namespace rowops

extern "C" uint32_t rowops_pipeline_timeouts(void) {
    const uint32_t parts[3] = {rowops::pipeline_timeouts_rows(), rowops::pipeline_timeouts_pairs(),
                               rowops::pipeline_timeouts_ln()};
    uint32_t v = 0;
    for (uint32_t p : parts) {
        if (p == 0xffffffffu) return p;
        v += p;
    }
    return v;
}
