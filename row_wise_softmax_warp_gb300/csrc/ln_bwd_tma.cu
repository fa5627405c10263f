// ln_bwd_tma.cu - LayerNorm backward stage 1 on rows of 384..1024 floats on
// 16-byte boundaries whose CTA blocks do not fit in shared memory whole
// (ln_bwd_cols in layernorm.cu takes those that do): blocks of rows streamed
// through the bulk-copy ring (pipeline.cuh); stage 2 (ln_params_reduce) is in
// layernorm.cu.
#include "launch.h"
#include "pipeline.cuh"

namespace rowops {
namespace {

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
// slower on GB300: 4096 x 768, 22.1 us against 18.1.)  A row is swept twice
// in shared memory (the sums of g' and g'*xhat, then dx), and dx goes
// straight to global memory; inv_std is loaded at the top of each row
// (loading it one row ahead measured slower).  When the rows are
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

int64_t ln_bwd_tma_ctas(int64_t rows, int64_t cols, int64_t max_ctas) {
    // Below 384 floats the lane-group kernel is faster (on GB300, 65536 x 256:
    // 45.7 us against 50.8; 16384 x 512: 35.5 against 32.4).
    if (cols < 384 || cols > 128 * kLnTmaMaxNV || rows <= 0) return 0;
    const int sms = sm_count();
    if (sms <= 0) return 0;
    // At most 2^17 / cols CTAs: on GB300, 8192 x 1024 runs in 23.7 us on 128
    // CTAs against 26.3 on 152 (16384 x 1024: 39.5 against 40.6; 8192 x 960:
    // 23.5 against 25.7; 32768 x 1024: 70.1 against 69.3), back to back.
    int64_t g = rows < sms ? rows : sms;
    const int64_t cap = (int64_t(1) << 17) / cols;
    if (g > cap) g = cap;
    if (max_ctas > 0 && g > max_ctas) g = max_ctas;
    return g;
}

bool launch_ln_bwd_tma(const float* dy, const float* gamma, const float* xhat, const float* inv_std, float* dx,
                       float* ws, int64_t rows, int64_t cols, int64_t max_ctas, cudaStream_t stream,
                       cudaError_t* err) {
    const int64_t grid = ln_bwd_tma_ctas(rows, cols, max_ctas);
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
    const size_t smem =
        size_t(nslot) * slot_bytes + size_t(cols) * sizeof(float) + 2 * size_t(nslot) * sizeof(uint64_t);
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

uint32_t pipeline_timeouts_ln() { return read_pipeline_timeouts(); }

}  // namespace rowops
