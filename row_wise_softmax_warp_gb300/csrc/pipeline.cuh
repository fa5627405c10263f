// pipeline.cuh - the bulk-copy (TMA) ring shared by the long-row kernels.
//
// One persistent CTA per SM: warp 0 is the producer (one lane issues
// cp.async.bulk copies, global -> shared, completion counted on an mbarrier)
// and warps 1..16 are consumers.  This header holds the pieces every such
// kernel uses: the mbarrier and bulk-copy wrappers, the bounded waits, the
// running (max, sum exp) folds, the split of a row at its first 16-byte
// boundary, the consumer warps' rendezvous and the cluster helpers.
//
// Every wait is bounded: a wait that runs out (which only a bug could cause)
// raises an abort flag that all waits of the CTA watch and counts one timeout
// in the including translation unit's g_pipeline_timeouts (each unit has its
// own; rowops_pipeline_timeouts adds them up).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace rowops {
namespace {

__device__ unsigned int g_pipeline_timeouts;

// Host: this translation unit's timeout count (0xffffffff if unreadable).
inline uint32_t read_pipeline_timeouts() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pipeline_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    return v;
}

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;
constexpr int kMaxSlots = 16;
constexpr uint32_t kSuspendNs = 100000;  // per try_wait
constexpr uint32_t kWaitPolls = 1u << 15;  // with the hint: a few seconds at most

constexpr size_t kMaxDynSmem = 226 * 1024;  // 227 KB per block, less room for static shared memory

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

}  // namespace
}  // namespace rowops
