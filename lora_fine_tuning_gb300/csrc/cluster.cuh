// Wrappers for kernels whose tensor-core work spans a pair of CTAs (a
// cluster of two on neighbouring SMs): cluster rank and barrier, shared::
// cluster addressing, cluster-scope mbarrier waits and remote arrivals, TMA
// copies that signal the pair leader's barrier, and the cta_group::2 forms of
// the tcgen05 allocation, MMA and commit.  Every tcgen05 instruction with a
// cta_group qualifier in such a kernel uses cta_group::2.
#pragma once

#include "common.cuh"

namespace lora {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of both CTAs.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the variable at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// The same, suspending the thread for up to kWaitSuspendNs while the phase is open.
__device__ __forceinline__ bool mbar_try_wait_cl_sleep(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    return done != 0;
}

static __device__ __noinline__ bool mbar_wait_cl_slow(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 4; ++i)
            if (mbar_try_wait_cl_sleep(bar, parity)) return true;
        if (*w.abort) return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            if (w.status) atomicCAS(w.status, 0, w.code | site);
            return false;
        }
    }
}

// Bounded wait on a local barrier with cluster-scope acquire (it may have
// received arrivals or transaction bytes from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cl(a, parity)) return true;
    return mbar_wait_cl_slow(a, parity, w, site);
}

static __device__ __noinline__ bool mbar_wait_cl_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_cl_sleep(a, parity))
        if (global_timer_ns() - t0 > limit_ns) return false;
    return true;
}

// Arrive on a barrier given by its shared::cluster address (possibly the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA into this CTA's shared memory, completing transaction bytes on a barrier
// that may live in the peer CTA (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Issued by the pair leader: D (both CTAs' TMEM) (+)= A (both CTAs' smem, M = 256)
// * B (each CTA holds half of the N columns).
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at this offset in every CTA of `mask` when the
// leader's tcgen05.mma issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// Bulk tensor store shared -> global (clipped at the tensor's edges), tracked
// in the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a flag over the `count` participating threads:
// every thread gets the same answer, so they can all take the same branch.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool flag) {
    uint32_t r;
    asm volatile(
        "{\n"
        ".reg .pred p, q;\n"
        "setp.ne.u32 q, %3, 0;\n"
        "barrier.red.or.pred p, %1, %2, q;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(r)
        : "r"(id), "r"(count), "r"(static_cast<uint32_t>(flag))
        : "memory");
    return r != 0;
}

}  // namespace lora
