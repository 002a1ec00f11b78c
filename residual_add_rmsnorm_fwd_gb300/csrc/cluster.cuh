// cluster.cuh -- thread-block cluster primitives for the split-row kernels:
// the CTA's place in its cluster, the cluster-wide barrier, stores into
// another CTA's shared memory (distributed shared memory) counted by its
// mbarrier, and a sum over every thread of a cluster that leaves the same
// binary32 total in all of them.
//
// barrier.cluster is a hardware barrier over the CTAs of one cluster, which
// the hardware schedules together; like __syncthreads it completes once
// every thread of the cluster has arrived.  The split kernels pass it twice
// (after setting up their barriers, and before exit), in every thread.
#pragma once

#include <stdint.h>

#include "bulk.cuh"
#include "common.cuh"

namespace rmsn {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t c;
    asm("mov.u32 %0, %%clusterid.x;" : "=r"(c));
    return c;
}

__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t c;
    asm("mov.u32 %0, %%nclusterid.x;" : "=r"(c));
    return c;
}

// Every thread of the cluster: this thread's earlier shared-memory writes
// become visible to the cluster's later reads (release / acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in cluster CTA `rank`'s shared memory of the variable at `local`
// in this CTA's.
__device__ __forceinline__ uint32_t cluster_map(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    return remote;
}

// Store v to another CTA's shared memory; its mbarrier (remote_bar) counts
// the 4 bytes when they have landed.
__device__ __forceinline__ void st_async_f32(uint32_t remote, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote), "f"(v),
                 "r"(remote_bar)
                 : "memory");
}

// Exchange area of the cluster sum: for two alternating reductions, an
// mbarrier and one slot per cluster rank (at most 8).
struct ClusterXchg {
    uint64_t bar[2];
    float slot[2][8];
};

// One thread initialises the exchange barriers; the caller then passes a
// cluster_sync() before the first cluster_sum, so no CTA's partial sum can
// reach a barrier that is not yet initialised.
__device__ __forceinline__ void xchg_init(ClusterXchg &xc) {
    if (threadIdx.x == 0) {
        mbar_init(&xc.bar[0], 1);
        mbar_init(&xc.bar[1], 1);
        fence_mbar_init();
    }
}

// Sum of v over every thread of the cluster, reduction number j (0, 1, 2, ...
// in every CTA), in two halves so that the caller can act in between (refill
// the stage the CTA has just copied out) while the other CTAs' sums travel.
// cluster_push: the CTA's sum (block_sum over `red`, bank j mod 2) is
// written by one thread into its own slot and pushed into slot `rank` of
// every other CTA with st.async.  cluster_total: each CTA's mbarrier j mod 2
// completes once its own arrival and the other CTAs' bytes are in, and every
// thread then adds the slots in rank order, so all threads of the cluster
// hold the bit-identical total.  No CTA waits for another to arrive
// anywhere: each waits only for the partial sums it needs.  Slots and barrier
// j mod 2 are used again by reduction j + 2, which another CTA can start only
// after this CTA has sent its partial of reduction j + 1, i.e. after it has
// read the slots of reduction j.  The wait is bounded: a wait still
// incomplete after `polls` polls records kErrPipelineTimeout in *err
// (pipe_wait); the arming thread (thread 0) waits on up to kWaitPolls so that
// it never re-arms an incomplete phase, and arms nothing more (stalled) if
// even that runs out.
__device__ __forceinline__ void cluster_push(float v, float *red, ClusterXchg &xc, uint32_t j, uint32_t rank,
                                             uint32_t cs, bool armer, const PipeWait &pw) {
    const int b = (int)(j & 1u);
    const float t = block_sum(v, red, b);
    if (armer) {
        xc.slot[b][rank] = t;
        if (!pw.stalled) {
            mbar_arrive_expect_tx(&xc.bar[b], (cs - 1) * 4u);
            for (uint32_t q = 1; q < cs; ++q) {
                const uint32_t peer = (rank + q) & (cs - 1);   // cs is 2, 4 or 8
                st_async_f32(cluster_map(&xc.slot[b][rank], peer), t, cluster_map(&xc.bar[b], peer));
            }
        }
    }
}

template <bool WAIT_CONST>
__device__ __forceinline__ float cluster_total(ClusterXchg &xc, uint32_t j, uint32_t cs, unsigned *err,
                                               uint32_t polls, bool armer, PipeWait &pw) {
    const int b = (int)(j & 1u);
    pipe_wait<WAIT_CONST>(&xc.bar[b], (j >> 1) & 1u, pw, polls, armer, err);
    float total = 0.0f;
    for (uint32_t q = 0; q < cs; ++q) total += xc.slot[b][q];
    return total;
}

template <bool WAIT_CONST>
__device__ __forceinline__ float cluster_sum(float v, float *red, ClusterXchg &xc, uint32_t j, uint32_t rank,
                                             uint32_t cs, unsigned *err, uint32_t polls, bool armer, PipeWait &pw) {
    cluster_push(v, red, xc, j, rank, cs, armer, pw);
    return cluster_total<WAIT_CONST>(xc, j, cs, err, polls, armer, pw);
}

}  // namespace rmsn
