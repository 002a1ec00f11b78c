// bulk.cuh -- the bulk-copy (TMA) pipeline primitives used by the ring
// kernels: mbarrier set-up, expect-tx, global -> shared bulk copies with
// byte-count completion, and a bounded wait.
//
// Every wait is bounded: a thread polls at most a limit of times, and a
// wait still incomplete after the call's poll limit records
// kErrPipelineTimeout in the device error word, so the kernel always ends.
// A thread whose wait has been late once polls kWaitPollsAfterTimeout times
// at most in its later waits, so a kernel whose pipeline has stalled ends
// soon instead of paying the full limit on every row.  The one thread of a
// CTA that arms a barrier (issues a stage's copies, or arms an exchange
// barrier) reports a late wait the same way but keeps waiting, up to
// kWaitPolls polls, so it never re-arms a barrier whose phase has not
// completed; if even that runs out it arms nothing more (the CTA has
// stalled).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace rmsn {

constexpr uint32_t kWaitPolls = 1u << 22;
constexpr uint32_t kWaitPollsAfterTimeout = 1u << 10;
constexpr unsigned kErrPipelineTimeout = 1u;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this CTA's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk-copy) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Poll phase `parity` of `bar` at most `limit` times; returns the number of
// polls that found it incomplete (limit: it never completed).
__device__ __forceinline__ uint32_t mbar_poll(uint64_t *bar, uint32_t parity, uint32_t limit) {
    uint32_t i = 0;
    while (i < limit && !mbar_try_wait(bar, parity)) ++i;
    return i;
}

// A thread's pipeline-wait state across a kernel.  `limit` is the polls its
// next wait may take: the call's limit, or kWaitPolls for the thread that
// arms the barriers (issues the copies, arms an exchange); after a wait has
// run out, kWaitPollsAfterTimeout, except that the arming thread keeps
// kWaitPolls until a phase never completes within it (it has then stalled).
struct PipeWait {
    uint32_t limit;
    bool late;      // a wait of this thread has been late (reported once)
    bool stalled;   // the arming thread only: a phase never completed
};

__device__ __forceinline__ PipeWait pipe_wait_init(uint32_t polls, bool armer) {
    PipeWait w;
    w.limit = armer ? kWaitPolls : polls;
    w.late = false;
    w.stalled = false;
    return w;
}

// Wait for phase `parity` of `bar`; `polls` is the call's limit (a launch
// parameter).  Two forms with the same behaviour while `polls` is
// kWaitPolls, the only value outside the time-out diagnostic:
//   CONST: until a wait has run out, poll against the constant kWaitPolls
//     (the call's limit then governs only the time-out test's held wait);
//   else:  poll against the thread's limit held in a register, and report a
//     wait still incomplete after `polls` polls while the arming thread
//     waits on.
// Which one a kernel uses is measured, not reasoned: the code around the poll
// loop shifts the scheduling of the whole row loop.  The constant form was
// 3 us faster for the bf16 H = 8192 backward and 4 us for plain LayerNorm at
// bf16 16384 x 4096; the register form 6 us faster for the f16 H = 6144
// backward and fused forward (`RING_WAIT_CONST` in the kernels).
template <bool CONST>
__device__ __forceinline__ void pipe_wait(uint64_t *bar, uint32_t parity, PipeWait &w, uint32_t polls, bool armer,
                                          unsigned *err) {
    const uint32_t short_limit = polls < kWaitPollsAfterTimeout ? polls : kWaitPollsAfterTimeout;
    if constexpr (CONST) {
        if (!w.late) {
            if (mbar_poll(bar, parity, kWaitPolls) >= kWaitPolls) {
                if (err != nullptr) atomicOr(err, kErrPipelineTimeout);
                w.late = true;
                w.stalled = armer;
            }
        } else if (mbar_poll(bar, parity, kWaitPollsAfterTimeout) >= kWaitPollsAfterTimeout) {
            w.stalled = armer;
        }
    } else {
        const uint32_t n = mbar_poll(bar, parity, w.limit);
        if (n >= polls || n >= w.limit) {
            if (!w.late && err != nullptr) atomicOr(err, kErrPipelineTimeout);
            w.late = true;
            if (!armer || n >= w.limit) {
                if (armer) w.stalled = true;
                w.limit = short_limit;
            }
        }
    }
}

// The wait form a ring or split kernel of storage type T uses (see pipe_wait).
template <typename T> struct RingWaitConst { static constexpr bool value = true; };
template <> struct RingWaitConst<__half> { static constexpr bool value = false; };

// Wait for phase `parity` of `bar` to complete, at most `polls` polls; a
// wait that runs out sets kErrPipelineTimeout in *err (when given).  Returns
// whether the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, unsigned *err,
                                                  uint32_t polls = kWaitPolls) {
    const uint32_t n = mbar_poll(bar, parity, polls);
    if (n >= polls && err != nullptr) atomicOr(err, kErrPipelineTimeout);
    return n < polls;
}

// The time-out test's wait on a barrier that nothing arms yet: it runs out
// after `polls` polls and records the time-out (out of line: it runs only
// under the test).
static __device__ __noinline__ void wait_unarmed(uint64_t *bar, unsigned *err, uint32_t polls) {
    if (mbar_poll(bar, 0, polls) >= polls && err != nullptr) atomicOr(err, kErrPipelineTimeout);
}

// Before a CTA whose issuing thread saw a wait give up exits: wait (bounded)
// for the last issued phase of each of its `nst` stage barriers, the rows
// 0 .. issued-1 having gone to stage k mod nst, so that no copy still lands
// in the CTA's shared memory after it has gone.
__device__ __forceinline__ void drain_ring(uint64_t *full, int nst, int64_t issued) {
    for (int j = 0; j < nst && j < issued; ++j) {
        const int64_t uses = (issued - 1 - j) / nst + 1;
        mbar_wait_bounded(&full[j], (uint32_t)((uses - 1) & 1), nullptr, kWaitPolls);
    }
}

}  // namespace rmsn
