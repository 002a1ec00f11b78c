// launch.h -- host-side launchers of the kernel families (internal to the
// library; the public ABI is include/rmsnorm.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace rmsn {

enum Dtype { kF32 = 0, kF16 = 1, kBF16 = 2 };

inline int elem_bytes(int dtype) { return dtype == kF32 ? 4 : 2; }
inline int vec_elems(int dtype) { return 16 / elem_bytes(dtype); }

// Launch a kernel on `st` and report the launch status.  (Programmatic
// dependent launch of every kernel was measured and left out: triggered at
// kernel entry it slowed the fused forward + backward step from 0.149 to
// 0.164 ms; triggered at each CTA's end it gained nothing on the step and
// lost 11% on per-sequence AdaLN.  Only the dweight reduction is launched
// that way, after the backward.)
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                          Args... args) {
    k<<<grid, block, smem, st>>>(args...);
    return cudaGetLastError();
}

// Blocks of `func` with `threads` threads and `smem` dynamic shared memory
// that fit on one SM of the current device (cached per device).
int occupancy(const void *func, int threads, size_t smem);

// Raise a kernel's dynamic shared-memory limit to `bytes` (once per device).
cudaError_t allow_dynamic_smem(const void *func, size_t bytes);

// A ring kernel launch: NV 16-byte column groups per thread, `threads` per
// CTA, `grid` persistent CTAs, the shared-memory ring geometry.
struct RingPlan {
    int nv;
    int threads;
    int grid;
    int max_ctas_per_sm;   // 0 = as many as fit
    size_t smem_bytes;
    RingShape shape;
};

// Ring shapes measured best on GB300 (see the kernel files): false when the
// row is too short to profit from the ring or too long for it.
bool fwd_ring_geometry(int H, int dtype, int mode, RingPlan *p);
bool bwd_ring_geometry(int H, int dtype, bool dres, RingPlan *p);

// A split-row launch: a cluster of `cs` CTAs per row, each owning one
// column segment; `grid` = clusters x cs.
struct SplitPlan {
    int cs;
    int nv;
    int threads;
    int grid;
    int max_ctas_per_sm;   // 0 = as many as fit
    size_t smem_bytes;
    SplitShape shape;
};

// Split geometry for aligned rows above 32 KB (false outside 32-256 KB):
// cluster size, segment, threads, stages and shared memory, with `streams`
// input rows per ring slot.
bool split_geometry(int H, int dtype, int streams, bool backward, SplitPlan *p);
// Persistent cluster count for kernel `k` (co-resident clusters, capped by
// max_ctas_per_sm and by M); false when no cluster fits.
bool finish_split_plan(const void *k, int64_t M, int sm_count, SplitPlan *p);
// Launch `k` with cluster dimension p.cs.
cudaError_t launch_cluster(const void *k, const SplitPlan &p, void **params, cudaStream_t st);

// Forward launchers take the FwdMode (plain, residual-fused, AdaLN).
// Forward with rows staged by bulk copies (16-byte aligned rows only).
bool plan_fwd_ring(int64_t M, int H, int dtype, int mode, int sm_count, RingPlan *out);
cudaError_t launch_fwd_ring(const FwdArgs &a, int dtype, int mode, const RingPlan &p, cudaStream_t st);

// Small H (below 256): a warp, or an aligned group of 1..32 lanes, per row
// (plain and residual-fused only; a.r selects the fused form).
cudaError_t launch_fwd_small(const FwdArgs &a, int dtype, bool vec, int sm_count, cudaStream_t st);

// 16-byte aligned rows of 512 B to 2 KB, plain and AdaLN: a warp per row.
bool fwd_warp_fits(int H, int dtype);
cudaError_t launch_fwd_warp(const FwdArgs &a, int dtype, int mode, int sm_count, cudaStream_t st);

// Row kept in registers between the sum of squares and the scale step.
bool fwd_row_fits(int H, int dtype, bool vec);
cudaError_t launch_fwd_row(const FwdArgs &a, int dtype, int mode, bool vec, int sm_count, cudaStream_t st);

// Rows that are not 16-byte aligned, with x, the residual and the outputs at
// one alignment phase: the register-row kernel in each row's aligned frame
// (128-bit accesses, masked first and last vectors).
bool fwd_phase_fits(int H, int dtype);
cudaError_t launch_fwd_phase(const FwdArgs &a, int dtype, int mode, int sm_count, cudaStream_t st);
// The same rows of 4-32 KB (plain, residual-fused, LayerNorm): the bulk-copy
// ring, each row's frame staged whole.
bool plan_fwd_ring_phase(int64_t M, int H, int dtype, int mode, int sm_count, RingPlan *out);
cudaError_t launch_fwd_ring_phase(const FwdArgs &a, int dtype, int mode, const RingPlan &p, cudaStream_t st);

// Aligned rows above 32 KB: a cluster of CTAs per row, one segment each.
bool plan_fwd_split(int64_t M, int H, int dtype, int mode, int sm_count, SplitPlan *out);
cudaError_t launch_fwd_split(const FwdArgs &a, int dtype, int mode, const SplitPlan &p, cudaStream_t st);

// H above the register budget: two passes over the row in chunks.
cudaError_t launch_fwd_chunked(const FwdArgs &a, int dtype, int mode, bool vec, int sm_count, cudaStream_t st);

// Backward: dx per row plus per-CTA dweight partials, then the fixed-order
// column reduction of the partials.
enum BwdKind { kBwdRow = 0, kBwdChunked = 1, kBwdRing = 2, kBwdSplit = 3, kBwdPhase = 4, kBwdRingPhase = 5 };
struct BwdPlan {
    int kind;          // BwdKind
    bool dres;         // adds the residual stream's gradient (fused-forward backward)
    int threads;
    int nv;            // 16-byte groups (or elements) per thread (row, ring and split kernels)
    int grid;          // persistent CTAs
    int partial_rows;  // rows of the partial buffer: one per CTA, or per cluster (split)
    int cs;            // CTAs per cluster (split kernel), else 1
    size_t smem_bytes;
    RingShape ring;
    SplitShape split;
};
const void *bwd_ring_kernel_for(int dtype, int nv, bool dres);
const void *bwd_split_kernel_for(int dtype, int nv, bool dres);
// Rows that are not 16-byte aligned, with dy, x, dx (and dresidual_out) at one
// alignment phase: the register-row backward in each row's aligned frame.
bool bwd_phase_pick(int H, int dtype, int *threads, int *nv);
const void *bwd_phase_kernel_for(int dtype, int nv, bool dres);
// The same rows of 2-32 KB: the bulk-copy ring, each row's frame staged whole.
bool bwd_ring_phase_geometry(int H, int dtype, bool dres, RingPlan *p);
const void *bwd_ring_phase_kernel_for(int dtype, int nv, bool dres);
// `phased`: the rows are not 16-byte aligned but share one phase (above).
BwdPlan plan_bwd(int64_t M, int H, int dtype, bool vec, bool phased, bool dres, int sm_count);
size_t bwd_partial_bytes(const BwdPlan &p, int H);
cudaError_t launch_bwd(const BwdArgs &a, const BwdPlan &p, int dtype, bool vec, float *dweight,
                       cudaStream_t st);

}  // namespace rmsn
