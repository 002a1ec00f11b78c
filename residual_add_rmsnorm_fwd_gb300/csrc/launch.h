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

// Blocks of `func` with `threads` threads and `smem` dynamic shared memory
// that fit on one SM of the current device (cached per device).
int occupancy(const void *func, int threads, size_t smem);

// Small H (below 256): a warp, or an aligned group of 1..32 lanes, per row.
cudaError_t launch_fwd_small(const FwdArgs &a, int dtype, bool vec, int sm_count, cudaStream_t st);

// Row kept in registers between the sum of squares and the scale step.
bool fwd_row_fits(int H, int dtype, bool vec);
cudaError_t launch_fwd_row(const FwdArgs &a, int dtype, bool vec, int sm_count, cudaStream_t st);

// H above the register budget: two passes over the row in chunks.
cudaError_t launch_fwd_chunked(const FwdArgs &a, int dtype, bool vec, int sm_count, cudaStream_t st);

// Backward: dx per row plus per-CTA dweight partials, then the fixed-order
// column reduction of the partials.
struct BwdPlan {
    bool row;        // register-resident row kernel (else the chunked kernel)
    int threads;
    int nv;          // vectors per thread (row kernel)
    int grid;        // persistent CTAs = rows of the partial buffer
};
BwdPlan plan_bwd(int64_t M, int H, int dtype, bool vec, int sm_count);
size_t bwd_partial_bytes(const BwdPlan &p, int H);
cudaError_t launch_bwd(const BwdArgs &a, const BwdPlan &p, int dtype, bool vec, float *dweight,
                       cudaStream_t st);

}  // namespace rmsn
