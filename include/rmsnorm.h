/*
 * rmsnorm.h -- C ABI of librmsnorm_gb300.so, an RMSNorm engine for GB300
 * (sm_103a).  All compute runs in the library's own CUDA kernels; the
 * library allocates no memory and keeps no state besides a per-device cache
 * of launch limits.
 *
 * The operation ("Skill: Write a Triton RMSNorm Kernel", ahel.ai, Purpose):
 *   y = x * rsqrt(mean(x^2 over the trailing dimension H) + eps) * weight
 * for each of M rows, with
 *   - the mean taken over the full row length H and eps inside the square
 *     root (Required reasoning 5-6; Correctness requirements),
 *   - a per-feature weight of shape (H,) indexed by column only and no bias
 *     (Required reasoning 7; Kernel design rules),
 *   - apply order y = (x_f32 * rrms) * w_f32 with one final rounding to the
 *     storage type (Required reasoning 8),
 *   - an optional weight: has_weight == 0 gives y = x * rrms, bit-identical
 *     to a weight of ones (the weightless norm instances of the "Rocm
 *     Kernels" page, section "Core Kernel Implementations / 1. RMSNorm").
 *
 * Common conventions for every entry point:
 *   - Pointers are device pointers owned by the caller; nothing is retained
 *     after the call returns.
 *   - A matrix argument holds M rows of H elements; element (i, h) is at
 *     index i * row_stride + h (in elements of the storage dtype).  Every
 *     matrix argument of one call shares row_stride, and row_stride >= H.
 *     Padding columns h in [H, row_stride) are never read or written.
 *   - dtype is the storage type of x, residual, weight, y, residual_out, dy
 *     and dx (rmsn_dtype).  Arithmetic is binary32; every stored result is
 *     rounded to nearest, ties to even.  rrms and dweight are binary32.
 *   - Every pointer must be aligned to its element size.  Rows whose byte
 *     offsets and lengths are multiples of 16 use 128-bit accesses.  Rows
 *     that are not (an odd H, a stride or a view that is not a multiple of 16
 *     bytes) still use 128-bit accesses, in each row's own 16-byte-aligned
 *     frame with its first and last vectors masked, when the row matrices of
 *     the call (x, residual, y, residual_out; dy, x, dx, dresidual_out)
 *     start at the same offset modulo 16 bytes; those kernels read (never
 *     write) the bytes that share a 16-byte granule with a row's first or
 *     last element.  Other layouts run a scalar-access variant of the same
 *     kernels (on the GPU).
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work and return; errors raised while the kernels run
 *     surface at the caller's next synchronisation.
 *   - All arguments are validated before anything is launched.  An invalid
 *     call returns a nonzero rmsn_status and launches nothing.  M == 0 is a
 *     valid no-op (row pointers and rrms may then be NULL).
 *   - An output may not overlap any other argument (byte ranges of the rows
 *     [0, M) are compared; RMSN_ERR_ALIAS), except in place: y may be x
 *     itself, residual_out the residual itself, and dx may be dy, x or
 *     dresidual_out itself (the same pointer; every element is read before
 *     its thread writes it, and a row's reduction completes before any of
 *     the row is written).  Partial overlaps are always rejected.
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RMSN_F32 = 0,
    RMSN_F16 = 1,  /* IEEE binary16 */
    RMSN_BF16 = 2  /* bfloat16 */
} rmsn_dtype;

typedef enum {
    RMSN_OK = 0,
    RMSN_ERR_INVALID = 1,     /* NULL required pointer, M < 0, H <= 0, row_stride < H,
                                 eps < 0 or not finite, unknown dtype, misaligned pointer */
    RMSN_ERR_ALIAS = 2,       /* an output overlaps another argument */
    RMSN_ERR_WORKSPACE = 3,   /* backward workspace missing, misaligned or too small */
    RMSN_ERR_CUDA = 4,        /* a CUDA runtime call or a kernel launch failed */
    RMSN_ERR_UNSUPPORTED = 5  /* no usable sm_103 device is current */
} rmsn_status;

/*
 * Forward.  ("Skill: Write a Triton RMSNorm Kernel": Purpose; Required
 * reasoning 1-10.)
 *   x       in   M x H, row_stride
 *   weight  in   H elements; ignored (may be NULL) when has_weight == 0
 *   y       out  M x H, row_stride
 *   rrms    out  M binary32 values 1/sqrt(mean(x^2) + eps), the statistic the
 *                backward reads (Required reasoning 10); NULL = not saved
 *   eps     >= 0 and finite.  eps == 0 is accepted: a row of zeros then
 *           yields NaN.
 * Returns RMSN_OK or an rmsn_status error code.
 */
int rmsnorm_fwd(const void *x, const void *weight, void *y, float *rrms,
                int64_t row_stride, int64_t M, int64_t H, float eps,
                int dtype, int has_weight, void *stream);

/*
 * Forward with the residual add fused in front of the norm.  ("Skill: Write
 * a Triton RMSNorm Kernel": Use this when, third bullet; Inputs 7; Kernel
 * design rules, fused residual.)
 *   s = x + residual is formed in binary32 before squaring;
 *   residual_out = s rounded to dtype (the next block's residual stream);
 *   y = norm(s) * weight, normalising the unrounded binary32 s.
 *   x, residual   in   M x H, row_stride
 *   weight        in   H elements; ignored when has_weight == 0
 *   y             out  M x H, row_stride
 *   residual_out  out  M x H, row_stride
 *   rrms          out  M binary32 values (NULL = not saved)
 * The backward of this call is rmsnorm_bwd with x := residual_out; its dx
 * is the gradient for both x and residual.
 */
int rmsnorm_fwd_residual(const void *x, const void *residual, const void *weight,
                         void *y, void *residual_out, float *rrms,
                         int64_t row_stride, int64_t M, int64_t H, float eps,
                         int dtype, int has_weight, void *stream);

/*
 * AdaLN forward: the norm followed by the DiT block's adaptive conditioning,
 * in one pass ("Rocm Kernels" page, 4. AdaLN, and its Kernel-Specific
 * Guidelines, AdaLN):
 *   y = (x * rrms) * weight * (1 + scale) + shift
 * with rrms as in rmsnorm_fwd, every step in binary32 and one rounding of y
 * to the storage type.  Row i reads conditioning row c = i / rows_per_cond
 * (integer division) of scale and shift:
 *   - rows_per_cond == 1: per-token conditioning, scale and shift of shape
 *     [batch, seq, H] flattened to M rows;
 *   - rows_per_cond == seq: one conditioning row per sequence, scale and
 *     shift of shape [batch, 1, H] broadcast over the sequence's rows (the
 *     second shape the page accepts; rows of one sequence are consecutive).
 *   x             in   M x H, row_stride
 *   weight        in   H elements; ignored when has_weight == 0
 *   scale, shift  in   ceil(M / rows_per_cond) x H, cond_stride >= H
 *   y             out  M x H, row_stride (may be x itself)
 *   rrms          out  M binary32 values (NULL = not saved)
 *   rows_per_cond >= 1.  128-bit accesses additionally need cond_stride
 *   times the element size a multiple of 16 and 16-byte aligned scale and
 *   shift.  No backward is provided for this call.
 */
int rmsnorm_adaln_fwd(const void *x, const void *weight, const void *scale, const void *shift,
                      void *y, float *rrms, int64_t row_stride, int64_t cond_stride,
                      int64_t rows_per_cond, int64_t M, int64_t H, float eps,
                      int dtype, int has_weight, void *stream);

/*
 * Residual + LayerNorm forward.  (The devpost "SpeedROCm" page, How the
 * solution addresses the problem, item 4: each residual add fused with the
 * LayerNorm that consumes it.  The pages print no LayerNorm formula; this is
 * the textbook one, with the mean subtraction the RMSNorm skill page
 * contrasts RMSNorm with, Do not use this when, second bullet.)  Per row:
 *   s = x (+ residual), binary32; residual_out = s rounded to dtype
 *   mean = sum(s) / H;  var = sum((s - mean)^2) / H  (biased; the centred
 *     sum comes from the row held on chip, or from a re-read of rows longer
 *     than the register and shared-memory budget)
 *   rstd = 1 / sqrt(var + eps);  y = ((s - mean) * rstd) * weight + bias
 *   x, residual   in   M x H, row_stride (residual: fused form only)
 *   weight, bias  in   H elements each; ignored (may be NULL) when
 *                      has_weight / has_bias == 0 (weight 1, bias 0)
 *   y             out  M x H, row_stride (may be x itself)
 *   residual_out  out  M x H, row_stride (fused form; may be the residual)
 *   mean, rstd    out  M binary32 values each, or NULL
 * No backward is provided for these calls.
 */
int layernorm_fwd(const void *x, const void *weight, const void *bias, void *y,
                  float *mean, float *rstd, int64_t row_stride, int64_t M, int64_t H,
                  float eps, int dtype, int has_weight, int has_bias, void *stream);
int layernorm_fwd_residual(const void *x, const void *residual, const void *weight,
                           const void *bias, void *y, void *residual_out, float *mean,
                           float *rstd, int64_t row_stride, int64_t M, int64_t H, float eps,
                           int dtype, int has_weight, int has_bias, void *stream);

/*
 * Size in bytes of the workspace rmsnorm_bwd (and rmsnorm_bwd_residual)
 * needs for (M, H, dtype) on the current device: binary32 dweight partials,
 * one row of H per persistent CTA, or per cluster of CTAs for aligned rows of
 * 32-256 KB; the largest over the layouts and the two entry points.  Writes
 * *bytes; the value is fixed for a given device, M, H and dtype.  0 means no
 * workspace is needed.
 */
int rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H, int dtype, size_t *bytes);

/*
 * Backward.  ("Skill: Write a Triton RMSNorm Kernel": Required reasoning 12;
 * Correctness requirements on the saved rrms and the dweight axis.)
 * With g = dy * w and xhat = x * rrms (w = 1 when has_weight == 0):
 *   dx_h      = rrms * (g_h - xhat_h * (1/H) * sum_k g_k * xhat_k)
 *   dweight_h = sum over rows i of dy_ih * xhat_ih
 *   dy         in   M x H, row_stride
 *   x          in   M x H, row_stride: the forward's normalised input
 *                   (residual_out for the residual-fused forward)
 *   weight     in   H elements; ignored when has_weight == 0
 *   rrms       in   M binary32 values saved by the forward (not recomputed)
 *   dx         out  M x H, row_stride
 *   dweight    out  H binary32 values, or NULL to skip it; ignored when
 *                   has_weight == 0.  Deterministic: per-CTA (or per-cluster)
 *                   partial sums over a fixed row assignment, then a
 *                   fixed-order column sum, so repeated calls on one device
 *                   give identical bits.
 *   workspace  scratch of at least rmsnorm_bwd_workspace_bytes(M, H, dtype)
 *              bytes, 16-byte aligned; needed only when dweight is computed
 *              (may be NULL otherwise).  Contents on entry are ignored.
 */
int rmsnorm_bwd(const void *dy, const void *x, const void *weight, const float *rrms,
                void *dx, float *dweight, void *workspace, size_t workspace_bytes,
                int64_t row_stride, int64_t M, int64_t H,
                int dtype, int has_weight, void *stream);

/*
 * Backward of rmsnorm_fwd_residual when residual_out also feeds later
 * layers.  (The RMSNorm skill page, Use this when, third bullet: the
 * post-add sum is written back as the next block's residual stream; the
 * pages leave its backward implicit.)  s = x + residual feeds both y and
 * residual_out, so
 *   ds = (rmsnorm_bwd's dx for dy) + dresidual_out,
 * computed in the same pass (one read of dresidual_out instead of a separate
 * add kernel); ds is the gradient of x and of residual alike.
 *   dy             in   M x H, row_stride: gradient of y
 *   dresidual_out  in   M x H, row_stride: gradient arriving through residual_out
 *   x              in   M x H, row_stride: the forward's residual_out
 *   weight, rrms, dweight, workspace: as for rmsnorm_bwd (dresidual_out does
 *   not reach dweight); the workspace size from rmsnorm_bwd_workspace_bytes
 *   covers this call too.
 *   dx             out  M x H, row_stride: ds
 */
int rmsnorm_bwd_residual(const void *dy, const void *dresidual_out, const void *x, const void *weight,
                         const float *rrms, void *dx, float *dweight, void *workspace,
                         size_t workspace_bytes, int64_t row_stride, int64_t M, int64_t H,
                         int dtype, int has_weight, void *stream);

/*
 * Backward for callers that cannot allocate device memory.  No counterpart
 * on the pages: it exists for callers such as serving engines that reserve
 * all device memory at start-up and forbid allocation afterwards, plugin
 * interfaces that give an operator only its inputs and outputs, and hot
 * paths where a cudaMalloc (which can synchronise the device) is not
 * acceptable.  Same arguments, results and errors as rmsnorm_bwd without the
 * workspace: the dweight partials live in a fixed 16 MiB array in the
 * library's device memory (held on every GPU that loads the library until
 * the process exits).  The call allocates nothing.
 *   - A shape whose partials, for the kernel the call selects, exceed 16 MiB
 *     is rejected with RMSN_ERR_WORKSPACE before any launch
 *     (rmsnorm_bwd_workspace_bytes, the largest over every layout, bounds
 *     them from above).
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.
 *   - All calls share the array.  Calls whose kernels may overlap on the GPU
 *     (different streams with no ordering between them) race on it; order
 *     them on one stream.
 */
int rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *weight, const float *rrms,
                        void *dx, float *dweight,
                        int64_t row_stride, int64_t M, int64_t H,
                        int dtype, int has_weight, void *stream);

/*
 * Device-side error flags of the current device, read and cleared.
 * Synchronises the device first.  Bit 0 (RMSN_DEVERR_PIPELINE_TIMEOUT): a
 * kernel's bounded wait for its bulk (TMA) row copies gave up; the outputs
 * of the calls since the last read are then unreliable.  The kernels never
 * hang on such a wait: they record the flag and finish.
 */
#define RMSN_DEVERR_PIPELINE_TIMEOUT 1u
int rmsnorm_read_device_errors(unsigned *flags);

/*
 * Diagnostic of the failure path above, for tests of a caller's failure
 * detection; not for production calls.  No counterpart on the pages.  Until
 * it is called again with (0, 0), every later call of this process:
 *   - bounds the waits below by `polls` polls (1 .. 2^22) instead of 2^22:
 *     the held wait (next item) always, and in the kernels that take their
 *     wait limit from the call (binary16 storage) every wait of threads
 *     other than the one per CTA that issues the copies, which still waits
 *     on up to 2^22 polls, so no copy is left in flight and no barrier is
 *     re-armed early;
 *   - with hold_first_copy == 1, makes the issuing thread of every CTA of
 *     the bulk-copy ring kernels (16-byte aligned rows of 4-32 KB for the
 *     plain, LayerNorm and shared-conditioning AdaLN forwards, 8-32 KB for
 *     the residual-fused and per-token AdaLN forwards, 2-32 KB for the
 *     backwards, and their aligned-frame variants for rows that are not
 *     16-byte aligned) wait for its first row before it has issued any copy, so
 *     that wait runs out on purpose and sets RMSN_DEVERR_PIPELINE_TIMEOUT;
 *     the kernel then issues its copies and finishes.
 * Outputs of calls made under these settings are unreliable.  The settings
 * are process-wide, not per device or stream.  Returns RMSN_ERR_INVALID for
 * polls > 2^22, for polls == 0 with hold_first_copy != 0, or for
 * hold_first_copy outside {0, 1}.
 */
int rmsnorm_debug_pipeline_timeout(unsigned polls, int hold_first_copy);

/* Static, human-readable text for a status code (never NULL). */
const char *rmsnorm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
