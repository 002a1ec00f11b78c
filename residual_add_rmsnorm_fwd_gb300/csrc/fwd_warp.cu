// fwd_warp.cu -- RMSNorm forward (plain and AdaLN) for 16-byte aligned rows
// of 512 B to 2 KB (H = 256..1024 in 16-bit types): one warp per row.
//
// At these lengths a CTA per row spreads a row over so many threads that
// each holds only a few 16-byte groups, and the per-row work every thread
// repeats (addressing, the reduction, the CTA barrier, the rsqrt) costs as
// much as the row's arithmetic.  A warp per row gives every lane up to 32
// elements and reduces with xor shuffles alone (no shared memory, no
// barrier), so that fixed cost is paid by 32 lanes instead of 128-256
// threads and warps never wait for one another.  Measured on GB300 against
// the CTA-per-row register kernel (bf16, about 100 MB per call): H = 256,
// 4043 -> 5279 GB/s; H = 512, 5286 -> 5667; H = 1024, 5190 -> 5571, and
// AdaLN with per-sequence conditioning at H = 1024, 3931 -> 4214.  At 4 KB
// rows, for the residual-fused form (two input rows per lane) and for
// per-token conditioning it measured slower, so those stay on the register
// kernel (the kernel body handles the residual-fused form too; the host does
// not route it here).
//
// Each lane keeps its x groups packed in registers between the sum of
// squares and the scale step, so the row is read from HBM once ("Skill:
// Write a Triton RMSNorm Kernel", Required reasoning 3-10).  The weight, and AdaLN's scale
// and shift ("Rocm Kernels" page, 4. AdaLN), are read in the scale step from
// the cached path: the weight row and a per-sequence conditioning row are
// shared by many rows and stay in L1.
#include "launch.h"

namespace rmsn {

template <typename T, int NPL, int MODE, int U>
__global__ void __launch_bounds__(256) fwd_warp_kernel(FwdArgs a) {
    constexpr bool RESID = MODE == kResid;
    constexpr bool ADALN = MODE == kAdaln;
    constexpr int VEC = Vec16<T>::n;
    constexpr int PR = Pairs16<T>::n;
    using P = Pack<T, VEC>;
    // x and y (the residual and residual_out) may be one array (in-place
    // calls): not restrict
    const T *x = static_cast<const T *>(a.x);
    const T *r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    const T *__restrict__ scale = static_cast<const T *>(a.scale);
    const T *__restrict__ shift = static_cast<const T *>(a.shift);
    T *y = static_cast<T *>(a.y);
    T *s_out = static_cast<T *>(a.s_out);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);

    // U rows per warp per pass (consecutive rows); warp-uniform loop
    for (int64_t row0 = warp0 * U; row0 < a.M; row0 += nwarps * U) {
        P xp[U][NPL], rp[U][NPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t base = (row0 + u) * a.stride;
#pragma unroll
            for (int k = 0; k < NPL; ++k) {
                const int c = lane + k * 32;
                if (row0 + u < a.M && c < nvec) {
                    xp[u][k] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                    if constexpr (RESID) rp[u][k] = ld_stream<T, VEC>(r + base + (int64_t)c * VEC);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = row0 + u;
            if (row >= a.M) break;   // warp-uniform
            const int64_t base = row * a.stride;
            // s = x (+ residual) in binary32 pairs; sum of squares
            f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < NPL; ++k) {
                const int c = lane + k * 32;
                if (c < nvec) {
                    f32x2 sv[PR];
                    widen16<T>(xp[u][k], sv);
                    if constexpr (RESID) {
                        f32x2 rv[PR];
                        widen16<T>(rp[u][k], rv);
#pragma unroll
                        for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], rv[q]);
                        st_global<T, VEC>(s_out + base + (int64_t)c * VEC, narrow16<T>(sv));
                    }
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[q], sv[q], ss2);
                }
            }
            const float total = group_sum<32>(f2_sum(ss2));
            const float rrms = rsqrtf(total * ih + a.eps);
            if (lane == 0 && a.rrms != nullptr) a.rrms[row] = rrms;
            const f32x2 rr2 = f2_make(rrms, rrms);
            // row / rows_per_cond in 32 bits: both are below 2^31
            const int64_t cbase =
                ADALN ? (int64_t)((uint32_t)row / (uint32_t)a.rows_per_cond) * a.cond_stride : 0;
            // y = (s * rrms) * w [AdaLN: (s * rrms) * (w * (1 + scale)) + shift], one rounding to the storage type
#pragma unroll
            for (int k = 0; k < NPL; ++k) {
                const int c = lane + k * 32;
                if (c < nvec) {
                    f32x2 sv[PR], wv[PR];
                    widen16<T>(xp[u][k], sv);
                    if constexpr (RESID) {
                        f32x2 rv[PR];
                        widen16<T>(rp[u][k], rv);
#pragma unroll
                        for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], rv[q]);
                    }
                    widen16<T>(a.has_w ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>()), wv);
                    if constexpr (ADALN) {   // (s * rrms) * (w * (1 + scale)) + shift
                        f32x2 sc[PR], sh[PR];
                        widen16<T>(ld_cached<T, VEC>(scale + cbase + (int64_t)c * VEC), sc);
                        widen16<T>(ld_cached<T, VEC>(shift + cbase + (int64_t)c * VEC), sh);
#pragma unroll
                        for (int q = 0; q < PR; ++q)
                            sv[q] = f2_fma(f2_mul(sv[q], rr2), f2_fma(wv[q], sc[q], wv[q]), sh[q]);
                    } else {
#pragma unroll
                        for (int q = 0; q < PR; ++q) sv[q] = f2_mul(f2_mul(sv[q], rr2), wv[q]);
                    }
                    st_global<T, VEC>(y + base + (int64_t)c * VEC, narrow16<T>(sv));
                }
            }
        }
    }
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T, int NPL, int MODE, int U>
const void *kernel_ptr() {
    return reinterpret_cast<const void *>(fwd_warp_kernel<T, NPL, MODE, U>);
}

template <typename T, int NPL, int MODE, int U>
cudaError_t launch_u(const FwdArgs &a, int64_t cap_ctas, cudaStream_t st) {
    const int64_t rows_per_cta = (int64_t)kWarps * U;
    const int64_t need = (a.M + rows_per_cta - 1) / rows_per_cta;
    return launch_kernel(fwd_warp_kernel<T, NPL, MODE, U>, (unsigned)(need < cap_ctas ? need : cap_ctas),
                         kThreads, 0, st, a);
}

// Two rows per warp pass when that does not lengthen the busiest warp's
// share of rows and costs no occupancy: a row of 2 KB or less alone keeps
// few bytes in flight per warp.
template <typename T, int NPL, int MODE>
cudaError_t launch_t(const FwdArgs &a, int sm_count, cudaStream_t st) {
    const int occ = occupancy(kernel_ptr<T, NPL, MODE, 1>(), kThreads, 0);
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t cap = (int64_t)occ * sm_count;
    const int64_t warps = cap * kWarps;
    auto share = [&](int64_t u) { return ((a.M + u - 1) / u + warps - 1) / warps * u; };
    if (share(2) <= share(1) && occupancy(kernel_ptr<T, NPL, MODE, 2>(), kThreads, 0) >= occ)
        return launch_u<T, NPL, MODE, 2>(a, cap, st);
    return launch_u<T, NPL, MODE, 1>(a, cap, st);
}

template <typename T, int MODE>
cudaError_t launch_npl(const FwdArgs &a, int sm_count, cudaStream_t st) {
    const int nvec = a.H / Vec16<T>::n;
    switch ((nvec + 31) / 32) {   // rows of 512 B to 2 KB: 32..128 groups
    case 1: return launch_t<T, 1, MODE>(a, sm_count, st);
    case 2: return launch_t<T, 2, MODE>(a, sm_count, st);
    case 3: return launch_t<T, 3, MODE>(a, sm_count, st);
    case 4: return launch_t<T, 4, MODE>(a, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, int mode, int sm_count, cudaStream_t st) {
    switch (mode) {
    case kPlain: return launch_npl<T, kPlain>(a, sm_count, st);
    case kAdaln: return launch_npl<T, kAdaln>(a, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool fwd_warp_fits(int H, int dtype) {
    const int64_t row_bytes = (int64_t)H * elem_bytes(dtype);
    return row_bytes % 16 == 0 && row_bytes >= 512 && row_bytes <= 2048;
}

cudaError_t launch_fwd_warp(const FwdArgs &a, int dtype, int mode, int sm_count, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, mode, sm_count, st);
    case kF16: return launch_dt<__half>(a, mode, sm_count, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, mode, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
