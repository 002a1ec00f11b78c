// fwd_small.cu -- RMSNorm forward (plain and residual-fused) for small hidden
// sizes (H below 256), such as the per-head norm at H = 64.
//
// A whole CTA per row would leave most threads idle and pay a CTA-wide
// barrier per row, so each row is handled by an aligned group of LANES lanes
// of one warp (LANES = 1..32, the smallest power of two covering the row's
// 128-bit vectors, or its elements on the scalar path).  A warp processes
// 32 / LANES rows at a time and reduces each row with xor shuffles that stay
// inside its lane group: no shared memory, no barrier.  (The page advises
// warp-level reductions for hidden sizes below 256: "Skill: Write a Triton
// RMSNorm Kernel", Do not use this when, third bullet.)  Each lane group
// takes U consecutive row slots per pass and issues all their loads before
// any arithmetic, so U 16-byte loads per lane are in flight at once: with a
// 128-byte row, one row per lane group would leave HBM under-occupied.
#include "launch.h"

namespace rmsn {

template <typename T, int VEC, int LANES, int NPL, bool RESID, int U>
__global__ void __launch_bounds__(256) fwd_small_kernel(FwdArgs a) {
    using P = Pack<T, VEC>;
    constexpr int RPW = 32 / LANES;  // rows per warp per slot
    // x and y (the residual and residual_out) may be one array (in-place
    // calls): not restrict
    const T *x = static_cast<const T *>(a.x);
    const T *r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *y = static_cast<T *>(a.y);
    T *s_out = static_cast<T *>(a.s_out);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H
    const int lane = threadIdx.x & 31;
    const int slot = lane / LANES;   // which of the warp's rows
    const int li = lane % LANES;     // lane within the row's group

    P wp[NPL];
#pragma unroll
    for (int k = 0; k < NPL; ++k) {
        const int c = li + k * LANES;
        wp[k] = (a.has_w && c < nvec) ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
    }

    const int64_t warps_per_grid = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    constexpr int ROWS = RPW * U;    // rows per warp per pass
    // warp-uniform loop: every lane takes part in the shuffles
    for (int64_t row0 = warp_id * ROWS; row0 < a.M; row0 += warps_per_grid * ROWS) {
        P xp[U][NPL], rp[U][NPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = row0 + u * RPW + slot;
            const int64_t base = row * a.stride;
#pragma unroll
            for (int k = 0; k < NPL; ++k) {
                const int c = li + k * LANES;
                if (row < a.M && c < nvec) {
                    xp[u][k] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                    if constexpr (RESID) rp[u][k] = ld_stream<T, VEC>(r + base + (int64_t)c * VEC);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = row0 + u * RPW + slot;
            const bool live = row < a.M;
            const int64_t base = row * a.stride;
            float ss = 0.0f;
            f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < NPL; ++k) {
                const int c = li + k * LANES;
                if (live && c < nvec) {
                    if constexpr (VEC > 1) {   // binary32 pairs, two lanes per instruction
                        f32x2 sv[VEC / 2];
                        widen16<T>(xp[u][k], sv);
                        if constexpr (RESID) {
                            f32x2 rv[VEC / 2];
                            widen16<T>(rp[u][k], rv);
#pragma unroll
                            for (int q = 0; q < VEC / 2; ++q) sv[q] = f2_add(sv[q], rv[q]);
                            st_global<T, VEC>(s_out + base + (int64_t)c * VEC, narrow16<T>(sv));
                        }
#pragma unroll
                        for (int q = 0; q < VEC / 2; ++q) ss2 = f2_fma(sv[q], sv[q], ss2);
                    } else {
                        float v = to_f32(xp[u][k].v[0]);
                        if constexpr (RESID) {
                            v += to_f32(rp[u][k].v[0]);
                            s_out[base + c] = from_f32<T>(v);
                        }
                        ss += v * v;
                    }
                }
            }
            if constexpr (VEC > 1) ss = f2_sum(ss2);
            const float total = group_sum<LANES>(ss);
            const float rrms = rsqrtf(total * ih + a.eps);
            if (live && li == 0 && a.rrms != nullptr) a.rrms[row] = rrms;
            const f32x2 rr2 = f2_make(rrms, rrms);
#pragma unroll
            for (int k = 0; k < NPL; ++k) {
                const int c = li + k * LANES;
                if (live && c < nvec) {
                    if constexpr (VEC > 1) {
                        f32x2 sv[VEC / 2], wv[VEC / 2];
                        widen16<T>(xp[u][k], sv);
                        if constexpr (RESID) {
                            f32x2 rv[VEC / 2];
                            widen16<T>(rp[u][k], rv);
#pragma unroll
                            for (int q = 0; q < VEC / 2; ++q) sv[q] = f2_add(sv[q], rv[q]);
                        }
                        widen16<T>(wp[k], wv);
#pragma unroll
                        for (int q = 0; q < VEC / 2; ++q) sv[q] = f2_mul(f2_mul(sv[q], rr2), wv[q]);
                        st_global<T, VEC>(y + base + (int64_t)c * VEC, narrow16<T>(sv));
                    } else {
                        float v = to_f32(xp[u][k].v[0]);
                        if constexpr (RESID) v += to_f32(rp[u][k].v[0]);
                        y[base + c] = from_f32<T>((v * rrms) * to_f32(wp[k].v[0]));
                    }
                }
            }
        }
    }
}

namespace {

constexpr int kThreads = 256;

template <typename T, int VEC, int LANES, int NPL, bool RESID, int U>
int64_t resident_ctas(int sm_count) {
    return (int64_t)occupancy(reinterpret_cast<const void *>(fwd_small_kernel<T, VEC, LANES, NPL, RESID, U>),
                              kThreads, 0) * sm_count;
}

template <typename T, int VEC, int LANES, int NPL, bool RESID, int U>
cudaError_t launch_u(const FwdArgs &a, int sm_count, cudaStream_t st) {
    const int64_t cap = resident_ctas<T, VEC, LANES, NPL, RESID, U>(sm_count);
    if (cap <= 0) return cudaErrorInvalidConfiguration;
    constexpr int rows_per_cta = (kThreads / 32) * (32 / LANES) * U;
    const int64_t need = (a.M + rows_per_cta - 1) / rows_per_cta;
    return launch_kernel(fwd_small_kernel<T, VEC, LANES, NPL, RESID, U>, (unsigned)(need < cap ? need : cap),
                         kThreads, 0, st, a);
}

// Row slots per lane group per pass, U in {1, 2, 4} (at most four 16-byte
// loads per lane in flight): the largest U that does not lengthen the
// busiest warp's share of rows.  Warps work independently, so the share is
// counted in warp passes: 393216 rows of 64 bf16 with four rows per warp
// pass over 9728 warps is 10.1 passes with U = 1 (11 rows of work per lane
// group) against 2.53 with U = 4 (12).
template <typename T, int VEC, int LANES, int NPL, bool RESID>
cudaError_t launch_t(const FwdArgs &a, int sm_count, cudaStream_t st) {
    constexpr int RPW = 32 / LANES;
    auto share = [&](int64_t u, int64_t ctas) {
        const int64_t warps = ctas * (kThreads / 32);
        const int64_t passes = (a.M + RPW * u - 1) / (RPW * u);
        return warps > 0 ? (passes + warps - 1) / warps * u : INT64_MAX;
    };
    const int64_t s1 = share(1, resident_ctas<T, VEC, LANES, NPL, RESID, 1>(sm_count));
    if (NPL == 1 && share(4, resident_ctas<T, VEC, LANES, NPL, RESID, 4>(sm_count)) <= s1)
        return launch_u<T, VEC, LANES, NPL, RESID, 4>(a, sm_count, st);
    if (NPL <= 2 && share(2, resident_ctas<T, VEC, LANES, NPL, RESID, 2>(sm_count)) <= s1)
        return launch_u<T, VEC, LANES, NPL, RESID, 2>(a, sm_count, st);
    return launch_u<T, VEC, LANES, NPL, RESID, 1>(a, sm_count, st);
}

template <typename T, int VEC, bool RESID>
cudaError_t launch_shape(const FwdArgs &a, int n, int sm_count, cudaStream_t st) {
    // n = vectors (or elements) per row, 1..255
    if (n <= 1) return launch_t<T, VEC, 1, 1, RESID>(a, sm_count, st);
    if (n <= 2) return launch_t<T, VEC, 2, 1, RESID>(a, sm_count, st);
    if (n <= 4) return launch_t<T, VEC, 4, 1, RESID>(a, sm_count, st);
    if (n <= 8) return launch_t<T, VEC, 8, 1, RESID>(a, sm_count, st);
    if (n <= 16) return launch_t<T, VEC, 16, 1, RESID>(a, sm_count, st);
    if (n <= 32) return launch_t<T, VEC, 32, 1, RESID>(a, sm_count, st);
    if (n <= 64) return launch_t<T, VEC, 32, 2, RESID>(a, sm_count, st);
    if constexpr (VEC == 1) {
        if (n <= 128) return launch_t<T, 1, 32, 4, RESID>(a, sm_count, st);
        if (n <= 256) return launch_t<T, 1, 32, 8, RESID>(a, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, bool vec, int sm_count, cudaStream_t st) {
    constexpr int V = Vec16<T>::n;
    const bool resid = a.r != nullptr;
    if (vec) {
        const int n = a.H / V;
        return resid ? launch_shape<T, V, true>(a, n, sm_count, st)
                     : launch_shape<T, V, false>(a, n, sm_count, st);
    }
    return resid ? launch_shape<T, 1, true>(a, a.H, sm_count, st)
                 : launch_shape<T, 1, false>(a, a.H, sm_count, st);
}

}  // namespace

cudaError_t launch_fwd_small(const FwdArgs &a, int dtype, bool vec, int sm_count, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, vec, sm_count, st);
    case kF16: return launch_dt<__half>(a, vec, sm_count, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, vec, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
