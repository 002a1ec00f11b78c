// fwd_row.cu -- RMSNorm forward (plain, residual-fused, AdaLN) and
// LayerNorm forward for hidden sizes whose row fits in the registers of one
// CTA: the general path for rows the warp and ring kernels do not take
// (unaligned layouts, AdaLN and LayerNorm below H = 256, fused rows of 2-8
// KB).
//
// One CTA per row, persistent: the grid holds as many CTAs as fit on the
// device and each CTA strides over rows.  A thread owns NV fixed column
// groups of VEC elements (128-bit accesses when the layout allows, else
// single elements), so the weight is loaded into registers once per CTA and
// the row stays in registers between the binary32 sum of squares and the
// scale step: x (and the residual) are read from HBM exactly once
// ("Skill: Write a Triton RMSNorm Kernel", Required reasoning 3; Performance
// requirements, persistent vs two-pass).
#include "launch.h"

namespace rmsn {

template <typename T, int VEC, int NV, int MODE, int U>
__global__ void __launch_bounds__(512) fwd_row_kernel(FwdArgs a) {
    constexpr bool RESID = MODE == kResid || MODE == kLnResid;
    constexpr bool ADALN = MODE == kAdaln;
    constexpr bool LN = MODE == kLn || MODE == kLnResid;
    using P = Pack<T, VEC>;
    // 16-byte groups compute on binary32 pairs (two-lane f32x2 instructions);
    // the scalar path (unaligned rows) one element at a time
    constexpr bool PAIRS = VEC > 1;
    constexpr int PR = PAIRS ? VEC / 2 : 1;
    __shared__ float red[2 * U * 32];
    // x and y (the residual and residual_out) may be one array (in-place
    // calls): not restrict
    const T *x = static_cast<const T *>(a.x);
    const T *r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    const T *__restrict__ bias = static_cast<const T *>(a.b);
    const T *__restrict__ scale = static_cast<const T *>(a.scale);
    const T *__restrict__ shift = static_cast<const T *>(a.shift);
    T *y = static_cast<T *>(a.y);
    T *s_out = static_cast<T *>(a.s_out);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;   // exact: H < 2^24
    // the row's mean divides by H (multiplying by a per-CTA 1 / H, as the
    // other kernels do, measured 4.5% slower here: AdaLN with per-token
    // conditioning, bf16 12288 x 2048)

    // weight (and LayerNorm bias) (H,), indexed by column only; ones (zeros)
    // when absent.  Kept packed (and x, residual too): widening again in the
    // scale step is cheaper than the registers binary32 copies would take
    // from occupancy.
    P wp[NV], bp[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        wp[i] = (a.has_w && c < nvec) ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
        if constexpr (LN)
            bp[i] = (bias != nullptr && c < nvec) ? ld_cached<T, VEC>(bias + (int64_t)c * VEC) : fill<T, VEC>(T(0.0f));
    }

    // U consecutive rows per pass: all their loads are issued before any
    // arithmetic, and their U sums share one CTA barrier
    int bank = 0;
    const int64_t groups = (a.M + U - 1) / U;
    for (int64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        P xp[U][NV], rp[U][NV], scp[U][NV], shp[U][NV];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = grp * U + u;
            const int64_t base = row * a.stride;
            const int64_t cbase = ADALN ? (int64_t)((uint32_t)row / (uint32_t)a.rows_per_cond) * a.cond_stride : 0;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * blockDim.x;
                if (row < a.M && c < nvec) {
                    xp[u][i] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                    if constexpr (RESID) rp[u][i] = ld_stream<T, VEC>(r + base + (int64_t)c * VEC);
                    if constexpr (ADALN) {   // conditioning rows may be shared by many rows: cached path
                        scp[u][i] = ld_cached<T, VEC>(scale + cbase + (int64_t)c * VEC);
                        shp[u][i] = ld_cached<T, VEC>(shift + cbase + (int64_t)c * VEC);
                    }
                }
            }
        }
        // s = x (+ residual) in binary32, from the packed registers
        auto s_pairs = [&](int u, int i, f32x2 (&sv)[PR]) {
            if constexpr (PAIRS) {
                widen16<T>(xp[u][i], sv);
                if constexpr (RESID) {
                    f32x2 rv[PR];
                    widen16<T>(rp[u][i], rv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], rv[q]);
                }
            }
        };
        auto s_one = [&](int u, int i) {
            float v = to_f32(xp[u][i].v[0]);
            if constexpr (RESID) v += to_f32(rp[u][i].v[0]);
            return v;
        };
        // binary32 sum of squares (RMSNorm) or sum (LayerNorm's mean); the
        // post-add sum is written back as the next residual stream
        float ss[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = grp * U + u;
            const int64_t base = row * a.stride;
            ss[u] = 0.0f;
            f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * blockDim.x;
                if (row < a.M && c < nvec) {
                    if constexpr (PAIRS) {
                        f32x2 sv[PR];
                        widen16<T>(xp[u][i], sv);
                        if constexpr (RESID) {
                            f32x2 rv[PR];
                            widen16<T>(rp[u][i], rv);
#pragma unroll
                            for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], rv[q]);
                            st_global<T, VEC>(s_out + base + (int64_t)c * VEC, narrow16<T>(sv));
                        }
                        if constexpr (LN) {
#pragma unroll
                            for (int q = 0; q < PR; ++q) ss2 = f2_add(ss2, sv[q]);
                        } else {
#pragma unroll
                            for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[q], sv[q], ss2);
                        }
                    } else {
                        const float v = s_one(u, i);
                        if constexpr (RESID) s_out[base + c] = from_f32<T>(v);
                        if constexpr (LN) ss[u] += v;
                        else ss[u] += v * v;
                    }
                }
            }
            if constexpr (PAIRS) ss[u] = f2_sum(ss2);
        }
        block_sum_n<U>(ss, red, bank);
        bank ^= 1;
        // LayerNorm: the mean, then the centred sum of squares from the same
        // registers (a second reduction, no second read of the row)
        float mu[U];
        if constexpr (LN) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t row = grp * U + u;
                mu[u] = ss[u] / hf;
                const f32x2 nm2 = f2_make(-mu[u], -mu[u]);
                ss[u] = 0.0f;
                f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int c = threadIdx.x + i * blockDim.x;
                    if (row < a.M && c < nvec) {
                        if constexpr (PAIRS) {
                            f32x2 sv[PR];
                            s_pairs(u, i, sv);
#pragma unroll
                            for (int q = 0; q < PR; ++q) {
                                const f32x2 d = f2_add(sv[q], nm2);
                                ss2 = f2_fma(d, d, ss2);
                            }
                        } else {
                            const float d = s_one(u, i) - mu[u];
                            ss[u] += d * d;
                        }
                    }
                }
                if constexpr (PAIRS) ss[u] = f2_sum(ss2);
            }
            block_sum_n<U>(ss, red, bank);
            bank ^= 1;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = grp * U + u;
            if (row >= a.M) continue;
            const int64_t base = row * a.stride;
            // mean over the full row length, eps inside the square root
            // (LayerNorm: rstd of the centred row; rrms holds it)
            const float rrms = rsqrtf(ss[u] / hf + a.eps);
            if (threadIdx.x == 0) {
                if (a.rrms != nullptr) a.rrms[row] = rrms;
                if constexpr (LN)
                    if (a.mean != nullptr) a.mean[row] = mu[u];
            }
            const f32x2 rr2 = f2_make(rrms, rrms);
            // y = (s * rrms) * w [LayerNorm: ((s - mean) * rstd) * w + b], one
            // rounding to the storage type
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * blockDim.x;
                if (c < nvec) {
                    if constexpr (PAIRS) {
                        f32x2 sv[PR], wv[PR];
                        widen16<T>(xp[u][i], sv);
                        if constexpr (RESID) {
                            f32x2 rv[PR];
                            widen16<T>(rp[u][i], rv);
#pragma unroll
                            for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], rv[q]);
                        }
                        widen16<T>(wp[i], wv);
                        if constexpr (LN) {
                            f32x2 bv[PR];
                            widen16<T>(bp[i], bv);
                            const f32x2 nm2 = f2_make(-mu[u], -mu[u]);
#pragma unroll
                            for (int q = 0; q < PR; ++q)
                                sv[q] = f2_fma(f2_mul(f2_add(sv[q], nm2), rr2), wv[q], bv[q]);
                        } else if constexpr (ADALN) {   // (s * rrms) * (w * (1 + scale)) + shift
                            f32x2 sc[PR], sh[PR];
                            widen16<T>(scp[u][i], sc);
                            widen16<T>(shp[u][i], sh);
#pragma unroll
                            for (int q = 0; q < PR; ++q)
                                sv[q] = f2_fma(f2_mul(sv[q], rr2), f2_fma(wv[q], sc[q], wv[q]), sh[q]);
                        } else {
#pragma unroll
                            for (int q = 0; q < PR; ++q) sv[q] = f2_mul(f2_mul(sv[q], rr2), wv[q]);
                        }
                        st_global<T, VEC>(y + base + (int64_t)c * VEC, narrow16<T>(sv));
                    } else {
                        float v = s_one(u, i);
                        if constexpr (LN) {
                            v = fmaf((v - mu[u]) * rrms, to_f32(wp[i].v[0]), to_f32(bp[i].v[0]));
                        } else if constexpr (ADALN) {
                            const float wi = to_f32(wp[i].v[0]);
                            v = fmaf(v * rrms, fmaf(wi, to_f32(scp[u][i].v[0]), wi), to_f32(shp[u][i].v[0]));
                        } else {
                            v = (v * rrms) * to_f32(wp[i].v[0]);
                        }
                        y[base + c] = from_f32<T>(v);
                    }
                }
            }
        }
    }
}

namespace {

constexpr int kMaxThreads = 512;
constexpr int kVecNV[] = {1, 2, 3, 4};
constexpr int kScalarNV[] = {1, 2, 4, 8, 16};

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Column groups per thread: the smallest CTA of at most 128, else 256, else
// 512 threads that covers the row (measured: 128 threads x 2 groups is best
// at H = 2048 bf16).
bool pick(int nvec, bool vec, int &threads, int &nv) {
    const int *set = vec ? kVecNV : kScalarNV;
    const int n = vec ? 4 : 5;
    for (int cap : {128, 256, kMaxThreads}) {
        for (int k = 0; k < n; ++k) {
            const int t = round_up((nvec + set[k] - 1) / set[k], 32);
            if (t <= cap) {
                threads = t;
                nv = set[k];
                return true;
            }
        }
    }
    return false;
}

template <typename T, int VEC, int NV, int MODE, int U>
cudaError_t launch_u(const FwdArgs &a, int threads, int64_t grid, cudaStream_t st) {
    return launch_kernel(fwd_row_kernel<T, VEC, NV, MODE, U>, (unsigned)grid, (unsigned)threads, 0, st, a);
}

// Rows per pass: 2 keeps twice the bytes in flight per thread, but the rows
// are then dealt out in pairs, which can leave a larger last round (12288
// rows over 1368 CTAs: 8.98 rounds of one row, 4.49 rounds of two -- ten
// rows of work for the slowest CTA instead of nine).  Take 2 only for
// vector rows of at most 4 KB and only when it does not lengthen the
// slowest CTA's share.
template <typename T, int VEC, int NV, int MODE>
cudaError_t launch_t(const FwdArgs &a, int threads, int sm_count, cudaStream_t st) {
    const int occ = occupancy(reinterpret_cast<const void *>(fwd_row_kernel<T, VEC, NV, MODE, 1>), threads, 0);
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t cap = (int64_t)occ * sm_count;
    auto share = [&](int64_t u) {   // rows handled by the busiest CTA
        const int64_t groups = (a.M + u - 1) / u;
        return (groups + cap - 1) / cap * u;
    };
    if constexpr (VEC > 1 && NV <= 2) {
        if (share(2) <= share(1)) {
            const int occ2 =
                occupancy(reinterpret_cast<const void *>(fwd_row_kernel<T, VEC, NV, MODE, 2>), threads, 0);
            if (occ2 >= occ) {
                const int64_t groups = (a.M + 1) / 2;
                return launch_u<T, VEC, NV, MODE, 2>(a, threads, groups < cap ? groups : cap, st);
            }
        }
    }
    return launch_u<T, VEC, NV, MODE, 1>(a, threads, a.M < cap ? a.M : cap, st);
}

template <typename T, int VEC, int MODE>
cudaError_t launch_nv(const FwdArgs &a, int nv, int threads, int sm_count, cudaStream_t st) {
    if constexpr (VEC > 1) {
        switch (nv) {
        case 1: return launch_t<T, VEC, 1, MODE>(a, threads, sm_count, st);
        case 2: return launch_t<T, VEC, 2, MODE>(a, threads, sm_count, st);
        case 3: return launch_t<T, VEC, 3, MODE>(a, threads, sm_count, st);
        case 4: return launch_t<T, VEC, 4, MODE>(a, threads, sm_count, st);
        }
    } else {
        switch (nv) {
        case 1: return launch_t<T, 1, 1, MODE>(a, threads, sm_count, st);
        case 2: return launch_t<T, 1, 2, MODE>(a, threads, sm_count, st);
        case 4: return launch_t<T, 1, 4, MODE>(a, threads, sm_count, st);
        case 8: return launch_t<T, 1, 8, MODE>(a, threads, sm_count, st);
        case 16: return launch_t<T, 1, 16, MODE>(a, threads, sm_count, st);
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T, int VEC>
cudaError_t launch_mode(const FwdArgs &a, int mode, int nv, int threads, int sm_count, cudaStream_t st) {
    switch (mode) {
    case kPlain: return launch_nv<T, VEC, kPlain>(a, nv, threads, sm_count, st);
    case kResid: return launch_nv<T, VEC, kResid>(a, nv, threads, sm_count, st);
    case kAdaln: return launch_nv<T, VEC, kAdaln>(a, nv, threads, sm_count, st);
    case kLn: return launch_nv<T, VEC, kLn>(a, nv, threads, sm_count, st);
    case kLnResid: return launch_nv<T, VEC, kLnResid>(a, nv, threads, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, int mode, bool vec, int sm_count, cudaStream_t st) {
    constexpr int V = Vec16<T>::n;
    int threads = 0, nv = 0;
    if (!pick(vec ? a.H / V : a.H, vec, threads, nv)) return cudaErrorInvalidValue;
    return vec ? launch_mode<T, V>(a, mode, nv, threads, sm_count, st)
               : launch_mode<T, 1>(a, mode, nv, threads, sm_count, st);
}

}  // namespace

bool fwd_row_fits(int H, int dtype, bool vec) {
    int threads, nv;
    return pick(vec ? H / vec_elems(dtype) : H, vec, threads, nv);
}

cudaError_t launch_fwd_row(const FwdArgs &a, int dtype, int mode, bool vec, int sm_count, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, mode, vec, sm_count, st);
    case kF16: return launch_dt<__half>(a, mode, vec, sm_count, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, mode, vec, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
