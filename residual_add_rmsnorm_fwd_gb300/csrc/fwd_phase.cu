// fwd_phase.cu -- RMSNorm forward (plain, residual-fused, AdaLN) and
// LayerNorm forward for rows that are not 16-byte aligned (odd hidden sizes,
// strides that are not a multiple of 16 bytes, views that start between
// 16-byte boundaries), when x, the residual and the outputs share their
// alignment phase.
//
// The row is read and written with 128-bit accesses in its own aligned frame
// and only the first and last frame vectors are masked element by element
// (phase.cuh); the weight, bias and conditioning rows are cut out of their
// own aligned vectors by the row's shift.  Otherwise the kernel is the
// register-row kernel: one CTA per row, persistent grid, the row in
// registers between the binary32 sum of squares and the scale step, so x
// (and the residual) are read from HBM once ("Skill: Write a Triton RMSNorm
// Kernel", Required reasoning 3 and 11; Performance requirements,
// vectorised accesses with masked tails).
#include "launch.h"
#include "phase.cuh"

namespace rmsn {

template <typename T, int NV, int MODE>
__global__ void __launch_bounds__(512) fwd_phase_kernel(FwdArgs a) {
    constexpr bool RESID = MODE == kResid || MODE == kLnResid;
    constexpr bool ADALN = MODE == kAdaln;
    constexpr bool LN = MODE == kLn || MODE == kLnResid;
    constexpr int V = 16 / sizeof(T);
    constexpr int PR = V / 2;
    using P = Pack<T, V>;
    __shared__ float red[64];
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
    const int H = a.H;
    const float hf = (float)H;   // exact: H < 2^24
    const int qw = a.has_w ? elem_phase(w) : 0;
    const int qb = (LN && bias != nullptr) ? elem_phase(bias) : 0;
    const int k0 = threadIdx.x, kstep = blockDim.x;

    // weight (and bias) windows of the last row phase seen: reloaded only
    // when the phase changes (never, when the stride is a multiple of 16 bytes)
    P wp[NV], bp[NV];
    int p_w = -1;
    int bank = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.stride;
        const int p = elem_phase(x + base);
        const int nf = (p + H + V - 1) / V;
        P xp[NV], rp[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = k0 + i * kstep;
            if (k < nf) {
                xp[i] = ld_frame<T>(x + base, k * V - p, H);
                if constexpr (RESID) rp[i] = ld_frame<T>(r + base, k * V - p, H);
            }
        }
        // s = x (+ residual) in binary32; masked elements are zeros
        auto s_pairs = [&](int i, f32x2 (&sv)[PR]) {
            widen16<T>(xp[i], sv);
            if constexpr (RESID) {
                f32x2 rv[PR];
                widen16<T>(rp[i], rv);
#pragma unroll
                for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], rv[q]);
            }
        };
        f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = k0 + i * kstep;
            if (k < nf) {
                f32x2 sv[PR];
                s_pairs(i, sv);
                if constexpr (RESID) st_frame<T>(s_out + base, k * V - p, H, narrow16<T>(sv));
                if constexpr (LN) {
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_add(ss2, sv[q]);
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[q], sv[q], ss2);
                }
            }
        }
        float total = block_sum(f2_sum(ss2), red, bank);
        bank ^= 1;
        float mu = 0.0f;
        if constexpr (LN) {   // the centred sum of squares from the same registers
            mu = total / hf;
            const f32x2 nm2 = f2_make(-mu, -mu);
            ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int k = k0 + i * kstep;
                if (k < nf) {
                    f32x2 sv[PR];
                    s_pairs(i, sv);
                    const int c0 = k * V - p;
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[q] = f2_add(sv[q], nm2);
                    if (c0 < 0 || c0 + V > H) {   // columns outside the row add nothing
#pragma unroll
                        for (int q = 0; q < PR; ++q) {
                            float d0, d1;
                            f2_split(sv[q], d0, d1);
                            const int c = c0 + 2 * q;
                            sv[q] = f2_make(c >= 0 && c < H ? d0 : 0.0f, c + 1 >= 0 && c + 1 < H ? d1 : 0.0f);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[q], sv[q], ss2);
                }
            }
            total = block_sum(f2_sum(ss2), red, bank);
            bank ^= 1;
        }
        // mean over the full row length, eps inside the square root
        // (LayerNorm: rstd of the centred row; rrms holds it)
        const float rrms = rsqrtf(total / hf + a.eps);
        if (threadIdx.x == 0) {
            if (a.rrms != nullptr) a.rrms[row] = rrms;
            if constexpr (LN)
                if (a.mean != nullptr) a.mean[row] = mu;
        }
        if (p != p_w) {
            if (a.has_w) ld_op_windows<T, NV>(w, qw, p, H, k0, kstep, nf, false, wp);
            else
#pragma unroll
                for (int i = 0; i < NV; ++i) wp[i] = fill<T, V>(one<T>());
            if constexpr (LN) {
                if (bias != nullptr) ld_op_windows<T, NV>(bias, qb, p, H, k0, kstep, nf, false, bp);
                else
#pragma unroll
                    for (int i = 0; i < NV; ++i) bp[i] = fill<T, V>(from_f32<T>(0.0f));
            }
            p_w = p;
        }
        P scp[NV], shp[NV];
        if constexpr (ADALN) {   // this row's conditioning row (its own phase)
            const int64_t cbase = (int64_t)((uint32_t)row / (uint32_t)a.rows_per_cond) * a.cond_stride;
            ld_op_windows<T, NV>(scale + cbase, elem_phase(scale + cbase), p, H, k0, kstep, nf, false, scp);
            ld_op_windows<T, NV>(shift + cbase, elem_phase(shift + cbase), p, H, k0, kstep, nf, false, shp);
        }
        const f32x2 rr2 = f2_make(rrms, rrms);
        // y = (s * rrms) * w [LayerNorm: ((s - mean) * rstd) * w + b; AdaLN:
        // (s * rrms) * (w * (1 + scale)) + shift], one rounding to storage
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = k0 + i * kstep;
            if (k < nf) {
                f32x2 sv[PR], wv[PR];
                s_pairs(i, sv);
                widen16<T>(wp[i], wv);
                if constexpr (LN) {
                    f32x2 bv[PR];
                    widen16<T>(bp[i], bv);
                    const f32x2 nm2 = f2_make(-mu, -mu);
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[q] = f2_fma(f2_mul(f2_add(sv[q], nm2), rr2), wv[q], bv[q]);
                } else if constexpr (ADALN) {
                    f32x2 sc[PR], sh[PR];
                    widen16<T>(scp[i], sc);
                    widen16<T>(shp[i], sh);
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[q] = f2_fma(f2_mul(sv[q], rr2), f2_fma(wv[q], sc[q], wv[q]), sh[q]);
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[q] = f2_mul(f2_mul(sv[q], rr2), wv[q]);
                }
                st_frame<T>(y + base, k * V - p, H, narrow16<T>(sv));
            }
        }
    }
}

namespace {

constexpr int kMaxThreads = 512;
constexpr int kNV[] = {1, 2, 3, 4};

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Frame vectors of the longest row frame: a row of H elements at phase
// V - 1 spans ceil((H + V - 1) / V) of them.
inline int frame_vectors(int H, int dtype) {
    const int V = vec_elems(dtype);
    return (H + 2 * V - 2) / V;
}

// The smallest CTA of at most 128, else 256, else 512 threads that covers
// the frame with 1..4 vectors per thread (as the register-row kernel).
bool pick(int nf, int &threads, int &nv) {
    for (int cap : {128, 256, kMaxThreads}) {
        for (int k : kNV) {
            const int t = round_up((nf + k - 1) / k, 32);
            if (t <= cap) {
                threads = t;
                nv = k;
                return true;
            }
        }
    }
    return false;
}

template <typename T, int NV, int MODE>
cudaError_t launch_t(const FwdArgs &a, int threads, int sm_count, cudaStream_t st) {
    auto k = fwd_phase_kernel<T, NV, MODE>;
    const int occ = occupancy(reinterpret_cast<const void *>(k), threads, 0);
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t cap = (int64_t)occ * sm_count;
    return launch_kernel(k, (unsigned)(a.M < cap ? a.M : cap), (unsigned)threads, 0, st, a);
}

template <typename T, int MODE>
cudaError_t launch_nv(const FwdArgs &a, int nv, int threads, int sm_count, cudaStream_t st) {
    switch (nv) {
    case 1: return launch_t<T, 1, MODE>(a, threads, sm_count, st);
    case 2: return launch_t<T, 2, MODE>(a, threads, sm_count, st);
    case 3: return launch_t<T, 3, MODE>(a, threads, sm_count, st);
    case 4: return launch_t<T, 4, MODE>(a, threads, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, int mode, int sm_count, cudaStream_t st) {
    int threads = 0, nv = 0;
    if (!pick(frame_vectors(a.H, sizeof(T) == 4 ? kF32 : kBF16), threads, nv)) return cudaErrorInvalidValue;
    switch (mode) {
    case kPlain: return launch_nv<T, kPlain>(a, nv, threads, sm_count, st);
    case kResid: return launch_nv<T, kResid>(a, nv, threads, sm_count, st);
    case kAdaln: return launch_nv<T, kAdaln>(a, nv, threads, sm_count, st);
    case kLn: return launch_nv<T, kLn>(a, nv, threads, sm_count, st);
    case kLnResid: return launch_nv<T, kLnResid>(a, nv, threads, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool fwd_phase_fits(int H, int dtype) {
    int threads, nv;
    return pick(frame_vectors(H, dtype), threads, nv);
}

cudaError_t launch_fwd_phase(const FwdArgs &a, int dtype, int mode, int sm_count, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, mode, sm_count, st);
    case kF16: return launch_dt<__half>(a, mode, sm_count, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, mode, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
