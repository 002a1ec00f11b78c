// fwd_chunked.cu -- RMSNorm forward (plain, residual-fused, AdaLN) and
// residual + LayerNorm forward for hidden sizes above the register budget of
// the row kernel.
//
// Two passes over each row with identical chunk bounds ("Skill: Write a
// Triton RMSNorm Kernel", Required reasoning 11; Kernel design rules, last
// rule): pass 1 accumulates the binary32 sum of squares chunk by chunk;
// pass 2 re-reads the chunks (the row was just read, so the re-read is
// mostly served by L2), recomputes the identical binary32 s = x + residual,
// and writes residual_out and y (AdaLN: (s * rrms) * (w * (1 + scale)) +
// shift, "Rocm Kernels" page, 4. AdaLN).  LayerNorm makes three passes: the sum (the
// mean), the centred sum of squares, then the output.  One CTA per row,
// persistent grid.
#include "launch.h"

namespace rmsn {

template <typename T, int VEC, int MODE>
__global__ void __launch_bounds__(512) fwd_chunked_kernel(FwdArgs a) {
    constexpr bool RESID = MODE == kResid || MODE == kLnResid;
    constexpr bool ADALN = MODE == kAdaln;
    constexpr bool LN = MODE == kLn || MODE == kLnResid;
    using P = Pack<T, VEC>;
    constexpr int U = 2;  // vectors per thread per chunk (independent loads in flight)
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
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H
    const int chunk = blockDim.x * U;

    int bank = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.stride;
        const int64_t cbase = ADALN ? (int64_t)((uint32_t)row / (uint32_t)a.rows_per_cond) * a.cond_stride : 0;
        // one pass over the row's chunks: accumulates sum(s^2), sum(s) or
        // (LayerNorm's second pass) sum((s - centre)^2), s = x (+ residual)
        auto reduce_pass = [&](int kind, float centre) {
            float acc = 0.0f;
            for (int c0 = 0; c0 < nvec; c0 += chunk) {
                P xp[U], rp[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * blockDim.x + threadIdx.x;
                    if (c < nvec) {
                        xp[u] = ld_plain<T, VEC>(x + base + (int64_t)c * VEC);
                        if constexpr (RESID) rp[u] = ld_plain<T, VEC>(r + base + (int64_t)c * VEC);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * blockDim.x + threadIdx.x;
                    if (c < nvec) {
                        float v[VEC];
                        unpack(xp[u], v);
                        if constexpr (RESID) {
                            float rv[VEC];
                            unpack(rp[u], rv);
#pragma unroll
                            for (int j = 0; j < VEC; ++j) v[j] += rv[j];
                        }
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            if (kind == 1) {
                                acc += v[j];
                            } else {
                                const float d = v[j] - centre;
                                acc += d * d;
                            }
                        }
                    }
                }
            }
            return acc;
        };
        float mu = 0.0f;
        float total;
        if constexpr (LN) {   // the mean, then the centred sum of squares (a second re-read)
            total = block_sum(reduce_pass(1, 0.0f), red, bank);
            bank ^= 1;
            mu = total * ih;
            total = block_sum(reduce_pass(0, mu), red, bank);
            bank ^= 1;
        } else {
            total = block_sum(reduce_pass(0, 0.0f), red, bank);
            bank ^= 1;
        }
        const float rrms = rsqrtf(total * ih + a.eps);
        if (threadIdx.x == 0) {
            if (a.rrms != nullptr) a.rrms[row] = rrms;
            if constexpr (LN)
                if (a.mean != nullptr) a.mean[row] = mu;
        }

        for (int c0 = 0; c0 < nvec; c0 += chunk) {
            P xp[U], rp[U], wp[U], bp[U], scp[U], shp[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    xp[u] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                    if constexpr (RESID) rp[u] = ld_stream<T, VEC>(r + base + (int64_t)c * VEC);
                    wp[u] = a.has_w ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
                    if constexpr (LN)
                        bp[u] = bias != nullptr ? ld_cached<T, VEC>(bias + (int64_t)c * VEC)
                                                : fill<T, VEC>(from_f32<T>(0.0f));
                    if constexpr (ADALN) {
                        scp[u] = ld_cached<T, VEC>(scale + cbase + (int64_t)c * VEC);
                        shp[u] = ld_cached<T, VEC>(shift + cbase + (int64_t)c * VEC);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    float v[VEC], wv[VEC];
                    unpack(xp[u], v);
                    if constexpr (RESID) {
                        float rv[VEC];
                        unpack(rp[u], rv);
#pragma unroll
                        for (int j = 0; j < VEC; ++j) v[j] += rv[j];
                        st_global<T, VEC>(s_out + base + (int64_t)c * VEC, pack<T, VEC>(v));
                    }
                    unpack(wp[u], wv);
                    if constexpr (LN) {   // ((s - mean) * rstd) * w + b
                        float bv[VEC];
                        unpack(bp[u], bv);
#pragma unroll
                        for (int j = 0; j < VEC; ++j) v[j] = fmaf((v[j] - mu) * rrms, wv[j], bv[j]);
                    } else if constexpr (ADALN) {   // (s * rrms) * (w * (1 + scale)) + shift
                        float sc[VEC], sh[VEC];
                        unpack(scp[u], sc);
                        unpack(shp[u], sh);
#pragma unroll
                        for (int j = 0; j < VEC; ++j) v[j] = fmaf(v[j] * rrms, fmaf(wv[j], sc[j], wv[j]), sh[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < VEC; ++j) v[j] = (v[j] * rrms) * wv[j];
                    }
                    st_global<T, VEC>(y + base + (int64_t)c * VEC, pack<T, VEC>(v));
                }
            }
        }
    }
}

namespace {

constexpr int kThreads = 512;

template <typename T, int VEC, int MODE>
cudaError_t launch_t(const FwdArgs &a, int sm_count, cudaStream_t st) {
    auto k = fwd_chunked_kernel<T, VEC, MODE>;
    const int occ = occupancy(reinterpret_cast<const void *>(k), kThreads, 0);
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t cap = (int64_t)occ * sm_count;
    return launch_kernel(k, (unsigned)(a.M < cap ? a.M : cap), kThreads, 0, st, a);
}

template <typename T, int VEC>
cudaError_t launch_mode(const FwdArgs &a, int mode, int sm_count, cudaStream_t st) {
    switch (mode) {
    case kPlain: return launch_t<T, VEC, kPlain>(a, sm_count, st);
    case kResid: return launch_t<T, VEC, kResid>(a, sm_count, st);
    case kAdaln: return launch_t<T, VEC, kAdaln>(a, sm_count, st);
    case kLn: return launch_t<T, VEC, kLn>(a, sm_count, st);
    case kLnResid: return launch_t<T, VEC, kLnResid>(a, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, int mode, bool vec, int sm_count, cudaStream_t st) {
    constexpr int V = Vec16<T>::n;
    return vec ? launch_mode<T, V>(a, mode, sm_count, st) : launch_mode<T, 1>(a, mode, sm_count, st);
}

}  // namespace

cudaError_t launch_fwd_chunked(const FwdArgs &a, int dtype, int mode, bool vec, int sm_count, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, mode, vec, sm_count, st);
    case kF16: return launch_dt<__half>(a, mode, vec, sm_count, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, mode, vec, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
