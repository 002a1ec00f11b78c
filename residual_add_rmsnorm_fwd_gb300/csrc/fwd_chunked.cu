// fwd_chunked.cu -- RMSNorm forward (plain and residual-fused) for hidden
// sizes above the register budget of the row kernel.
//
// Two passes over each row with identical chunk bounds ("Skill: Write a
// Triton RMSNorm Kernel", Required reasoning 11; Kernel design rules, last
// rule): pass 1 accumulates the binary32 sum of squares chunk by chunk;
// pass 2 re-reads the chunks (the row was just read, so the re-read is
// mostly served by L2), recomputes the identical binary32 s = x + residual,
// and writes residual_out and y.  One CTA per row, persistent grid.
#include "launch.h"

namespace rmsn {

template <typename T, int VEC, bool RESID>
__global__ void __launch_bounds__(512) fwd_chunked_kernel(FwdArgs a) {
    using P = Pack<T, VEC>;
    constexpr int U = 2;  // vectors per thread per chunk (independent loads in flight)
    __shared__ float red[64];
    const T *__restrict__ x = static_cast<const T *>(a.x);
    const T *__restrict__ r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *__restrict__ y = static_cast<T *>(a.y);
    T *__restrict__ s_out = static_cast<T *>(a.s_out);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const int chunk = blockDim.x * U;

    int bank = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.stride;
        float ss = 0.0f;
        for (int c0 = 0; c0 < nvec; c0 += chunk) {
            P xp[U], rp[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    xp[u] = ld_cached<T, VEC>(x + base + (int64_t)c * VEC);
                    if constexpr (RESID) rp[u] = ld_cached<T, VEC>(r + base + (int64_t)c * VEC);
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
                    for (int j = 0; j < VEC; ++j) ss += v[j] * v[j];
                }
            }
        }
        const float total = block_sum(ss, red, bank);
        bank ^= 1;
        const float rrms = rsqrtf(total / hf + a.eps);
        if (a.rrms != nullptr && threadIdx.x == 0) a.rrms[row] = rrms;

        for (int c0 = 0; c0 < nvec; c0 += chunk) {
            P xp[U], rp[U], wp[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    xp[u] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                    if constexpr (RESID) rp[u] = ld_stream<T, VEC>(r + base + (int64_t)c * VEC);
                    wp[u] = a.has_w ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
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
#pragma unroll
                    for (int j = 0; j < VEC; ++j) v[j] = (v[j] * rrms) * wv[j];
                    st_global<T, VEC>(y + base + (int64_t)c * VEC, pack<T, VEC>(v));
                }
            }
        }
    }
}

namespace {

constexpr int kThreads = 512;

template <typename T, int VEC, bool RESID>
cudaError_t launch_t(const FwdArgs &a, int sm_count, cudaStream_t st) {
    auto k = fwd_chunked_kernel<T, VEC, RESID>;
    const int occ = occupancy(reinterpret_cast<const void *>(k), kThreads, 0);
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t cap = (int64_t)occ * sm_count;
    return launch_kernel(k, (unsigned)(a.M < cap ? a.M : cap), kThreads, 0, st, a);
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, bool vec, int sm_count, cudaStream_t st) {
    constexpr int V = Vec16<T>::n;
    const bool resid = a.r != nullptr;
    if (vec) return resid ? launch_t<T, V, true>(a, sm_count, st) : launch_t<T, V, false>(a, sm_count, st);
    return resid ? launch_t<T, 1, true>(a, sm_count, st) : launch_t<T, 1, false>(a, sm_count, st);
}

}  // namespace

cudaError_t launch_fwd_chunked(const FwdArgs &a, int dtype, bool vec, int sm_count, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, vec, sm_count, st);
    case kF16: return launch_dt<__half>(a, vec, sm_count, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, vec, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
