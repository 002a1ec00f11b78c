// common.cuh -- device helpers shared by the RMSNorm kernels: storage-type
// traits, 128-bit / scalar global accesses, and warp / CTA sum reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

// ---------------------------------------------------------------------------
// Kernel argument blocks (passed by value)
// ---------------------------------------------------------------------------

struct FwdArgs {
    const void *x;        // M x H, row stride `stride`
    const void *r;        // residual (fused forward) or nullptr
    const void *w;        // H weights (read only when has_w)
    void *y;              // M x H output
    void *s_out;          // residual_out (fused forward) or nullptr
    float *rrms;          // M, or nullptr
    int64_t stride;       // row stride in elements
    int64_t M;
    int H;
    float eps;
    int has_w;
};

struct BwdArgs {
    const void *dy;
    const void *x;
    const void *w;
    const float *rrms;
    void *dx;
    float *partial;       // G x H per-CTA dweight partials, or nullptr
    int64_t stride;
    int64_t M;
    int H;
    int has_w;
};

// ---------------------------------------------------------------------------
// Storage types
// ---------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

template <typename T> __device__ __forceinline__ T one() { return from_f32<T>(1.0f); }

// Elements per 128-bit access.
template <typename T> struct Vec16 { static constexpr int n = 16 / (int)sizeof(T); };

// N elements of T kept in their storage format (N * sizeof(T) is 16 bytes
// for the vector path, sizeof(T) for the scalar path).
template <typename T, int N> struct alignas(sizeof(T) * N) Pack {
    T v[N];
};

// Read-only streaming load: the data is not reused by this CTA, so it
// bypasses L1 allocation (L2 still caches it).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 u;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
        : "l"(p));
    return u;
}

template <typename T, int N>
__device__ __forceinline__ Pack<T, N> ld_stream(const T *p) {
    Pack<T, N> r;
    if constexpr (sizeof(T) * N == 16) {
        uint4 u = ld_stream_v4(p);
        r = *reinterpret_cast<const Pack<T, N> *>(&u);
    } else {
        static_assert(N == 1, "scalar path loads one element");
        r.v[0] = p[0];
    }
    return r;
}

// Load through the read-only path with normal L1 caching (weights, reused
// by every row a CTA handles).
template <typename T, int N>
__device__ __forceinline__ Pack<T, N> ld_cached(const T *p) {
    Pack<T, N> r;
    if constexpr (sizeof(T) * N == 16) {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        r = *reinterpret_cast<const Pack<T, N> *>(&u);
    } else {
        static_assert(N == 1, "scalar path loads one element");
        r.v[0] = p[0];
    }
    return r;
}

template <typename T, int N>
__device__ __forceinline__ void st_global(T *p, const Pack<T, N> &v) {
    if constexpr (sizeof(T) * N == 16) {
        *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(&v);
    } else {
        static_assert(N == 1, "scalar path stores one element");
        p[0] = v.v[0];
    }
}

template <typename T, int N>
__device__ __forceinline__ Pack<T, N> fill(T v) {
    Pack<T, N> r;
#pragma unroll
    for (int j = 0; j < N; ++j) r.v[j] = v;
    return r;
}

// ---------------------------------------------------------------------------
// Reductions.  The xor butterfly leaves the bit-identical sum in every lane
// (each step adds the same two values in either order), so every thread of a
// row sees exactly the same total and therefore the same rrms.
// ---------------------------------------------------------------------------

template <int WIDTH = 32>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Sum over the CTA.  `red` holds two banks of 32 floats; callers alternate
// `bank` between consecutive reductions so one __syncthreads per reduction
// suffices (a bank is rewritten only after the next reduction's barrier).
__device__ __forceinline__ float block_sum(float v, float *red, int bank) {
    v = group_sum<32>(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *buf = red + bank * 32;
    if (lane == 0) buf[warp] = v;
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    float t = lane < nwarps ? buf[lane] : 0.0f;
    return group_sum<32>(t);
}

}  // namespace rmsn
