// common.cuh -- device helpers shared by the RMSNorm kernels: storage-type
// traits, 128-bit / scalar global accesses, and warp / CTA sum reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

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
    unsigned *err;        // device error word (bounded pipeline waits report here)
    uint32_t wait_polls;  // polls before a pipeline wait gives up (kWaitPolls unless under test)
    int hold_first;       // test of the time-out path: the issuing thread of each ring CTA waits
                          // for its first row before issuing any copy (0 in normal use)
    // AdaLN conditioning: token row i reads scale/shift row i / rows_per_cond
    const void *scale;
    const void *shift;
    int64_t cond_stride;
    int64_t rows_per_cond;   // 1..M (clamped to M by the host), so row / rows_per_cond fits 32 bits
    int64_t cond_groups;     // shared AdaLN on the ring: conditioning rows each given their own CTAs, or 0
    // LayerNorm: bias (H,) or nullptr, and the saved per-row mean (M) or
    // nullptr; rrms then holds the per-row rstd
    const void *b;
    float *mean;
};

// Forward variants: plain norm, residual-fused, AdaLN (norm * w * (1 + scale)
// + shift).  kAdalnShared is AdaLN whose conditioning rows each serve at
// least four of a CTA's strides of rows (one row per sequence): the bulk-copy
// ring then reads a conditioning row through L1 when the CTA's rows enter
// it and keeps w * (1 + scale) and shift in registers, instead of staging
// it beside every x row; the other kernels read conditioning through L1.
// kLn / kLnResid are LayerNorm, plain and residual-fused: ((s - mean) *
// rstd) * w + b with the mean and the centred variance of the row.
enum FwdMode { kPlain = 0, kResid = 1, kAdaln = 2, kAdalnShared = 3, kLn = 4, kLnResid = 5 };

struct BwdArgs {
    const void *dy;
    const void *dres;     // gradient arriving through the fused forward's residual_out, or nullptr
    const void *x;
    const void *w;
    const float *rrms;
    void *dx;
    float *partial;       // G x H per-CTA dweight partials, or nullptr
    int64_t stride;
    int64_t M;
    int H;
    int has_w;
    unsigned *err;
    uint32_t wait_polls;  // as in FwdArgs
    int hold_first;       // as in FwdArgs
    int use_smem_acc;     // chunked kernel: partial row accumulated in shared memory
};

// Geometry of a shared-memory row ring (bulk-copy kernels).
struct RingShape {
    int stages;           // rows in flight per CTA
    uint32_t row_bytes;   // H * sizeof(T), a multiple of 16
    uint32_t row_pitch;   // row_bytes rounded up to 128
};

// Geometry of a split-row kernel: each CTA of a cluster owns `seg_groups`
// 16-byte groups of the row (the last CTA the rest) and stages them in a
// ring like a whole row.
struct SplitShape {
    int stages;           // segments in flight per CTA (per input stream)
    int seg_groups;       // 16-byte groups per CTA segment
    uint32_t seg_pitch;   // seg_groups * 16 rounded up to 128
};

// Bytes reserved at the start of a ring kernel's dynamic shared memory for
// its mbarriers (one 8-byte barrier per stage, at most 16 stages).
constexpr int kRingHeaderBytes = 128;
constexpr int kRingMaxStages = 16;
// The backward ring always has two stages (measured best; the kernel takes the
// count as a constant, so the stage index and mbarrier phase of row k are
// bit operations).
constexpr int kBwdRingStages = 2;

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

// Streaming load of a row the CTA reads once: no L1 allocation (L2 still
// caches it).  A coherent load, not the non-coherent read-only path: the
// row may be an in-place call's output, written later in the same kernel.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 u;
    asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
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

// Coherent load with normal L1 caching: a row read again soon (the chunked
// kernels' first pass), which may be an in-place call's output.
template <typename T, int N>
__device__ __forceinline__ Pack<T, N> ld_plain(const T *p) {
    Pack<T, N> r;
    if constexpr (sizeof(T) * N == 16) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        r = *reinterpret_cast<const Pack<T, N> *>(&u);
    } else {
        static_assert(N == 1, "scalar path loads one element");
        r.v[0] = p[0];
    }
    return r;
}

// Load through the read-only path with normal L1 caching: only for data no
// call writes (weights, bias, AdaLN conditioning rows, saved rrms), reused by
// every row a CTA handles.
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

// ---------------------------------------------------------------------------
// Pairs of binary32 values held in one 64-bit register pair, operated on by
// the two-lane binary32 instructions (add/mul/fma .rn.f32x2): each lane is
// rounded exactly as the scalar instruction would round it.
// ---------------------------------------------------------------------------

using f32x2 = unsigned long long;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
    f32x2 u;
    asm("mov.b64 %0, {%1, %2};" : "=l"(u) : "f"(lo), "f"(hi));
    return u;
}
__device__ __forceinline__ void f2_split(f32x2 u, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(u));
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ float f2_sum(f32x2 u) {
    float lo, hi;
    f2_split(u, lo, hi);
    return lo + hi;
}

// Two IEEE binary16 values (one 32-bit word, low half first) -> binary32
// pair, exactly, with the mixed-precision add (binary16 operand widened
// inside a binary32 add) on the FP32 pipe rather than the conversion pipe:
// h + (-0) = h for every h, including -0, infinities and NaN.
__device__ __forceinline__ f32x2 widen_f16x2(uint32_t w) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, 0f80000000;\n\t"
        "add.rn.f32.f16 %1, h, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
    return f2_make(lo, hi);
}

// Pairs in one 16-byte vector of storage type T.
template <typename T> struct Pairs16 { static constexpr int n = 16 / (int)sizeof(T) / 2; };

// 16 bytes of storage -> binary32 pairs (exact).
template <typename T>
__device__ __forceinline__ void widen16(const Pack<T, 16 / sizeof(T)> &p, f32x2 (&o)[Pairs16<T>::n]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&p);
    if constexpr (std::is_same<T, float>::value) {
        o[0] = f2_make(__uint_as_float(w[0]), __uint_as_float(w[1]));
        o[1] = f2_make(__uint_as_float(w[2]), __uint_as_float(w[3]));
    } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = f2_make(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = widen_f16x2(w[q]);
    }
}

// binary32 pairs -> 16 bytes of storage, each value rounded to nearest even.
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> narrow16(const f32x2 (&v)[Pairs16<T>::n]) {
    Pack<T, 16 / sizeof(T)> p;
    uint32_t *w = reinterpret_cast<uint32_t *>(&p);
#pragma unroll
    for (int q = 0; q < Pairs16<T>::n; ++q) {
        float lo, hi;
        f2_split(v[q], lo, hi);
        if constexpr (std::is_same<T, float>::value) {
            w[2 * q] = __float_as_uint(lo);
            w[2 * q + 1] = __float_as_uint(hi);
        } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
            w[q] = *reinterpret_cast<const uint32_t *>(&t);
        } else {
            const __half2 t = __floats2half2_rn(lo, hi);
            w[q] = *reinterpret_cast<const uint32_t *>(&t);
        }
    }
    return p;
}

// Whole-pack conversions.  16-byte packs of 2-byte types are handled as four
// 32-bit words holding two elements each, so a pack stays in 4 registers:
// bfloat16 is the upper half of a binary32, so widening is a shift or a mask;
// binary16 widens with the half2 intrinsic; narrowing rounds two values at a
// time to nearest even with the paired conversion intrinsics.
template <typename T, int N>
__device__ __forceinline__ void unpack(const Pack<T, N> &p, float (&f)[N]) {
    if constexpr (sizeof(T) == 2 && N % 2 == 0) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&p);
#pragma unroll
        for (int q = 0; q < N / 2; ++q) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                f[2 * q] = __uint_as_float(w[q] << 16);
                f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
            } else {
                f2_split(widen_f16x2(w[q]), f[2 * q], f[2 * q + 1]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) f[j] = to_f32(p.v[j]);
    }
}

template <typename T, int N>
__device__ __forceinline__ Pack<T, N> pack(const float (&f)[N]) {
    Pack<T, N> p;
    if constexpr (sizeof(T) == 2 && N % 2 == 0) {
        uint32_t *w = reinterpret_cast<uint32_t *>(&p);
#pragma unroll
        for (int q = 0; q < N / 2; ++q) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                const __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);
                w[q] = *reinterpret_cast<const uint32_t *>(&t);
            } else {
                const __half2 t = __floats2half2_rn(f[2 * q], f[2 * q + 1]);
                w[q] = *reinterpret_cast<const uint32_t *>(&t);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) p.v[j] = from_f32<T>(f[j]);
    }
    return p;
}

template <typename T, int N>
__device__ __forceinline__ Pack<T, N> fill(T v) {
    Pack<T, N> r;
#pragma unroll
    for (int j = 0; j < N; ++j) r.v[j] = v;
    return r;
}

// Programmatic dependent launch: a grid launched after this one with
// programmatic stream serialisation (the dweight reduction after a backward)
// may be scheduled once every CTA of this grid has signalled or exited; it
// still waits (griddepcontrol.wait) for this grid's completion and memory
// before it reads anything this grid wrote.  Signalled as a CTA's last
// step, so the dependent's CTAs only take SM slots this grid has released.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Sums over the CTA of U values at once, behind one barrier.  `red` holds
// two banks of U * 32 floats, alternated as for block_sum.
template <int U>
__device__ __forceinline__ void block_sum_n(float (&v)[U], float *red, int bank) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *buf = red + bank * U * 32;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        v[u] = group_sum<32>(v[u]);
        if (lane == 0) buf[u * 32 + warp] = v[u];
    }
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = group_sum<32>(lane < nwarps ? buf[u * 32 + lane] : 0.0f);
}

}  // namespace rmsn
