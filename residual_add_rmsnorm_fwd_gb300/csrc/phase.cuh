// phase.cuh -- 128-bit accesses to rows that are not 16-byte aligned.
//
// A row whose first element sits p elements past a 16-byte boundary (its
// phase, 0 <= p < V, V = 16 / sizeof(T)) is read and written in its own
// aligned frame: frame vector k holds the columns k*V - p ... k*V - p + V - 1,
// so every frame vector but the first (columns below 0) and the last
// (columns from H) is a whole 16-byte access, and those two are masked
// element by element.  The matrices of one call share the row stride, so
// when their base addresses agree modulo 16 every row has one phase in all
// of them and a thread's frame vector k is the same columns in x, the
// residual and the outputs.
//
// A row at phase p spans nf = ceil((p + H) / V) frame vectors, at most one
// more than the ceil(H / V) vectors of an aligned row.  When it spans one
// more, its first vector holds columns 0 .. V-p-1 in elements p .. V-1 and
// its last vector the columns from (nf-1)V - p in elements 0 .. e-1, with
// e = p + H - (nf-1)V <= p: the two parts fit one vector.  So a row is
// handled in ceil(H / V) slots, slot k being frame vector k, and slot 0 also
// carrying the last frame vector when the row has one more (each part zero
// where the other one is, so the two merge by a bitwise or).  The kernels
// then have the thread geometry of an aligned row of the same length.
//
// Column-indexed operands (weight, bias, AdaLN conditioning rows) have a
// phase of their own, q.  The V columns of a frame vector then straddle two
// aligned vectors of the operand's frame; both are loaded (through L1) and
// the V elements are cut out of the pair by a shift of e = (q - p) mod V
// elements.  e is the same for every frame vector of a row, so the shift is
// one uniform branch per row to straight-line code.
#pragma once

#include "common.cuh"

namespace rmsn {

// Element phase of p: elements between the preceding 16-byte boundary and p.
template <typename T>
__device__ __forceinline__ int elem_phase(const T *p) {
    return (int)((reinterpret_cast<uintptr_t>(p) / sizeof(T)) & (16 / sizeof(T) - 1));
}

// Columns [c0, c0 + V) of a row (row = its column 0): a 16-byte access when
// all V columns lie in [0, H) -- then row + c0 is 16-byte aligned by the
// frame's construction -- else one element at a time, zero outside.
// Coherent loads: the row may be an in-place call's output.
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> ld_frame(const T *row, int c0, int H) {
    constexpr int V = 16 / sizeof(T);
    if (c0 >= 0 && c0 + V <= H) return ld_stream<T, V>(row + c0);
    Pack<T, V> r;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int c = c0 + j;
        r.v[j] = (c >= 0 && c < H) ? row[c] : from_f32<T>(0.0f);
    }
    return r;
}

template <typename T>
__device__ __forceinline__ void st_frame(T *row, int c0, int H, const Pack<T, 16 / sizeof(T)> &v) {
    constexpr int V = 16 / sizeof(T);
    if (c0 >= 0 && c0 + V <= H) {
        st_global<T, V>(row + c0, v);
        return;
    }
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int c = c0 + j;
        if (c >= 0 && c < H) row[c] = v.v[j];
    }
}

// A frame vector whose columns c0 ... c0 + V - 1 may reach outside [0, H)
// (the first or last of a row): those elements set to zero.
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> mask_frame(Pack<T, 16 / sizeof(T)> v, int c0, int H) {
#pragma unroll
    for (int j = 0; j < 16 / (int)sizeof(T); ++j)
        if (c0 + j < 0 || c0 + j >= H) v.v[j] = from_f32<T>(0.0f);
    return v;
}

// Slots of a row of H elements (16-byte vectors of an aligned row).
template <typename T>
__host__ __device__ __forceinline__ int frame_slots(int H) {
    return (H + 16 / (int)sizeof(T) - 1) / (16 / (int)sizeof(T));
}

// Bitwise or of two packs (two parts of slot 0, each zero where the other is).
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> or_packs(const Pack<T, 16 / sizeof(T)> &a,
                                                           const Pack<T, 16 / sizeof(T)> &b) {
    Pack<T, 16 / sizeof(T)> r;
    const uint32_t *x = reinterpret_cast<const uint32_t *>(&a);
    const uint32_t *y = reinterpret_cast<const uint32_t *>(&b);
    uint32_t *o = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int t = 0; t < 4; ++t) o[t] = x[t] | y[t];
    return r;
}

// Whether element j of slot k of a row at phase p holds a column of the row
// (wrap: the row spans one frame vector more than its slots).
template <typename T>
__device__ __forceinline__ bool slot_elem_in_row(int k, int j, int p, int H, bool wrap) {
    const int c = k * (16 / (int)sizeof(T)) + j - p;
    const int cw = frame_slots<T>(H) * (16 / (int)sizeof(T)) + j - p;
    return (c >= 0 && c < H) || (k == 0 && wrap && cw >= 0 && cw < H);
}

// Slot k of a row (row = its column 0, phase p) from a stage holding the
// row's frame vectors at 16-byte steps: columns outside the row zeroed, slot
// 0 merged with the last frame vector when the row wraps.
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> ld_slot_stage(const unsigned char *stg, int k, int p, int H,
                                                                bool wrap) {
    constexpr int V = 16 / sizeof(T);
    using P = Pack<T, V>;
    const int c0 = k * V - p;
    P v = *reinterpret_cast<const P *>(stg + (size_t)k * 16);
    if (c0 < 0 || c0 + V > H) v = mask_frame<T>(v, c0, H);
    if (k == 0 && wrap) {
        const int ns = frame_slots<T>(H);
        v = or_packs<T>(v, mask_frame<T>(*reinterpret_cast<const P *>(stg + (size_t)ns * 16), ns * V - p, H));
    }
    return v;
}

// Slot k of a row read from global memory (coherent loads).
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> ld_slot(const T *row, int k, int p, int H, bool wrap) {
    constexpr int V = 16 / sizeof(T);
    Pack<T, V> v = ld_frame<T>(row, k * V - p, H);
    if (k == 0 && wrap) v = or_packs<T>(v, ld_frame<T>(row, frame_slots<T>(H) * V - p, H));
    return v;
}

// Slot k of a row written back (only the row's own columns).
template <typename T>
__device__ __forceinline__ void st_slot(T *row, int k, int p, int H, bool wrap, const Pack<T, 16 / sizeof(T)> &v) {
    constexpr int V = 16 / sizeof(T);
    st_frame<T>(row, k * V - p, H, v);
    if (k == 0 && wrap) st_frame<T>(row, frame_slots<T>(H) * V - p, H, v);
}

// Whether the row at phase p spans one frame vector more than its slots.
template <typename T>
__device__ __forceinline__ bool row_wraps(int p, int H) {
    constexpr int V = 16 / sizeof(T);
    return (p + H + V - 1) / V > frame_slots<T>(H);
}

// A CTA's dweight partial row from the binary32 pairs of its frame vectors
// or slots (every row of the CTA at phase pc): element j of vector k is
// column k*V + j - pc, or -- slot 0 of a row that wraps into its slots --
// column ns*V + j - pc; columns outside [0, H) hold zeros and are not
// written.  SLOTS: the kernel holds the row's slots (else its frame vectors).
template <typename T, int NV, bool SLOTS>
__device__ __forceinline__ void store_partial(float *prow, const f32x2 (&acc)[NV][8 / sizeof(T)], int pc, int H,
                                              int k0, int kstep) {
    constexpr int V = 16 / sizeof(T);
    const int ns = frame_slots<T>(H);
    const bool wrap = SLOTS && row_wraps<T>(pc, H);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = k0 + i * kstep;
#pragma unroll
        for (int q = 0; q < V / 2; ++q) {
            float v[2];
            f2_split(acc[i][q], v[0], v[1]);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int j = 2 * q + t;
                int c = k * V + j - pc;
                if (k == 0 && c < 0 && wrap) c = ns * V + j - pc;   // the wrapped part
                if ((!SLOTS || k < ns) && c >= 0 && c < H) prow[c] = v[t];
            }
        }
    }
}

// Aligned vector j of a column-indexed operand's own frame (q = its phase):
// columns [j*V - q, j*V - q + V), through the read-only path; elements
// outside [0, H) are `fillv`.
template <typename T>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> ld_opframe(const T *v, int q, int j, int H, T fillv) {
    constexpr int V = 16 / sizeof(T);
    const int c0 = j * V - q;
    if (c0 >= 0 && c0 + V <= H) return ld_cached<T, V>(v + c0);
    Pack<T, V> r;
#pragma unroll
    for (int jj = 0; jj < V; ++jj) {
        const int c = c0 + jj;
        r.v[jj] = (c >= 0 && c < H) ? __ldg(v + c) : fillv;
    }
    return r;
}

// Elements E ... E + V - 1 of the 2V elements lo ++ hi (E a constant).
template <typename T, int E>
__device__ __forceinline__ Pack<T, 16 / sizeof(T)> cut(const Pack<T, 16 / sizeof(T)> &lo,
                                                        const Pack<T, 16 / sizeof(T)> &hi) {
    const uint32_t *a = reinterpret_cast<const uint32_t *>(&lo);
    const uint32_t *b = reinterpret_cast<const uint32_t *>(&hi);
    const uint32_t w[8] = {a[0], a[1], a[2], a[3], b[0], b[1], b[2], b[3]};
    Pack<T, 16 / sizeof(T)> r;
    uint32_t *o = reinterpret_cast<uint32_t *>(&r);
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int t = 0; t < 4; ++t) o[t] = w[E + t];
    } else if constexpr (E % 2 == 0) {
#pragma unroll
        for (int t = 0; t < 4; ++t) o[t] = w[E / 2 + t];
    } else {   // upper half of one word, lower half of the next
#pragma unroll
        for (int t = 0; t < 4; ++t) o[t] = __byte_perm(w[E / 2 + t], w[E / 2 + t + 1], 0x5432);
    }
    return r;
}

// Column-indexed operand v (phase q) seen from rows of phase p: where frame
// vector k's columns sit in v's frame.  Frame vector k starts at column
// k*V - p, which is element e of v's aligned vector k + jofs.
struct OpShift {
    int e;      // 0 .. V-1
    int jofs;   // -1 or 0
};

template <typename T>
__device__ __forceinline__ OpShift op_shift(int q, int p) {
    constexpr int V = 16 / sizeof(T);
    const int d = q - p;   // -(V-1) .. V-1
    return d < 0 ? OpShift{d + V, -1} : OpShift{d, 0};
}

// Calls f(std::integral_constant<int, e>) for the runtime shift e (uniform
// across the CTA for a row, so the branch does not diverge).
template <typename T, typename F>
__device__ __forceinline__ void with_shift(int e, F &&f) {
    using std::integral_constant;
    if constexpr (sizeof(T) == 4) {
        switch (e) {
        case 0: f(integral_constant<int, 0>{}); break;
        case 1: f(integral_constant<int, 1>{}); break;
        case 2: f(integral_constant<int, 2>{}); break;
        default: f(integral_constant<int, 3>{}); break;
        }
    } else {
        switch (e) {
        case 0: f(integral_constant<int, 0>{}); break;
        case 1: f(integral_constant<int, 1>{}); break;
        case 2: f(integral_constant<int, 2>{}); break;
        case 3: f(integral_constant<int, 3>{}); break;
        case 4: f(integral_constant<int, 4>{}); break;
        case 5: f(integral_constant<int, 5>{}); break;
        case 6: f(integral_constant<int, 6>{}); break;
        default: f(integral_constant<int, 7>{}); break;
        }
    }
}

// Columns [k*V - p, k*V - p + V) of the column-indexed operand v (zero
// outside [0, H)), for k = k0 + i * kstep (i < N, k < kcount: the row's
// slots, or its frame vectors), k = 0 also with the columns of the row's
// last frame vector when the row wraps into its slots: the operand's two
// aligned vectors per frame vector, cut by the row's shift.
template <typename T, int N>
__device__ __forceinline__ void ld_op_windows(const T *v, int q, int p, int H, int k0, int kstep, int kcount,
                                              bool wrap, Pack<T, 16 / sizeof(T)> (&out)[N]) {
    const OpShift s = op_shift<T>(q, p);
    const int ns = frame_slots<T>(H);
    const T zero = from_f32<T>(0.0f);
    with_shift<T>(s.e, [&](auto E) {
        constexpr int e = decltype(E)::value;
        auto window = [&](int k) {
            const int j = k + s.jofs;
            const Pack<T, 16 / sizeof(T)> lo = ld_opframe<T>(v, q, j, H, zero);
            if constexpr (e == 0) return lo;
            else return cut<T, e>(lo, ld_opframe<T>(v, q, j + 1, H, zero));
        };
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int k = k0 + i * kstep;
            if (k < kcount) out[i] = window(k);
        }
        if (k0 == 0 && wrap) out[0] = or_packs<T>(out[0], window(ns));
    });
}

}  // namespace rmsn
