// bwd_phase.cu -- RMSNorm backward (plain and with the residual stream's
// gradient) for rows that are not 16-byte aligned, when dy, x, dx (and
// dresidual_out) share their alignment phase.
//
// dx and the per-row dot product are computed in each row's aligned frame
// with 128-bit accesses (phase.cuh), as the register-row backward does for
// aligned rows ("Skill: Write a Triton RMSNorm Kernel", Required reasoning
// 12).  The dweight terms stay in registers across a CTA's rows, which needs
// every row of a CTA to put the same columns in the same frame vectors: the
// host makes the grid G a multiple of V whenever a CTA has more than one row,
// so the CTA's rows, G * stride elements apart, all have the CTA's phase.
// Each column is summed over the CTA's rows in row order, so dweight stays
// bit-reproducible.
#include "launch.h"
#include "phase.cuh"

namespace rmsn {

template <typename T, int NV, bool DRES>
__global__ void __launch_bounds__(512) bwd_phase_kernel(BwdArgs a) {
    constexpr int V = 16 / sizeof(T);
    constexpr int PR = V / 2;
    using P = Pack<T, V>;
    __shared__ float red[64];
    // dx may be dy, x or dres itself (in-place calls): not restrict
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    const T *x = static_cast<const T *>(a.x);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *dx = static_cast<T *>(a.dx);
    const int H = a.H;
    const float ih = 1.0f / (float)H;   // one division per CTA; exact for power-of-two H
    const int qw = a.has_w ? elem_phase(w) : 0;
    const int k0 = threadIdx.x, kstep = blockDim.x;

    // dweight terms of this thread's frame vectors k = k0 + i * kstep, element
    // j: column k*V + j - pc, pc the phase of every row of this CTA (the host
    // makes the grid a multiple of V whenever a CTA has more than one row, so
    // rows G apart are G * stride elements apart, a multiple of 16 bytes)
    const int pc = elem_phase(x + (int64_t)blockIdx.x * a.stride);
    f32x2 acc[NV][PR];
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int q = 0; q < PR; ++q) acc[i][q] = f2_make(0.0f, 0.0f);

    P wp[NV];
    int p_w = -1;
    int bank = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.stride;
        const int p = elem_phase(x + base);
        const int nf = (p + H + V - 1) / V;
        const float rr = __ldg(a.rrms + row);
        const f32x2 rr2 = f2_make(rr, rr);
        if (p != p_w) {
            if (a.has_w) ld_op_windows<T, NV>(w, qw, p, H, k0, kstep, nf, false, wp);
            else
#pragma unroll
                for (int i = 0; i < NV; ++i) wp[i] = fill<T, V>(one<T>());
            p_w = p;
        }
        P gp[NV], xp[NV], rp[NV];
        f32x2 dot2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = k0 + i * kstep;
            if (k < nf) {
                gp[i] = ld_frame<T>(dy + base, k * V - p, H);
                xp[i] = ld_frame<T>(x + base, k * V - p, H);
                if constexpr (DRES) rp[i] = ld_frame<T>(dres + base, k * V - p, H);
                f32x2 d[PR], xv[PR], wv[PR];
                widen16<T>(gp[i], d);
                widen16<T>(xp[i], xv);
                widen16<T>(wp[i], wv);
#pragma unroll
                for (int q = 0; q < PR; ++q) {
                    const f32x2 xh = f2_mul(xv[q], rr2);
                    dot2 = f2_fma(f2_mul(d[q], wv[q]), xh, dot2);
                    acc[i][q] = f2_fma(d[q], xh, acc[i][q]);   // dweight terms (zero outside the row)
                }
            }
        }
        const float c_row = block_sum(f2_sum(dot2), red, bank) * ih;

        // dx = rrms * (g - xhat * c) (+ dres), as the ring backward evaluates it
        const float kx = -(rr * rr) * c_row;
        const f32x2 kx2 = f2_make(kx, kx);
        const f32x2 nc2 = f2_make(-c_row, -c_row);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = k0 + i * kstep;
            if (k < nf) {
                f32x2 d[PR], xv[PR], wv[PR];
                widen16<T>(gp[i], d);
                widen16<T>(xp[i], xv);
                widen16<T>(wp[i], wv);
                if constexpr (DRES) {
                    f32x2 rv[PR];
                    widen16<T>(rp[i], rv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) d[q] = f2_fma(f2_mul(d[q], wv[q]), rr2, f2_fma(xv[q], kx2, rv[q]));
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q)
                        d[q] = f2_mul(rr2, f2_fma(f2_mul(xv[q], rr2), nc2, f2_mul(d[q], wv[q])));
                }
                st_frame<T>(dx + base, k * V - p, H, narrow16<T>(d));
            }
        }

        bank ^= 1;
    }

    if (a.partial != nullptr) store_partial<T, NV, false>(a.partial + (int64_t)blockIdx.x * H, acc, pc, H, k0, kstep);
    allow_dependent_launch();
}

namespace {

constexpr int kMaxThreads = 512;
constexpr int kNV[] = {1, 2, 3, 4};

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Frame vectors of the longest row frame (a row at phase V - 1).
inline int frame_vectors(int H, int dtype) {
    const int V = vec_elems(dtype);
    return (H + 2 * V - 2) / V;
}

// At most 512 threads, 1..4 frame vectors each.
bool pick(int nf, int &threads, int &nv) {
    for (int k : kNV) {
        const int t = round_up((nf + k - 1) / k, 32);
        if (t <= kMaxThreads) {
            threads = t;
            nv = k;
            return true;
        }
    }
    return false;
}

template <typename T, bool DRES>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 1: return reinterpret_cast<const void *>(bwd_phase_kernel<T, 1, DRES>);
    case 2: return reinterpret_cast<const void *>(bwd_phase_kernel<T, 2, DRES>);
    case 3: return reinterpret_cast<const void *>(bwd_phase_kernel<T, 3, DRES>);
    case 4: return reinterpret_cast<const void *>(bwd_phase_kernel<T, 4, DRES>);
    }
    return nullptr;
}

}  // namespace

bool bwd_phase_pick(int H, int dtype, int *threads, int *nv) {
    return pick(frame_vectors(H, dtype), *threads, *nv);
}

const void *bwd_phase_kernel_for(int dtype, int nv, bool dres) {
    switch (dtype) {
    case kF32: return dres ? kernel_nv<float, true>(nv) : kernel_nv<float, false>(nv);
    case kF16: return dres ? kernel_nv<__half, true>(nv) : kernel_nv<__half, false>(nv);
    case kBF16: return dres ? kernel_nv<__nv_bfloat16, true>(nv) : kernel_nv<__nv_bfloat16, false>(nv);
    }
    return nullptr;
}

}  // namespace rmsn
