// bwd_phase.cu -- RMSNorm backward (plain and with the residual stream's
// gradient) for rows that are not 16-byte aligned, when dy, x, dx (and
// dresidual_out) share their alignment phase.
//
// dx and the per-row dot product are computed in each row's aligned frame
// with 128-bit accesses (phase.cuh), as the register-row backward does for
// aligned rows ("Skill: Write a Triton RMSNorm Kernel", Required reasoning
// 12).  The dweight partials need a thread-to-column map that does not move
// from row to row, so they are kept in the column frame instead: a thread
// owns the columns m*V ... m*V + V - 1 of its frame vectors m.  A frame
// vector of a row at phase p holds the last V - p of those columns in its
// elements p ... V - 1 and the first p of them sit in the next frame vector,
// which the next lane holds: the thread takes them with p warp shuffles (the
// last lane of a warp from the next warp's first lane, through shared memory
// behind the row's reduction barrier).  Each column is summed over the CTA's
// rows in row order, so dweight stays bit-reproducible.
#include "launch.h"
#include "phase.cuh"

namespace rmsn {

template <typename T, int NV, bool DRES>
__global__ void __launch_bounds__(512) bwd_phase_kernel(BwdArgs a) {
    constexpr int V = 16 / sizeof(T);
    constexpr int PR = V / 2;
    using P = Pack<T, V>;
    __shared__ float red[64];
    // first lane of every warp: its dweight terms, for the previous warp's
    // last lane (two banks, alternated per row like `red`)
    __shared__ float edge[2][16][NV][V];
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const bool want_dw = a.partial != nullptr;

    float acc[NV][V];   // dweight terms of columns m*V + j, m = k0 + i * kstep
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int j = 0; j < V; ++j) acc[i][j] = 0.0f;

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
            if (a.has_w) ld_op_windows<T, NV>(w, qw, p, H, k0, kstep, nf, from_f32<T>(0.0f), wp);
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
                for (int q = 0; q < PR; ++q) dot2 = f2_fma(f2_mul(d[q], wv[q]), f2_mul(xv[q], rr2), dot2);
            } else {   // past the row: zeros, so the dweight terms below are zero
                gp[i] = fill<T, V>(from_f32<T>(0.0f));
                xp[i] = gp[i];
            }
        }
        // dweight terms dy * xhat of frame vector i (zero outside the row)
        auto terms = [&](int i, float (&t)[V]) {
            f32x2 d[PR], xv[PR];
            widen16<T>(gp[i], d);
            widen16<T>(xp[i], xv);
#pragma unroll
            for (int q = 0; q < PR; ++q) f2_split(f2_mul(d[q], f2_mul(xv[q], rr2)), t[2 * q], t[2 * q + 1]);
        };
        if (want_dw && lane == 0) {   // thread 0's vector i is also thread T-1's next vector for i - 1
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                float t[V];
                terms(i, t);
#pragma unroll
                for (int j = 0; j < V; ++j) edge[bank][warp][i][j] = t[j];
            }
        }
        // the reduction barrier also publishes `edge`
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

        // dweight: column m*V + j is element j + p of frame vector m (j < V - p)
        // or element j + p - V of frame vector m + 1, held by the next lane
        // (the next warp's first lane for the last lane, thread 0's next
        // vector for the CTA's last thread)
        if (want_dw) {
            with_shift<T>(p, [&](auto Pc) {
                constexpr int PP = decltype(Pc)::value;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    float tw[V];
                    terms(i, tw);
                    float nx[PP + 1];   // elements 0 .. PP-1 of frame vector m + 1
#pragma unroll
                    for (int j = 0; j < PP; ++j) nx[j] = __shfl_down_sync(0xffffffffu, tw[j], 1);
                    if (lane == 31) {
                        const bool last = warp == nwarps - 1;
#pragma unroll
                        for (int j = 0; j < PP; ++j)
                            nx[j] = last ? (i + 1 < NV ? edge[bank][0][i + 1 < NV ? i + 1 : 0][j] : 0.0f)
                                         : edge[bank][warp + 1][i][j];
                    }
#pragma unroll
                    for (int j = 0; j < V; ++j) acc[i][j] += j < V - PP ? tw[j + PP] : nx[j + PP - V];
                }
            });
        }
        bank ^= 1;
    }

    if (want_dw) {
        float *prow = a.partial + (int64_t)blockIdx.x * H;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int m = k0 + i * kstep;
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int c = m * V + j;
                if (c < H) prow[c] = acc[i][j];
            }
        }
    }
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

// At most 512 threads (16 warps: the size of `edge`), 1..4 frame vectors each.
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
