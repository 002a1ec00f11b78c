// bwd_ring.cu -- RMSNorm backward with the dy and x rows staged in shared
// memory by bulk copies (TMA), for 16-byte aligned rows.
//
// Same arithmetic as the register-resident backward kernel (bwd.cu):
//     dot  = sum_h (dy_h * w_h) * (x_h * rrms)          (CTA reduction)
//     dx_h = rrms * (dy_h * w_h - (x_h * rrms) * dot / H)  (+ dres_h, DRES)
//     partial[b][h] += dy_h * (x_h * rrms)               (CTA b's rows)
// With DRES (the backward of the residual-fused forward) a third row, the
// gradient arriving through residual_out, is staged and added to dx.
// but the rows arrive through a ring of NST shared-memory stages kept full by
// one thread's cp.async.bulk copies (mbarrier byte counts), so the next rows
// stream in from HBM while the current one is reduced and written.  The
// thread-to-column map is fixed, so each thread keeps its dweight partials
// for its columns in registers across all rows of its CTA.  A thread keeps
// its packed dy and x groups in registers across the reduction barrier, so
// the stage is refilled right after that barrier (measured faster than
// re-reading the stage after the barrier and refilling one row later).
#include "bulk.cuh"
#include "launch.h"

namespace rmsn {

// Register budget per thread: the two-group variants (up to 384 threads)
// are held to 80 registers, so three CTAs of 256 threads fit an SM -- without
// spills that measured fastest (78 registers against 64 with spills at four
// CTAs: 94.5% against 93.9% of the copy peak on the default step); the other
// variants measured fastest with ptxas's own choice.
constexpr int bwd_ring_max_regs(int nv) { return nv == 2 ? 80 : 128; }

template <typename T, int NV, bool DRES>
__global__ void __launch_bounds__(512) __maxnreg__(bwd_ring_max_regs(NV)) bwd_ring_kernel(BwdArgs a, RingShape rs) {
    constexpr int VEC = Vec16<T>::n;
    constexpr int PR = Pairs16<T>::n;
    constexpr int NS = DRES ? 3 : 2;   // streams staged per row: dy, x (and dres)
    using P = Pack<T, VEC>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[64];
    __shared__ int64_t stall_rows;   // thread 0: rows issued before it stalled (-1: all)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    unsigned char *stages = smem + kRingHeaderBytes;

    // dx may be dy, x or dres itself (in-place calls): not restrict
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    const T *x = static_cast<const T *>(a.x);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *dx = static_cast<T *>(a.dx);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H
    constexpr int nst = kBwdRingStages;   // rs.stages is the same value
    const int64_t G = gridDim.x;
    const int64_t nrows = (a.M - 1 - blockIdx.x) / G + 1;  // the grid never exceeds M

    auto stage = [&](int s, int j) { return stages + (size_t)(s * NS + j) * rs.row_pitch; };
    auto issue = [&](int64_t k, int s) {   // row k of this CTA into stage s (= k mod nst)
        const int64_t base = (blockIdx.x + k * G) * a.stride;
        mbar_arrive_expect_tx(&full[s], NS * rs.row_bytes);
        bulk_g2s(stage(s, 0), dy + base, rs.row_bytes, &full[s]);
        bulk_g2s(stage(s, 1), x + base, rs.row_bytes, &full[s]);
        if constexpr (DRES) bulk_g2s(stage(s, 2), dres + base, rs.row_bytes, &full[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        stall_rows = -1;
        // the time-out test (hold_first): wait for row 0 before any copy is
        // issued, so the wait runs out with nothing in flight
        if (a.hold_first) wait_unarmed(&full[0], a.err, a.wait_polls);
    }
    __syncthreads();
    // thread 0 issues every copy
    // thread 0 arms the barriers; its waits run to kWaitPolls (see bulk.cuh)
    const bool armer = threadIdx.x == 0;
    PipeWait pw = pipe_wait_init(a.wait_polls, armer);
    if (threadIdx.x == 0)
        for (int k = 0; k < nst && k < nrows; ++k) issue(k, k);

    P wp[NV];
    f32x2 acc[NV][PR];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        wp[i] = (a.has_w && c < nvec) ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
#pragma unroll
        for (int q = 0; q < PR; ++q) acc[i][q] = f2_make(0.0f, 0.0f);
    }

    int bank = 0;
    float rr_next = __ldg(a.rrms + blockIdx.x);
    for (int64_t k = 0; k < nrows; ++k) {
        // stage s = k mod nst and its mbarrier phase (k / nst) mod 2 (nst is
        // a power-of-two constant: a mask and a shift)
        const int s = (int)((uint32_t)k % (uint32_t)nst);
        const uint32_t phase = ((uint32_t)k / (uint32_t)nst) & 1u;
        const int64_t base = (blockIdx.x + k * G) * a.stride;
        const float rr = rr_next;
        if (k + 1 < nrows) rr_next = __ldg(a.rrms + blockIdx.x + (k + 1) * G);
        const f32x2 rr2 = f2_make(rr, rr);
        pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);

        P gp[NV], xp[NV], rp[NV];
        f32x2 dot2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                gp[i] = *reinterpret_cast<const P *>(stage(s, 0) + (size_t)c * 16);
                xp[i] = *reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16);
                if constexpr (DRES) rp[i] = *reinterpret_cast<const P *>(stage(s, 2) + (size_t)c * 16);
                f32x2 d[PR], xv[PR], wv[PR];
                widen16<T>(gp[i], d);
                widen16<T>(xp[i], xv);
                widen16<T>(wp[i], wv);
#pragma unroll
                for (int q = 0; q < PR; ++q) {
                    const f32x2 xh = f2_mul(xv[q], rr2);
                    dot2 = f2_fma(f2_mul(d[q], wv[q]), xh, dot2);
                    acc[i][q] = f2_fma(d[q], xh, acc[i][q]);
                }
            }
        }
        // the reduction barrier also frees stage s for the row nst ahead
        const float c_row = block_sum(f2_sum(dot2), red, bank) * ih;
        bank ^= 1;
        if (threadIdx.x == 0 && k + nst < nrows) {
            if (!pw.stalled) {   // thread 0 saw stage s's phase complete: refill it
                fence_proxy_async_smem();
                issue(k + nst, s);
            } else if (stall_rows < 0) {
                stall_rows = k + nst;   // rows issued before thread 0 stalled
            }
        }
        // dx = rrms * (g - xhat * c).  With DRES it is evaluated as
        // g * rrms + (x * (-rrms^2 c) + dres), the residual stream's gradient
        // riding in the addend (measured faster there); without, as
        // rrms * (g + xhat * (-c)) (measured faster there).
        const float kx = -(rr * rr) * c_row;
        const f32x2 kx2 = f2_make(kx, kx);
        const f32x2 nc2 = f2_make(-c_row, -c_row);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
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
                st_global<T, VEC>(dx + base + (int64_t)c * VEC, narrow16<T>(d));
            }
        }
    }

    if (a.partial != nullptr) {
        float *prow = a.partial + (int64_t)blockIdx.x * a.H;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
#pragma unroll
                for (int q = 0; q < PR; q += 2) {
                    float a0, a1, a2, a3;
                    f2_split(acc[i][q], a0, a1);
                    f2_split(acc[i][q + 1], a2, a3);
                    *reinterpret_cast<float4 *>(prow + (int64_t)c * VEC + 2 * q) = make_float4(a0, a1, a2, a3);
                }
            }
        }
    }
    // Only a stalled CTA can exit with copies in flight: thread 0 gives the
    // last issued phase of every stage one more bounded wait.
    if (pw.stalled) drain_ring(full, nst, stall_rows < 0 ? nrows : stall_rows);
    allow_dependent_launch();
}

namespace {

template <typename T, bool DRES>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 1: return reinterpret_cast<const void *>(bwd_ring_kernel<T, 1, DRES>);
    case 2: return reinterpret_cast<const void *>(bwd_ring_kernel<T, 2, DRES>);
    case 3: return reinterpret_cast<const void *>(bwd_ring_kernel<T, 3, DRES>);
    case 4: return reinterpret_cast<const void *>(bwd_ring_kernel<T, 4, DRES>);
    }
    return nullptr;
}

}  // namespace

const void *bwd_ring_kernel_for(int dtype, int nv, bool dres) {
    switch (dtype) {
    case kF32: return dres ? kernel_nv<float, true>(nv) : kernel_nv<float, false>(nv);
    case kF16: return dres ? kernel_nv<__half, true>(nv) : kernel_nv<__half, false>(nv);
    case kBF16: return dres ? kernel_nv<__nv_bfloat16, true>(nv) : kernel_nv<__nv_bfloat16, false>(nv);
    }
    return nullptr;
}

}  // namespace rmsn
