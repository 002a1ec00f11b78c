// bwd_split.cu -- RMSNorm backward for 16-byte aligned rows longer than one
// CTA can hold (above 32 KB), up to 256 KB: a thread-block cluster per row.
//
// The arithmetic is the register-resident backward's (bwd.cu):
//     dot  = sum_h (dy_h * w_h) * (x_h * rrms)
//     dx_h = rrms * (dy_h * w_h - (x_h * rrms) * dot / H)   (+ dres_h)
//     partial[c][h] += dy_h * (x_h * rrms)   for the rows of cluster c
// Each of the CS CTAs of a cluster owns one contiguous column segment of the
// cluster's rows and streams its dy and x (and dres) segments through a ring
// of bulk-copy stages; dot is the sum of the CTAs' partial sums, exchanged
// through distributed shared memory and added in the same order in every
// CTA.  A thread's columns are fixed, so its dweight terms stay in registers
// across all rows of the cluster; at the end each CTA writes its segment of
// the cluster's partial row, and the fixed-order column reduction over the
// clusters' partial rows gives dweight.  The row is read from HBM once,
// where the two-pass form for long rows reads it twice.  With DRES the dres
// segment is not held in registers across the reduction: each thread reads
// it from the stage while it forms dx, and the stage is refilled after a
// CTA barrier at the end of the row (at 32 KB segments the held copy made
// the kernel spill at 128 registers: bf16 H = 32768, 223 -> 171 us).
#include "cluster.cuh"
#include "launch.h"

namespace rmsn {

template <typename T, int NV, bool DRES>
__global__ void __launch_bounds__(512) bwd_split_kernel(BwdArgs a, SplitShape sh) {
    constexpr int VEC = Vec16<T>::n;
    constexpr int PR = Pairs16<T>::n;
    constexpr int NS = DRES ? 3 : 2;
    using P = Pack<T, VEC>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[64];
    __shared__ int64_t stall_rows;   // thread 0: rows issued before it stalled (-1: all)
    __shared__ ClusterXchg xc;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    unsigned char *stages = smem + kRingHeaderBytes;

    // dx may be dy, x or dres itself (in-place calls): not restrict
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    const T *x = static_cast<const T *>(a.x);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *dx = static_cast<T *>(a.dx);
    const uint32_t rank = cluster_rank(), cs = cluster_size();
    const int nvec = a.H / VEC;
    const int seg0 = (int)rank * sh.seg_groups;
    const int nseg = min(sh.seg_groups, nvec - seg0);   // > 0 for every rank (host rule)
    const uint32_t seg_bytes = (uint32_t)nseg * 16u;
    const float ih = 1.0f / (float)a.H;
    const int nst = sh.stages;
    const int64_t NC = cluster_count();
    const int64_t ci = cluster_index();
    const int64_t nrows = (a.M - 1 - ci) / NC + 1;   // the cluster count never exceeds M
    const int64_t col0 = (int64_t)seg0 * VEC;

    auto stage = [&](int s, int j) { return stages + (size_t)(s * NS + j) * sh.seg_pitch; };
    auto issue = [&](int64_t k, int s) {
        const int64_t base = (ci + k * NC) * a.stride + col0;
        mbar_arrive_expect_tx(&full[s], NS * seg_bytes);
        bulk_g2s(stage(s, 0), dy + base, seg_bytes, &full[s]);
        bulk_g2s(stage(s, 1), x + base, seg_bytes, &full[s]);
        if constexpr (DRES) bulk_g2s(stage(s, 2), dres + base, seg_bytes, &full[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        stall_rows = -1;
    }
    xchg_init(xc);
    cluster_sync();   // every CTA's exchange barriers are set up before any partial sum is sent
    // thread 0 issues every copy and arms the exchange barriers
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
        wp[i] = (a.has_w && c < nseg) ? ld_cached<T, VEC>(w + col0 + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
#pragma unroll
        for (int q = 0; q < PR; ++q) acc[i][q] = f2_make(0.0f, 0.0f);
    }

    uint32_t nred = 0;   // cluster reductions so far
    float rr_next = __ldg(a.rrms + ci);
    // stage s = k mod nst and its mbarrier phase (k / nst) mod 2, advanced per row
    int s = 0;
    uint32_t phase = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t base = (ci + k * NC) * a.stride + col0;
        const float rr = rr_next;
        if (k + 1 < nrows) rr_next = __ldg(a.rrms + ci + (k + 1) * NC);
        const f32x2 rr2 = f2_make(rr, rr);
        pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);

        P gp[NV], xp[NV];
        f32x2 dot2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nseg) {
                gp[i] = *reinterpret_cast<const P *>(stage(s, 0) + (size_t)c * 16);
                xp[i] = *reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16);
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
        // the CTA barrier inside the reduction also frees stage s for the row
        // nst ahead: refilled before the other CTAs' partial sums are waited
        // for with 2-byte types (bf16 H = 32768-131072 and f16 H = 24576:
        // 1-2% faster), after it with binary32 (7% slower refilled early at H
        // = 16384); with DRES the dres segment is read from stage s after the
        // reduction, so the stage is refilled only after every thread has
        // read it (below)
        constexpr bool EARLY_REFILL = !DRES && sizeof(T) == 2;
        cluster_push(f2_sum(dot2), red, xc, nred, rank, cs, armer, pw);
        if (EARLY_REFILL && threadIdx.x == 0 && k + nst < nrows) {
            if (!pw.stalled) {   // thread 0 saw stage s's phase complete: refill it
                fence_proxy_async_smem();
                issue(k + nst, s);
            } else if (stall_rows < 0) {
                stall_rows = k + nst;   // rows issued before thread 0 stalled
            }
        }
        const float c_row = cluster_total<RingWaitConst<T>::value>(xc, nred++, cs, a.err, a.wait_polls, armer, pw) * ih;
        if (!DRES && !EARLY_REFILL && threadIdx.x == 0 && k + nst < nrows) {
            if (!pw.stalled) {
                fence_proxy_async_smem();
                issue(k + nst, s);
            } else if (stall_rows < 0) {
                stall_rows = k + nst;
            }
        }
        const float kx = -(rr * rr) * c_row;
        const f32x2 kx2 = f2_make(kx, kx);
        const f32x2 nc2 = f2_make(-c_row, -c_row);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nseg) {
                f32x2 d[PR], xv[PR], wv[PR];
                widen16<T>(gp[i], d);
                widen16<T>(xp[i], xv);
                widen16<T>(wp[i], wv);
                if constexpr (DRES) {   // g * rrms + (x * (-rrms^2 c) + dres)
                    f32x2 rv[PR];
                    widen16<T>(*reinterpret_cast<const P *>(stage(s, 2) + (size_t)c * 16), rv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) d[q] = f2_fma(f2_mul(d[q], wv[q]), rr2, f2_fma(xv[q], kx2, rv[q]));
                } else {                 // rrms * (g + xhat * (-c))
#pragma unroll
                    for (int q = 0; q < PR; ++q)
                        d[q] = f2_mul(rr2, f2_fma(f2_mul(xv[q], rr2), nc2, f2_mul(d[q], wv[q])));
                }
                st_global<T, VEC>(dx + base + (int64_t)c * VEC, narrow16<T>(d));
            }
        }
        if constexpr (DRES) {   // every thread has read its dres groups of stage s
            __syncthreads();
            if (threadIdx.x == 0 && k + nst < nrows) {
                if (!pw.stalled) {
                    fence_proxy_async_smem();
                    issue(k + nst, s);
                } else if (stall_rows < 0) {
                    stall_rows = k + nst;
                }
            }
        }
        if (++s == nst) {
            s = 0;
            phase ^= 1u;
        }
    }

    if (a.partial != nullptr) {   // this CTA's segment of the cluster's partial row
        float *prow = a.partial + ci * a.H + col0;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nseg) {
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
    // no CTA leaves while another may still address its shared memory
    cluster_sync();
}

namespace {

template <typename T, bool DRES>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 2: return reinterpret_cast<const void *>(bwd_split_kernel<T, 2, DRES>);
    case 4: return reinterpret_cast<const void *>(bwd_split_kernel<T, 4, DRES>);
    }
    return nullptr;
}

}  // namespace

const void *bwd_split_kernel_for(int dtype, int nv, bool dres) {
    switch (dtype) {
    case kF32: return dres ? kernel_nv<float, true>(nv) : kernel_nv<float, false>(nv);
    case kF16: return dres ? kernel_nv<__half, true>(nv) : kernel_nv<__half, false>(nv);
    case kBF16: return dres ? kernel_nv<__nv_bfloat16, true>(nv) : kernel_nv<__nv_bfloat16, false>(nv);
    }
    return nullptr;
}

}  // namespace rmsn
