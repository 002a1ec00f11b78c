// fwd_split.cu -- RMSNorm forward (plain, residual-fused, AdaLN) and
// LayerNorm forward for 16-byte aligned rows longer than one CTA can hold
// (above 32 KB: bfloat16 / binary16 H > 16384, binary32 H > 8192), up to
// 256 KB.
//
// A thread-block cluster of CS CTAs (2, 4 or 8) takes one row at a time and
// splits it into CS contiguous column segments of at most 16 KB (32 KB with
// eight CTAs), one per CTA.  Each CTA streams its segment of the cluster's
// rows through a ring of shared-memory stages filled by bulk copies (TMA)
// and kept in registers from the sum of squares to the scale step, exactly
// as the ring kernel does for a whole row; the row's sum is the sum of the
// CTAs' partial sums, exchanged through distributed shared memory behind one
// cluster barrier and added in the same order in every CTA, so every CTA of
// the cluster scales with the same rrms.  The row is read from HBM once, where
// the pages' chunked form for long rows ("Skill: Write a Triton RMSNorm
// Kernel", Required reasoning 11; Kernel design rules, last rule) reads it
// twice.  LayerNorm makes two cluster reductions per row (the sum, then the
// centred sum of squares); AdaLN ("Rocm Kernels" page, 4. AdaLN) stages
// per-token conditioning segments beside x, or keeps w * (1 + scale) and the
// shift of a shared conditioning row in registers.
#include "cluster.cuh"
#include "launch.h"

namespace rmsn {

template <typename T, int NV, int MODE>
__global__ void __launch_bounds__(512) fwd_split_kernel(FwdArgs a, SplitShape sh) {
    constexpr bool RESID = MODE == kResid || MODE == kLnResid;
    constexpr bool LN = MODE == kLn || MODE == kLnResid;
    constexpr bool STAGE_COND = MODE == kAdaln;           // scale/shift segments staged beside x
    constexpr int VEC = Vec16<T>::n;
    constexpr int PR = Pairs16<T>::n;
    constexpr int NS = STAGE_COND ? 3 : (RESID ? 2 : 1);  // segments staged per ring slot
    constexpr bool EARLY_REFILL = sizeof(T) == 2 && MODE == kPlain;   // stage refill before the exchange wait
    using P = Pack<T, VEC>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[64];
    __shared__ int64_t stall_rows;   // thread 0: rows issued before it stalled (-1: all)
    __shared__ ClusterXchg xc;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    unsigned char *stages = smem + kRingHeaderBytes;

    // x and y (the residual and residual_out) may be one array (in-place
    // calls): not restrict
    const T *x = static_cast<const T *>(a.x);
    const T *r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    const T *__restrict__ scale = static_cast<const T *>(a.scale);
    const T *__restrict__ shift = static_cast<const T *>(a.shift);
    const T *__restrict__ bias = static_cast<const T *>(a.b);
    T *y = static_cast<T *>(a.y);
    T *s_out = static_cast<T *>(a.s_out);
    const uint32_t rank = cluster_rank(), cs = cluster_size();
    const int nvec = a.H / VEC;
    const int seg0 = (int)rank * sh.seg_groups;                 // this CTA's first 16-byte group
    const int nseg = min(sh.seg_groups, nvec - seg0);           // > 0 for every rank (host rule)
    const uint32_t seg_bytes = (uint32_t)nseg * 16u;
    const float ih = 1.0f / (float)a.H;
    const int nst = sh.stages;
    const int64_t NC = cluster_count();
    const int64_t ci = cluster_index();
    const int64_t nrows = (a.M - 1 - ci) / NC + 1;   // the cluster count never exceeds M
    const int64_t col0 = (int64_t)seg0 * VEC;        // first column of the segment

    auto stage = [&](int s, int j) { return stages + (size_t)(s * NS + j) * sh.seg_pitch; };
    auto issue = [&](int64_t k, int s) {   // the segment of the cluster's row k into stage s
        const int64_t row = ci + k * NC;
        const int64_t base = row * a.stride + col0;
        mbar_arrive_expect_tx(&full[s], NS * seg_bytes);
        bulk_g2s(stage(s, 0), x + base, seg_bytes, &full[s]);
        if constexpr (RESID) bulk_g2s(stage(s, 1), r + base, seg_bytes, &full[s]);
        if constexpr (STAGE_COND) {
            const int64_t cbase = (int64_t)((uint32_t)row / (uint32_t)a.rows_per_cond) * a.cond_stride + col0;
            bulk_g2s(stage(s, 1), scale + cbase, seg_bytes, &full[s]);
            bulk_g2s(stage(s, 2), shift + cbase, seg_bytes, &full[s]);
        }
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

    // weight of the segment's columns, widened once (ones without weight);
    // with shared conditioning rows w * (1 + scale) of the current one and
    // its shift instead, refreshed when the cluster's row enters another
    f32x2 wv[NV][PR];
    auto load_w = [&](int i) {
        const int c = threadIdx.x + i * blockDim.x;
        return (a.has_w && c < nseg) ? ld_cached<T, VEC>(w + col0 + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
    };
    if constexpr (MODE != kAdalnShared) {
#pragma unroll
        for (int i = 0; i < NV; ++i) widen16<T>(load_w(i), wv[i]);
    }
    P shc[NV];
    int64_t c_next = 0;
    P bp[NV];
    if constexpr (LN) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            bp[i] = (bias != nullptr && c < nseg) ? ld_cached<T, VEC>(bias + col0 + (int64_t)c * VEC)
                                                  : fill<T, VEC>(from_f32<T>(0.0f));
        }
    }

    uint32_t nred = 0;   // cluster reductions so far
    int s = 0;
    uint32_t phase = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t row = ci + k * NC;
        const int64_t base = row * a.stride + col0;
        if constexpr (MODE == kAdalnShared) {
            if (row >= c_next) {
                const uint32_t cr = (uint32_t)row / (uint32_t)a.rows_per_cond;
                c_next = (int64_t)(cr + 1) * a.rows_per_cond;
                const int64_t cbase = (int64_t)cr * a.cond_stride + col0;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int c = threadIdx.x + i * blockDim.x;
                    if (c < nseg) {
                        f32x2 wt[PR], sc[PR];
                        widen16<T>(load_w(i), wt);
                        widen16<T>(ld_cached<T, VEC>(scale + cbase + (int64_t)c * VEC), sc);
#pragma unroll
                        for (int q = 0; q < PR; ++q) wv[i][q] = f2_fma(wt[q], sc[q], wt[q]);   // w * (1 + scale)
                        shc[i] = ld_cached<T, VEC>(shift + cbase + (int64_t)c * VEC);
                    }
                }
            }
        }
        pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);

        f32x2 sv[NV][PR];
        P scp[NV], shp[NV];
        f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nseg) {
                widen16<T>(*reinterpret_cast<const P *>(stage(s, 0) + (size_t)c * 16), sv[i]);
                if constexpr (RESID) {
                    f32x2 rv[PR];
                    widen16<T>(*reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16), rv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[i][q] = f2_add(sv[i][q], rv[q]);
                    st_global<T, VEC>(s_out + base + (int64_t)c * VEC, narrow16<T>(sv[i]));
                }
                if constexpr (STAGE_COND) {
                    scp[i] = *reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16);
                    shp[i] = *reinterpret_cast<const P *>(stage(s, 2) + (size_t)c * 16);
                }
                if constexpr (LN) {
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_add(ss2, sv[i][q]);
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[i][q], sv[i][q], ss2);
                }
            }
        }
        // the CTA barrier inside the reduction also means every thread of this
        // CTA has copied stage s out, so it can be refilled: before the other
        // CTAs' partial sums are waited for in the 2-byte plain norm, whose one
        // staged stream leaves the ring short of bytes in flight (bf16 H =
        // 32768-131072: 5-7% faster), after it elsewhere (fused bf16 H =
        // 32768 / 65536 and fp32: 2-7% slower refilled early)
        cluster_push(f2_sum(ss2), red, xc, nred, rank, cs, armer, pw);
        if constexpr (EARLY_REFILL) {
            if (threadIdx.x == 0 && k + nst < nrows) {
                if (!pw.stalled) {   // thread 0 saw stage s's phase complete: refill it
                    fence_proxy_async_smem();
                    issue(k + nst, s);
                } else if (stall_rows < 0) {
                    stall_rows = k + nst;   // rows issued before thread 0 stalled
                }
            }
        }
        float total = cluster_total<RingWaitConst<T>::value>(xc, nred++, cs, a.err, a.wait_polls, armer, pw);
        if constexpr (!EARLY_REFILL) {
            if (threadIdx.x == 0 && k + nst < nrows) {
                if (!pw.stalled) {
                    fence_proxy_async_smem();
                    issue(k + nst, s);
                } else if (stall_rows < 0) {
                    stall_rows = k + nst;
                }
            }
        }
        float mu = 0.0f;
        if constexpr (LN) {
            mu = total * ih;
            const f32x2 nm2 = f2_make(-mu, -mu);
            ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * blockDim.x;
                if (c < nseg) {
#pragma unroll
                    for (int q = 0; q < PR; ++q) {
                        sv[i][q] = f2_add(sv[i][q], nm2);
                        ss2 = f2_fma(sv[i][q], sv[i][q], ss2);
                    }
                }
            }
            total = cluster_sum<RingWaitConst<T>::value>(f2_sum(ss2), red, xc, nred++, rank, cs, a.err, a.wait_polls, armer, pw);
        }
        const float rrms = rsqrtf(total * ih + a.eps);
        if (rank == 0 && threadIdx.x == 0) {
            if (a.rrms != nullptr) a.rrms[row] = rrms;
            if constexpr (LN)
                if (a.mean != nullptr) a.mean[row] = mu;
        }
        const f32x2 rr2 = f2_make(rrms, rrms);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nseg) {
                f32x2 yv[PR];
                if constexpr (MODE == kAdalnShared) {
                    f32x2 shv[PR];
                    widen16<T>(shc[i], shv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_fma(f2_mul(sv[i][q], rr2), wv[i][q], shv[q]);
                } else if constexpr (LN) {
                    f32x2 bv[PR];
                    widen16<T>(bp[i], bv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_fma(f2_mul(sv[i][q], rr2), wv[i][q], bv[q]);
                } else if constexpr (STAGE_COND) {   // (s * rrms) * (w * (1 + scale)) + shift
                    f32x2 sc[PR], shv[PR];
                    widen16<T>(scp[i], sc);
                    widen16<T>(shp[i], shv);
#pragma unroll
                    for (int q = 0; q < PR; ++q)
                        yv[q] = f2_fma(f2_mul(sv[i][q], rr2), f2_fma(wv[i][q], sc[q], wv[i][q]), shv[q]);
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_mul(f2_mul(sv[i][q], rr2), wv[i][q]);
                }
                st_global<T, VEC>(y + base + (int64_t)c * VEC, narrow16<T>(yv));
            }
        }
        if (++s == nst) {
            s = 0;
            phase ^= 1u;
        }
    }
    // Only a stalled CTA can exit with copies in flight: thread 0 gives the
    // last issued phase of every stage one more bounded wait.
    if (pw.stalled) drain_ring(full, nst, stall_rows < 0 ? nrows : stall_rows);
    // no CTA leaves while another may still address its shared memory
    cluster_sync();
}

namespace {

template <typename T, int MODE>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 2: return reinterpret_cast<const void *>(fwd_split_kernel<T, 2, MODE>);
    case 4: return reinterpret_cast<const void *>(fwd_split_kernel<T, 4, MODE>);
    }
    return nullptr;
}

template <typename T>
const void *kernel_mode(int mode, int nv) {
    switch (mode) {
    case kPlain: return kernel_nv<T, kPlain>(nv);
    case kResid: return kernel_nv<T, kResid>(nv);
    case kAdaln: return kernel_nv<T, kAdaln>(nv);
    case kAdalnShared: return kernel_nv<T, kAdalnShared>(nv);
    case kLn: return kernel_nv<T, kLn>(nv);
    case kLnResid: return kernel_nv<T, kLnResid>(nv);
    }
    return nullptr;
}

const void *kernel_for(int dtype, int mode, int nv) {
    switch (dtype) {
    case kF32: return kernel_mode<float>(mode, nv);
    case kF16: return kernel_mode<__half>(mode, nv);
    case kBF16: return kernel_mode<__nv_bfloat16>(mode, nv);
    }
    return nullptr;
}

}  // namespace

bool plan_fwd_split(int64_t M, int H, int dtype, int mode, int sm_count, SplitPlan *out) {
    SplitPlan p{};
    const int streams = mode == kAdaln ? 3 : ((mode == kResid || mode == kLnResid) ? 2 : 1);
    if (!split_geometry(H, dtype, streams, false, &p)) return false;
    const void *k = kernel_for(dtype, mode, p.nv);
    if (k == nullptr) return false;
    return finish_split_plan(k, M, sm_count, &p) && (*out = p, true);
}

cudaError_t launch_fwd_split(const FwdArgs &a, int dtype, int mode, const SplitPlan &p, cudaStream_t st) {
    const void *k = kernel_for(dtype, mode, p.nv);
    if (k == nullptr) return cudaErrorInvalidValue;
    FwdArgs args = a;
    SplitShape shape = p.shape;
    void *params[] = {&args, &shape};
    return launch_cluster(k, p, params, st);
}

}  // namespace rmsn
