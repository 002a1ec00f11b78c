// fwd_ring.cu -- RMSNorm forward (plain, residual-fused, AdaLN) and
// LayerNorm forward with rows staged in shared memory by bulk copies (TMA),
// for 16-byte aligned rows of LLM hidden sizes (from 4 KB with one input
// stream, 8 KB with two or three).
//
// Persistent grid: CTA b owns rows b, b + G, b + 2G, ...  A ring of NST
// shared-memory stages, each holding one row of x (and of the residual, or
// the row's AdaLN scale and shift), is kept full by one thread issuing
// cp.async.bulk copies whose completion is counted by an mbarrier per stage.
// So up to NST rows per CTA are in flight from HBM while the CTA computes,
// independently of the register budget.  Each thread copies its NV 16-byte
// column groups from the stage into registers, forms s = x (+ residual) in
// binary32 (two lanes per f32x2 instruction), writes residual_out, reduces
// sum(s^2) over the CTA, and writes y = (s * rrms) * w from registers: the
// row is read from HBM once ("Skill: Write a Triton RMSNorm Kernel",
// Required reasoning 3-10; Performance requirements).  AdaLN ("Rocm
// Kernels" page, 4. AdaLN) is evaluated as (s * rrms) * (w * (1 + scale)) +
// shift in every kernel, with w * (1 + scale) = fma(w, scale, w) (rounded
// once) and the last multiply and add fused, so conditioning shared by rows
// gives the bits of the same rows repeated: per-token
// conditioning rows are staged beside x; conditioning rows shared by many
// rows (one per sequence) are read through L1 only when the CTA's row moves
// to another one, and kept as w * (1 + scale) and shift in registers, so a
// row costs one fused multiply-add per element more than the plain norm.
// LayerNorm (kLn, kLnResid) reduces the row twice from the same registers:
// the sum for the mean, then the centred sum of squares; y = ((s - mean) *
// rstd) * w + b.  The stage is refilled with row k + NST as soon as the
// first reduction barrier shows every thread has copied it out.
#include "bulk.cuh"
#include "launch.h"

namespace rmsn {

// Register budget per thread, from the measured geometry: two-group
// kernels run up to 1024 threads per SM with one input row per slot (8 CTAs
// of 128 at 4 KB rows, 4 of 256 at 8 KB, 2 of 512 at 16 KB) and with fused
// LayerNorm (4 of 256 at 8 KB): 64 registers; fused RMSNorm and per-token
// AdaLN at most 768 (2 or 3 CTAs of 256-384): 80.  Four-group kernels run
// one CTA of up to 512 threads.
constexpr int fwd_ring_max_regs(int nv, int mode) {
    return nv == 2 ? ((mode == kResid || mode == kAdaln) ? 80 : 64) : 128;
}

template <typename T, int NV, int MODE>
__global__ void __launch_bounds__(512) __maxnreg__(fwd_ring_max_regs(NV, MODE))
    fwd_ring_kernel(FwdArgs a, RingShape rs) {
    constexpr bool RESID = MODE == kResid || MODE == kLnResid;
    constexpr bool ADALN = MODE == kAdaln || MODE == kAdalnShared;
    constexpr bool LN = MODE == kLn || MODE == kLnResid;
    constexpr bool STAGE_COND = MODE == kAdaln;           // scale/shift rows staged beside x
    constexpr int VEC = Vec16<T>::n;
    constexpr int PR = Pairs16<T>::n;                     // binary32 pairs per 16-byte group
    constexpr int NS = STAGE_COND ? 3 : (RESID ? 2 : 1);  // rows staged per ring slot
    using P = Pack<T, VEC>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[64];
    __shared__ int64_t stall_rows;   // thread 0: rows issued before it stalled (-1: all)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    unsigned char *stages = smem + kRingHeaderBytes;

    // x and y (the residual and residual_out) may be one array (in-place
    // calls), so they are not declared restrict; weight, bias and
    // conditioning rows are never written by any call
    const T *x = static_cast<const T *>(a.x);
    const T *r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    const T *__restrict__ scale = static_cast<const T *>(a.scale);
    const T *__restrict__ shift = static_cast<const T *>(a.shift);
    const T *__restrict__ bias = static_cast<const T *>(a.b);
    T *y = static_cast<T *>(a.y);
    T *s_out = static_cast<T *>(a.s_out);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H
    const int nst = rs.stages;
    // CTA b takes rows r0, r0 + G, r0 + 2G, ... (r0 = b; the grid never
    // exceeds M).  Shared AdaLN conditioning with cond_groups > 0 instead
    // splits the grid into one group of CTAs per conditioning row, sized in
    // proportion to its rows (CTAs [c R / M, (c + 1) R / M) for conditioning
    // row c, R = rows_per_cond x grid; the host gives each group four CTAs or
    // more, the last one at least one): each CTA strides through its own
    // conditioning row's rows only, so it reads one conditioning row, at its
    // start.  With the plain stride every CTA crosses each boundary at the
    // same time and all of them stall on the same lines together (about 1 us
    // per boundary at bf16 12288 x 2048).
    int64_t G = gridDim.x, r0 = blockIdx.x, r_end = a.M;
    if constexpr (MODE == kAdalnShared) {
        if (a.cond_groups > 0) {
            const int64_t n = a.cond_groups, b = blockIdx.x, g = gridDim.x;
            const int64_t R = a.rows_per_cond * g;
            int64_t c = ((b + 1) * a.M - 1) / R;              // this CTA's conditioning row
            if (c > n - 1) c = n - 1;
            const int64_t first = c * R / a.M;                 // the group's CTAs: [first, next)
            const int64_t next = c == n - 1 ? g : (c + 1) * R / a.M;
            G = next - first;
            r0 = c * a.rows_per_cond + (b - first);
            r_end = min((c + 1) * a.rows_per_cond, a.M);
        }
    }
    const int64_t nrows = r0 < r_end ? (r_end - 1 - r0) / G + 1 : 0;

    auto stage = [&](int s, int j) { return stages + (size_t)(s * NS + j) * rs.row_pitch; };
    auto issue = [&](int64_t k, int s) {   // row k of this CTA into stage s (= k mod nst)
        const int64_t row = r0 + k * G;
        const int64_t base = row * a.stride;
        mbar_arrive_expect_tx(&full[s], NS * rs.row_bytes);
        bulk_g2s(stage(s, 0), x + base, rs.row_bytes, &full[s]);
        if constexpr (RESID) bulk_g2s(stage(s, 1), r + base, rs.row_bytes, &full[s]);
        if constexpr (STAGE_COND) {
            const int64_t cbase = (int64_t)((uint32_t)row / (uint32_t)a.rows_per_cond) * a.cond_stride;
            bulk_g2s(stage(s, 1), scale + cbase, rs.row_bytes, &full[s]);
            bulk_g2s(stage(s, 2), shift + cbase, rs.row_bytes, &full[s]);
        }
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

    // weight (H,), by column only, widened once per CTA; ones without weight.
    // With shared conditioning rows wv holds w * (1 + scale) of the current
    // conditioning row instead, and shc its shift: refreshed only when the
    // CTA's next row belongs to another conditioning row.  The refresh loads
    // are issued before the row's stage wait and w * (1 + scale) is formed
    // after it, so their latency hides behind the wait (bf16 12288 x 2048,
    // one conditioning row: the first row of a CTA was ready about 1 us later
    // than in the plain norm when the product was formed before the wait).
    f32x2 wv[NV][PR];
    auto load_w = [&](int i) {
        const int c = threadIdx.x + i * blockDim.x;
        return (a.has_w && c < nvec) ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
    };
    if constexpr (MODE != kAdalnShared) {
#pragma unroll
        for (int i = 0; i < NV; ++i) widen16<T>(load_w(i), wv[i]);
    }
    P shc[NV];
    int64_t c_next = 0;   // first row of the next conditioning row: refresh when reached
    P bp[NV];   // LayerNorm bias, kept packed; zeros without one
    if constexpr (LN) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            bp[i] = (bias != nullptr && c < nvec) ? ld_cached<T, VEC>(bias + (int64_t)c * VEC)
                                                  : fill<T, VEC>(from_f32<T>(0.0f));
        }
    }

    int bank = 0;
    // stage s = k mod nst and its mbarrier phase = (k / nst) mod 2, advanced
    // per row (no division in the loop)
    int s = 0;
    uint32_t phase = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t row = r0 + k * G;
        const int64_t base = row * a.stride;
        if constexpr (MODE != kAdalnShared) {
            pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);
        } else {
            // rows of a CTA only increase: divide only when a boundary is passed
            // (the same in every thread)
            if (row >= c_next) {
                // the new conditioning row's weight and scale, packed; every
                // thread sets all of wv and shc (columns past the row: w = 1,
                // scale = shift = 0, never stored), so the old ones are dead here
                P wpk[NV], scpk[NV];
                const uint32_t cr = (uint32_t)row / (uint32_t)a.rows_per_cond;
                c_next = (int64_t)(cr + 1) * a.rows_per_cond;
                const int64_t cbase = (int64_t)cr * a.cond_stride;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int c = threadIdx.x + i * blockDim.x;
                    const bool in = c < nvec;
                    wpk[i] = load_w(i);
                    scpk[i] = in ? ld_cached<T, VEC>(scale + cbase + (int64_t)c * VEC) : fill<T, VEC>(from_f32<T>(0.0f));
                    shc[i] = in ? ld_cached<T, VEC>(shift + cbase + (int64_t)c * VEC) : fill<T, VEC>(from_f32<T>(0.0f));
                }
                pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    f32x2 wt[PR], sc[PR];
                    widen16<T>(wpk[i], wt);
                    widen16<T>(scpk[i], sc);
#pragma unroll
                    for (int q = 0; q < PR; ++q) wv[i][q] = f2_fma(wt[q], sc[q], wt[q]);   // w * (1 + scale)
                }
            } else {
                pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);
            }
        }

        // s = x (+ residual) in binary32, kept in registers for the scale step;
        // the post-add sum is written back as the next residual stream
        f32x2 sv[NV][PR];
        P scp[NV], shp[NV];
        f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                widen16<T>(*reinterpret_cast<const P *>(stage(s, 0) + (size_t)c * 16), sv[i]);
                if constexpr (RESID) {
                    f32x2 rv[PR];
                    widen16<T>(*reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16), rv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[i][q] = f2_add(sv[i][q], rv[q]);
                    st_global<T, VEC>(s_out + base + (int64_t)c * VEC, narrow16<T>(sv[i]));
                }
                if constexpr (STAGE_COND) {   // out of the stage before the barrier frees it
                    scp[i] = *reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16);
                    shp[i] = *reinterpret_cast<const P *>(stage(s, 2) + (size_t)c * 16);
                }
                if constexpr (LN) {   // LayerNorm: the plain sum first (the mean)
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_add(ss2, sv[i][q]);
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[i][q], sv[i][q], ss2);
                }
            }
        }
        // the barrier inside the reduction also means every thread has
        // copied stage s out, so it can be refilled
        float total = block_sum(f2_sum(ss2), red, bank);
        bank ^= 1;
        if (threadIdx.x == 0 && k + nst < nrows) {
            if (!pw.stalled) {   // thread 0 saw stage s's phase complete: refill it
                fence_proxy_async_smem();
                issue(k + nst, s);
            } else if (stall_rows < 0) {
                stall_rows = k + nst;   // rows issued before thread 0 stalled
            }
        }
        float mu = 0.0f;
        if constexpr (LN) {   // centre the row held in registers: s <- s - mean, then its sum of squares
            mu = total * ih;
            const f32x2 nm2 = f2_make(-mu, -mu);
            ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * blockDim.x;
                if (c < nvec) {
#pragma unroll
                    for (int q = 0; q < PR; ++q) {
                        sv[i][q] = f2_add(sv[i][q], nm2);
                        ss2 = f2_fma(sv[i][q], sv[i][q], ss2);
                    }
                }
            }
            total = block_sum(f2_sum(ss2), red, bank);
            bank ^= 1;
        }
        const float rrms = rsqrtf(total * ih + a.eps);   // LayerNorm: rstd of the centred row
        if (threadIdx.x == 0) {
            if (a.rrms != nullptr) a.rrms[row] = rrms;
            if constexpr (LN)
                if (a.mean != nullptr) a.mean[row] = mu;
        }
        const f32x2 rr2 = f2_make(rrms, rrms);
        // y = (s * rrms) * w [AdaLN: (s * rrms) * (w * (1 + scale)) + shift], one rounding to the storage type
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                f32x2 yv[PR];
                if constexpr (MODE == kAdalnShared) {   // (s * rrms) * (w * (1 + scale)) + shift
                    f32x2 sh[PR];
                    widen16<T>(shc[i], sh);
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_fma(f2_mul(sv[i][q], rr2), wv[i][q], sh[q]);
                } else if constexpr (LN) {   // ((s - mean) * rstd) * w + b
                    f32x2 bv[PR];
                    widen16<T>(bp[i], bv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_fma(f2_mul(sv[i][q], rr2), wv[i][q], bv[q]);
                } else if constexpr (STAGE_COND) {   // (s * rrms) * (w * (1 + scale)) + shift
                    f32x2 sc[PR], sh[PR];
                    widen16<T>(scp[i], sc);
                    widen16<T>(shp[i], sh);
#pragma unroll
                    for (int q = 0; q < PR; ++q)
                        yv[q] = f2_fma(f2_mul(sv[i][q], rr2), f2_fma(wv[i][q], sc[q], wv[i][q]), sh[q]);
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
}

namespace {

template <typename T, int NV, int MODE>
cudaError_t launch_t(const FwdArgs &a, const RingPlan &p, cudaStream_t st) {
    auto k = fwd_ring_kernel<T, NV, MODE>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(k), p.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_kernel(k, (unsigned)p.grid, (unsigned)p.threads, p.smem_bytes, st, a, p.shape);
}

// The ring geometry takes two or four 16-byte groups per thread.
template <typename T, int MODE>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 2: return reinterpret_cast<const void *>(fwd_ring_kernel<T, 2, MODE>);
    case 4: return reinterpret_cast<const void *>(fwd_ring_kernel<T, 4, MODE>);
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

template <typename T, int MODE>
cudaError_t launch_nv(const FwdArgs &a, const RingPlan &p, cudaStream_t st) {
    switch (p.nv) {
    case 2: return launch_t<T, 2, MODE>(a, p, st);
    case 4: return launch_t<T, 4, MODE>(a, p, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dt(const FwdArgs &a, int mode, const RingPlan &p, cudaStream_t st) {
    switch (mode) {
    case kPlain: return launch_nv<T, kPlain>(a, p, st);
    case kResid: return launch_nv<T, kResid>(a, p, st);
    case kAdaln: return launch_nv<T, kAdaln>(a, p, st);
    case kAdalnShared: return launch_nv<T, kAdalnShared>(a, p, st);
    case kLn: return launch_nv<T, kLn>(a, p, st);
    case kLnResid: return launch_nv<T, kLnResid>(a, p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool plan_fwd_ring(int64_t M, int H, int dtype, int mode, int sm_count, RingPlan *out) {
    RingPlan p{};
    if (!fwd_ring_geometry(H, dtype, mode, &p)) return false;
    const void *k = kernel_for(dtype, mode, p.nv);
    if (k == nullptr || allow_dynamic_smem(k, p.smem_bytes) != cudaSuccess) return false;
    int occ = occupancy(k, p.threads, p.smem_bytes);
    if (occ <= 0) return false;
    if (p.max_ctas_per_sm > 0 && occ > p.max_ctas_per_sm) occ = p.max_ctas_per_sm;
    const int64_t cap = (int64_t)occ * sm_count;
    p.grid = (int)(M < cap ? M : cap);
    *out = p;
    return true;
}

cudaError_t launch_fwd_ring(const FwdArgs &a, int dtype, int mode, const RingPlan &p, cudaStream_t st) {
    switch (dtype) {
    case kF32: return launch_dt<float>(a, mode, p, st);
    case kF16: return launch_dt<__half>(a, mode, p, st);
    case kBF16: return launch_dt<__nv_bfloat16>(a, mode, p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
