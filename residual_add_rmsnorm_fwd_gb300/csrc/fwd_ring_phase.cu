// fwd_ring_phase.cu -- RMSNorm forward (plain, residual-fused) and LayerNorm
// forward with rows staged by bulk copies, for rows of 4-32 KB that are not
// 16-byte aligned but whose matrices share one alignment phase (phase.cuh).
//
// The bulk-copy ring of fwd_ring.cu in each row's aligned frame: the copy of
// a row covers its frame, the 16-byte granules from the one holding column 0
// to the one holding column H - 1 (a granule lies inside the allocation that
// holds any of its bytes, as allocations start and end on 16-byte
// boundaries; the bytes outside the row are loaded and never used: they are
// zeroed in registers before any arithmetic).  The stage then holds frame
// vector k at byte 16 k, so every thread takes whole 16-byte vectors from
// it, and writes whole vectors back except the row's first and last, which
// are written element by element (never outside the row).  The weight and
// bias are cut out of their own aligned vectors by the row's shift
// (reloaded only when the phase changes from one of the CTA's rows to the
// next).  Everything else -- persistent grid, one thread issuing the copies,
// bounded mbarrier waits, the stage refilled after the reduction barrier --
// is the aligned ring's ("Skill: Write a Triton RMSNorm Kernel", Required
// reasoning 3-10; Performance requirements).
#include "bulk.cuh"
#include "launch.h"
#include "phase.cuh"

namespace rmsn {

// Register budget: as the aligned ring's two-group kernels (64, or 80 with
// two staged streams); four-group kernels run one CTA of up to 512 threads.
constexpr int fwd_ring_phase_max_regs(int nv, int mode) {
    return nv == 2 ? ((mode == kResid || mode == kLnResid) ? 80 : 64) : 128;
}

template <typename T, int NV, int MODE>
__global__ void __launch_bounds__(512) __maxnreg__(fwd_ring_phase_max_regs(NV, MODE))
    fwd_ring_phase_kernel(FwdArgs a, RingShape rs) {
    constexpr bool RESID = MODE == kResid || MODE == kLnResid;
    constexpr bool LN = MODE == kLn || MODE == kLnResid;
    constexpr int V = 16 / sizeof(T);
    constexpr int PR = V / 2;
    constexpr int NS = RESID ? 2 : 1;   // rows staged per ring slot
    using P = Pack<T, V>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[64];
    __shared__ int64_t stall_rows;   // the issuer: rows issued before it stalled (-1: all)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    unsigned char *stages = smem + kRingHeaderBytes;

    // x and y (the residual and residual_out) may be one array (in-place
    // calls): not restrict
    const T *x = static_cast<const T *>(a.x);
    const T *r = static_cast<const T *>(a.r);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    const T *__restrict__ bias = static_cast<const T *>(a.b);
    T *y = static_cast<T *>(a.y);
    T *s_out = static_cast<T *>(a.s_out);
    const int H = a.H;
    const float ih = 1.0f / (float)H;   // one division per CTA; exact for power-of-two H
    const int nst = rs.stages;
    const int qw = a.has_w ? elem_phase(w) : 0;
    const int qb = (LN && bias != nullptr) ? elem_phase(bias) : 0;
    const int k0 = threadIdx.x, kstep = blockDim.x;
    const int64_t G = gridDim.x, r0 = blockIdx.x;
    const int64_t nrows = (a.M - 1 - r0) / G + 1;   // the grid never exceeds M

    auto stage = [&](int s, int j) { return stages + (size_t)(s * NS + j) * rs.row_pitch; };
    auto issue = [&](int64_t k, int s) {   // row k of this CTA's frame into stage s (= k mod nst)
        const int64_t base = (r0 + k * G) * a.stride;
        const int p = elem_phase(x + base);
        const uint32_t bytes = (uint32_t)((p + H + V - 1) / V) * 16u;
        mbar_arrive_expect_tx(&full[s], NS * bytes);
        bulk_g2s(stage(s, 0), x + base - p, bytes, &full[s]);
        if constexpr (RESID) bulk_g2s(stage(s, 1), r + base - p, bytes, &full[s]);
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
    // one thread issues every copy and arms the barriers; its waits run to
    // kWaitPolls (see bulk.cuh).  It is the second warp's first thread, so
    // the extra work of slot 0 (the row's first and last columns, thread 0)
    // does not delay the refills.
    const int issuer = blockDim.x > 32 ? 32 : 0;
    const bool armer = threadIdx.x == issuer;
    PipeWait pw = pipe_wait_init(a.wait_polls, armer);
    if (armer)
        for (int k = 0; k < nst && k < nrows; ++k) issue(k, k);

    const int ns = frame_slots<T>(H);   // slots: as many as 16-byte vectors of an aligned row
    P wp[NV], bp[NV];   // weight (bias) windows of phase p_w
    int p_w = -1;
    int bank = 0;
    int s = 0;
    uint32_t phase = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t row = r0 + k * G;
        const int64_t base = row * a.stride;
        const int p = elem_phase(x + base);
        const bool wrap = row_wraps<T>(p, H);
        pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);

        // s = x (+ residual) in binary32; the frame's bytes outside the row are zeroed
        f32x2 sv[NV][PR];
        f32x2 ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = k0 + i * kstep;
            if (c < ns) {
                const bool inner = c != 0 && c != ns - 1;   // only slots 0 and ns - 1 reach outside the row
                P xv, rv;
                if (inner) {
                    xv = *reinterpret_cast<const P *>(stage(s, 0) + (size_t)c * 16);
                    if constexpr (RESID) rv = *reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16);
                } else {
                    xv = ld_slot_stage<T>(stage(s, 0), c, p, H, wrap);
                    if constexpr (RESID) rv = ld_slot_stage<T>(stage(s, 1), c, p, H, wrap);
                }
                widen16<T>(xv, sv[i]);
                if constexpr (RESID) {
                    f32x2 rw[PR];
                    widen16<T>(rv, rw);
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[i][q] = f2_add(sv[i][q], rw[q]);
                    // an inner vector now, slots 0 and ns - 1 after the barrier
                    if (inner) st_global<T, V>(s_out + base + (c * V - p), narrow16<T>(sv[i]));
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
        // the barrier inside the reduction also means every thread has
        // copied stage s out, so it can be refilled
        float total = block_sum(f2_sum(ss2), red, bank);
        bank ^= 1;
        if (armer && k + nst < nrows) {
            if (!pw.stalled) {   // the issuer saw stage s's phase complete: refill it
                fence_proxy_async_smem();
                issue(k + nst, s);
            } else if (stall_rows < 0) {
                stall_rows = k + nst;   // rows issued before the issuer stalled
            }
        }
        if constexpr (RESID) {   // the partial vectors of residual_out (the row's ends)
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = k0 + i * kstep;
                if (c < ns && (c == 0 || c == ns - 1)) st_slot<T>(s_out + base, c, p, H, wrap, narrow16<T>(sv[i]));
            }
        }
        float mu = 0.0f;
        if constexpr (LN) {   // centre the row held in registers, then its sum of squares
            mu = total * ih;
            const f32x2 nm2 = f2_make(-mu, -mu);
            ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = k0 + i * kstep;
                if (c < ns) {
#pragma unroll
                    for (int q = 0; q < PR; ++q) sv[i][q] = f2_add(sv[i][q], nm2);
                    if (c == 0 || c == ns - 1) {   // slots reaching outside the row: those elements add nothing
#pragma unroll
                        for (int q = 0; q < PR; ++q) {
                            float d0, d1;
                            f2_split(sv[i][q], d0, d1);
                            sv[i][q] = f2_make(slot_elem_in_row<T>(c, 2 * q, p, H, wrap) ? d0 : 0.0f,
                                               slot_elem_in_row<T>(c, 2 * q + 1, p, H, wrap) ? d1 : 0.0f);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < PR; ++q) ss2 = f2_fma(sv[i][q], sv[i][q], ss2);
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
        if (p != p_w) {
            if (a.has_w) ld_op_windows<T, NV>(w, qw, p, H, k0, kstep, ns, wrap, wp);
            else
#pragma unroll
                for (int i = 0; i < NV; ++i) wp[i] = fill<T, V>(one<T>());
            if constexpr (LN) {
                if (bias != nullptr) ld_op_windows<T, NV>(bias, qb, p, H, k0, kstep, ns, wrap, bp);
                else
#pragma unroll
                    for (int i = 0; i < NV; ++i) bp[i] = fill<T, V>(from_f32<T>(0.0f));
            }
            p_w = p;
        }
        const f32x2 rr2 = f2_make(rrms, rrms);
        // y = (s * rrms) * w [LayerNorm: ((s - mean) * rstd) * w + b], one rounding to the storage type
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = k0 + i * kstep;
            if (c < ns) {
                f32x2 wv[PR], yv[PR];
                widen16<T>(wp[i], wv);
                if constexpr (LN) {
                    f32x2 bv[PR];
                    widen16<T>(bp[i], bv);
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_fma(f2_mul(sv[i][q], rr2), wv[q], bv[q]);
                } else {
#pragma unroll
                    for (int q = 0; q < PR; ++q) yv[q] = f2_mul(f2_mul(sv[i][q], rr2), wv[q]);
                }
                if (c != 0 && c != ns - 1) st_global<T, V>(y + base + (c * V - p), narrow16<T>(yv));
                else st_slot<T>(y + base, c, p, H, wrap, narrow16<T>(yv));
            }
        }
        if (++s == nst) {
            s = 0;
            phase ^= 1u;
        }
    }
    // Only a stalled CTA can exit with copies in flight: the issuer gives the
    // last issued phase of every stage one more bounded wait.
    if (pw.stalled) drain_ring(full, nst, stall_rows < 0 ? nrows : stall_rows);
}

namespace {

template <typename T, int MODE>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 2: return reinterpret_cast<const void *>(fwd_ring_phase_kernel<T, 2, MODE>);
    case 4: return reinterpret_cast<const void *>(fwd_ring_phase_kernel<T, 4, MODE>);
    }
    return nullptr;
}

template <typename T>
const void *kernel_mode(int mode, int nv) {
    switch (mode) {
    case kPlain: return kernel_nv<T, kPlain>(nv);
    case kResid: return kernel_nv<T, kResid>(nv);
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

// The aligned ring's geometry for the row's slots (an aligned row of
// ceil(H / V) vectors), with stages one 16-byte vector longer for the frame.
bool plan_fwd_ring_phase(int64_t M, int H, int dtype, int mode, int sm_count, RingPlan *out) {
    if (mode != kPlain && mode != kResid && mode != kLn && mode != kLnResid) return false;
    const int V = vec_elems(dtype);
    const int slots = (H + V - 1) / V;
    RingPlan p{};
    if (!fwd_ring_geometry(slots * V, dtype, mode, &p)) return false;
    const int streams = (mode == kResid || mode == kLnResid) ? 2 : 1;
    p.shape.row_pitch = (uint32_t)(((slots + 1) * 16 + 127) / 128 * 128);
    p.smem_bytes = kRingHeaderBytes + (size_t)p.shape.stages * streams * p.shape.row_pitch;
    if (p.smem_bytes > 200 * 1024) return false;
    const void *k = kernel_for(dtype, mode, p.nv);
    if (k == nullptr || allow_dynamic_smem(k, p.smem_bytes) != cudaSuccess) return false;
    // one CTA per SM (fused rows from 12 KB): two of two stages instead, so
    // while slot 0's thread finishes the row's two partial vectors and holds
    // its CTA at the barrier, the other CTA's rows stream
    if (p.max_ctas_per_sm == 1) {
        const int streams = (mode == kResid || mode == kLnResid) ? 2 : 1;
        const size_t smem = kRingHeaderBytes + (size_t)2 * streams * p.shape.row_pitch;
        if (allow_dynamic_smem(k, smem) == cudaSuccess && occupancy(k, p.threads, smem) >= 2) {
            p.shape.stages = 2;
            p.smem_bytes = smem;
            p.max_ctas_per_sm = 2;
        }
    }
    int occ = occupancy(k, p.threads, p.smem_bytes);
    if (occ <= 0) return false;
    if (p.max_ctas_per_sm > 0 && occ > p.max_ctas_per_sm) occ = p.max_ctas_per_sm;
    // fewer CTAs per SM than the geometry asks for (the longer stages can
    // cost one): deeper stages keep the rows in flight per SM
    if (p.max_ctas_per_sm > 0 && occ < p.max_ctas_per_sm) {
        const int stages = (p.shape.stages * p.max_ctas_per_sm + occ - 1) / occ;
        const size_t smem = kRingHeaderBytes + (size_t)stages * streams * p.shape.row_pitch;
        if (stages <= kRingMaxStages && smem <= 200 * 1024 && allow_dynamic_smem(k, smem) == cudaSuccess &&
            occupancy(k, p.threads, smem) >= occ) {
            p.shape.stages = stages;
            p.smem_bytes = smem;
        }
    }
    const int64_t cap = (int64_t)occ * sm_count;
    p.grid = (int)(M < cap ? M : cap);
    *out = p;
    return true;
}

cudaError_t launch_fwd_ring_phase(const FwdArgs &a, int dtype, int mode, const RingPlan &p, cudaStream_t st) {
    const void *k = kernel_for(dtype, mode, p.nv);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = allow_dynamic_smem(k, p.smem_bytes);
    if (e != cudaSuccess) return e;
    FwdArgs args = a;
    RingShape shape = p.shape;
    void *params[] = {&args, &shape};
    return cudaLaunchKernel(k, dim3((unsigned)p.grid), dim3((unsigned)p.threads), params, p.smem_bytes, st);
}

}  // namespace rmsn
