// bwd_ring_phase.cu -- RMSNorm backward (plain and with the residual
// stream's gradient) with rows staged by bulk copies, for rows of 2-32 KB
// that are not 16-byte aligned but whose matrices share one alignment phase.
//
// The ring of bwd_ring.cu in each row's aligned frame, as fwd_ring_phase.cu
// does for the forward: the copies cover the row's frame (whole 16-byte
// granules, each inside the allocation holding any of its bytes; the bytes
// outside the row are zeroed in registers and never used), dx is written in
// whole 16-byte vectors except the row's first and last (element by element,
// never outside the row), and the weight is cut out of its own aligned
// vectors by the row's shift.  As in bwd_phase.cu, every row of a CTA has
// the CTA's phase (the host makes the grid a multiple of V whenever a CTA
// has more than one row), so each thread keeps the dweight terms of fixed
// columns in registers across the CTA's rows, summed in row order:
// dweight stays bit-reproducible ("Skill: Write a Triton RMSNorm Kernel",
// Required reasoning 12).
#include "bulk.cuh"
#include "launch.h"
#include "phase.cuh"

namespace rmsn {

// Register budget as the aligned ring backward's: the two-group variants
// held to 80 registers (three CTAs of 256 threads per SM).
constexpr int bwd_ring_phase_max_regs(int nv) { return nv == 2 ? 80 : 128; }

template <typename T, int NV, bool DRES>
__global__ void __launch_bounds__(512) __maxnreg__(bwd_ring_phase_max_regs(NV))
    bwd_ring_phase_kernel(BwdArgs a, RingShape rs) {
    constexpr int V = 16 / sizeof(T);
    constexpr int PR = V / 2;
    constexpr int NS = DRES ? 3 : 2;   // streams staged per row: dy, x (and dres)
    using P = Pack<T, V>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[64];
    __shared__ int64_t stall_rows;   // the issuer: rows issued before it stalled (-1: all)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    unsigned char *stages = smem + kRingHeaderBytes;

    // dx may be dy, x or dres itself (in-place calls): not restrict
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    const T *x = static_cast<const T *>(a.x);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *dx = static_cast<T *>(a.dx);
    const int H = a.H;
    const float ih = 1.0f / (float)H;   // one division per CTA; exact for power-of-two H
    constexpr int nst = kBwdRingStages;   // rs.stages is the same value
    const int qw = a.has_w ? elem_phase(w) : 0;
    const int k0 = threadIdx.x, kstep = blockDim.x;
    const int64_t G = gridDim.x;
    const int64_t nrows = (a.M - 1 - blockIdx.x) / G + 1;  // the grid never exceeds M

    auto stage = [&](int s, int j) { return stages + (size_t)(s * NS + j) * rs.row_pitch; };
    auto issue = [&](int64_t k, int s) {   // row k of this CTA's frame into stage s (= k mod nst)
        const int64_t base = (blockIdx.x + k * G) * a.stride;
        const int p = elem_phase(x + base);
        const uint32_t bytes = (uint32_t)((p + H + V - 1) / V) * 16u;
        mbar_arrive_expect_tx(&full[s], NS * bytes);
        bulk_g2s(stage(s, 0), dy + base - p, bytes, &full[s]);
        bulk_g2s(stage(s, 1), x + base - p, bytes, &full[s]);
        if constexpr (DRES) bulk_g2s(stage(s, 2), dres + base - p, bytes, &full[s]);
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

    // dweight terms of this thread's slots k = k0 + i * kstep, element j:
    // column k*V + j - pc (slot 0 also the wrapped columns), pc the phase of
    // every row of this CTA (the host makes the grid a multiple of V whenever
    // a CTA has more than one row, so rows G apart are G * stride elements
    // apart, a multiple of 16 bytes)
    const int ns = frame_slots<T>(H);
    const int pc = elem_phase(x + (int64_t)blockIdx.x * a.stride);
    f32x2 acc[NV][PR];
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int q = 0; q < PR; ++q) acc[i][q] = f2_make(0.0f, 0.0f);

    P wp[NV];   // weight windows of phase p_w
    int p_w = -1;
    int bank = 0;
    float rr_next = __ldg(a.rrms + blockIdx.x);
    for (int64_t k = 0; k < nrows; ++k) {
        const int s = (int)((uint32_t)k % (uint32_t)nst);
        const uint32_t phase = ((uint32_t)k / (uint32_t)nst) & 1u;
        const int64_t base = (blockIdx.x + k * G) * a.stride;
        const int p = elem_phase(x + base);
        const bool wrap = row_wraps<T>(p, H);
        const float rr = rr_next;
        if (k + 1 < nrows) rr_next = __ldg(a.rrms + blockIdx.x + (k + 1) * G);
        const f32x2 rr2 = f2_make(rr, rr);
        if (p != p_w) {
            if (a.has_w) ld_op_windows<T, NV>(w, qw, p, H, k0, kstep, ns, wrap, wp);
            else
#pragma unroll
                for (int i = 0; i < NV; ++i) wp[i] = fill<T, V>(one<T>());
            p_w = p;
        }
        pipe_wait<RingWaitConst<T>::value>(&full[s], phase, pw, a.wait_polls, armer, a.err);

        // the frame's bytes outside the row are zeroed, so they add nothing
        P gp[NV], xp[NV], rp[NV];
        f32x2 dot2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = k0 + i * kstep;
            if (c < ns) {
                if (c != 0 && c != ns - 1) {   // only slots 0 and ns - 1 reach outside the row
                    gp[i] = *reinterpret_cast<const P *>(stage(s, 0) + (size_t)c * 16);
                    xp[i] = *reinterpret_cast<const P *>(stage(s, 1) + (size_t)c * 16);
                    if constexpr (DRES) rp[i] = *reinterpret_cast<const P *>(stage(s, 2) + (size_t)c * 16);
                } else {
                    gp[i] = ld_slot_stage<T>(stage(s, 0), c, p, H, wrap);
                    xp[i] = ld_slot_stage<T>(stage(s, 1), c, p, H, wrap);
                    if constexpr (DRES) rp[i] = ld_slot_stage<T>(stage(s, 2), c, p, H, wrap);
                }
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
        // the reduction barrier frees stage s for the row nst ahead
        const float c_row = block_sum(f2_sum(dot2), red, bank) * ih;
        if (armer && k + nst < nrows) {
            if (!pw.stalled) {   // the issuer saw stage s's phase complete: refill it
                fence_proxy_async_smem();
                issue(k + nst, s);
            } else if (stall_rows < 0) {
                stall_rows = k + nst;   // rows issued before the issuer stalled
            }
        }
        // dx = rrms * (g - xhat * c) (+ dres), evaluated as the aligned ring does
        const float kx = -(rr * rr) * c_row;
        const f32x2 kx2 = f2_make(kx, kx);
        const f32x2 nc2 = f2_make(-c_row, -c_row);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = k0 + i * kstep;
            if (c < ns) {
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
                if (c != 0 && c != ns - 1) st_global<T, V>(dx + base + (c * V - p), narrow16<T>(d));
                else st_slot<T>(dx + base, c, p, H, wrap, narrow16<T>(d));
            }
        }
        bank ^= 1;
    }

    if (a.partial != nullptr) store_partial<T, NV, true>(a.partial + (int64_t)blockIdx.x * H, acc, pc, H, k0, kstep);
    // Only a stalled CTA can exit with copies in flight: the issuer gives the
    // last issued phase of every stage one more bounded wait.
    if (pw.stalled) drain_ring(full, nst, stall_rows < 0 ? nrows : stall_rows);
    allow_dependent_launch();
}

namespace {

template <typename T, bool DRES>
const void *kernel_nv(int nv) {
    switch (nv) {
    case 2: return reinterpret_cast<const void *>(bwd_ring_phase_kernel<T, 2, DRES>);
    case 3: return reinterpret_cast<const void *>(bwd_ring_phase_kernel<T, 3, DRES>);
    case 4: return reinterpret_cast<const void *>(bwd_ring_phase_kernel<T, 4, DRES>);
    }
    return nullptr;
}

}  // namespace

// The aligned ring's backward geometry for the row's slots (an aligned row
// of ceil(H / V) vectors), with stages one 16-byte vector longer for the frame.
bool bwd_ring_phase_geometry(int H, int dtype, bool dres, RingPlan *p) {
    const int V = vec_elems(dtype);
    const int slots = (H + V - 1) / V;
    if (!bwd_ring_geometry(slots * V, dtype, dres, p)) return false;
    p->shape.row_pitch = (uint32_t)(((slots + 1) * 16 + 127) / 128 * 128);
    p->smem_bytes = kRingHeaderBytes + (size_t)p->shape.stages * (dres ? 3 : 2) * p->shape.row_pitch;
    return p->smem_bytes <= 200 * 1024;
}

const void *bwd_ring_phase_kernel_for(int dtype, int nv, bool dres) {
    switch (dtype) {
    case kF32: return dres ? kernel_nv<float, true>(nv) : kernel_nv<float, false>(nv);
    case kF16: return dres ? kernel_nv<__half, true>(nv) : kernel_nv<__half, false>(nv);
    case kBF16: return dres ? kernel_nv<__nv_bfloat16, true>(nv) : kernel_nv<__nv_bfloat16, false>(nv);
    }
    return nullptr;
}

}  // namespace rmsn
