// bwd.cu -- RMSNorm backward: dx per row, and a deterministic dweight.
//
// ("Skill: Write a Triton RMSNorm Kernel", Required reasoning 12;
// Correctness requirements on the saved rrms and the dweight axis.)
// With g = dy * w and xhat = x * rrms (rrms read from the forward's saved
// buffer, never recomputed):
//     dx      = rrms * (g - xhat * (sum_h g_h * xhat_h) / H)
//     dweight = sum over rows of dy * xhat
//
// dweight is a cross-row reduction, so it is done in two launches with no
// atomics and no inter-CTA waiting:
//   1. a persistent grid of G CTAs; CTA b owns the rows b, b + G, b + 2G, ...
//      and accumulates dy * xhat for its rows in binary32, column by column,
//      then writes its partial sums to row b of a G x H workspace;
//   2. a column kernel sums the G partials of each column in a fixed order.
// The row-to-CTA assignment and both summation orders depend only on (M, H,
// dtype, device), so dweight is bit-reproducible run to run.
#include "launch.h"

namespace rmsn {

// Row kept in registers: a thread owns NV groups of VEC columns; its
// dweight partials for those columns stay in registers across all its rows.
template <typename T, int VEC, int NV, bool DRES>
__global__ void __launch_bounds__(512) bwd_row_kernel(BwdArgs a) {
    using P = Pack<T, VEC>;
    __shared__ float red[64];
    // dx may be dy, x or dres itself (in-place calls): not restrict
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    const T *x = static_cast<const T *>(a.x);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *dx = static_cast<T *>(a.dx);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H

    P wp[NV];
    float acc[NV][VEC];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        wp[i] = (a.has_w && c < nvec) ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[i][j] = 0.0f;
    }

    int bank = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.stride;
        const float rr = __ldg(a.rrms + row);
        P gp[NV], xp[NV], rp[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                gp[i] = ld_stream<T, VEC>(dy + base + (int64_t)c * VEC);
                xp[i] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                if constexpr (DRES) rp[i] = ld_stream<T, VEC>(dres + base + (int64_t)c * VEC);
            }
        }
        float dot = 0.0f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                float d[VEC], xv[VEC], wv[VEC];
                unpack(gp[i], d);
                unpack(xp[i], xv);
                unpack(wp[i], wv);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float xh = xv[j] * rr;
                    dot += (d[j] * wv[j]) * xh;
                    acc[i][j] += d[j] * xh;
                }
            }
        }
        const float c_row = block_sum(dot, red, bank) * ih;
        bank ^= 1;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                float d[VEC], xv[VEC], wv[VEC];
                unpack(gp[i], d);
                unpack(xp[i], xv);
                unpack(wp[i], wv);
#pragma unroll
                for (int j = 0; j < VEC; ++j) d[j] = rr * (d[j] * wv[j] - (xv[j] * rr) * c_row);
                if constexpr (DRES) {   // the residual stream's gradient joins ds
                    float rv[VEC];
                    unpack(rp[i], rv);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) d[j] += rv[j];
                }
                st_global<T, VEC>(dx + base + (int64_t)c * VEC, pack<T, VEC>(d));
            }
        }
    }

    if (a.partial != nullptr) {
        float *prow = a.partial + (int64_t)blockIdx.x * a.H;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = threadIdx.x + i * blockDim.x;
            if (c < nvec) {
                if constexpr (VEC % 4 == 0) {
#pragma unroll
                    for (int j = 0; j < VEC; j += 4)
                        *reinterpret_cast<float4 *>(prow + (int64_t)c * VEC + j) =
                            make_float4(acc[i][j], acc[i][j + 1], acc[i][j + 2], acc[i][j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) prow[(int64_t)c * VEC + j] = acc[i][j];
                }
            }
        }
    }
    allow_dependent_launch();
}

// H above the register budget: two passes over each row with identical chunk
// bounds.  The CTA's dweight partial row belongs to this CTA alone, each
// column to one thread: it is accumulated in shared memory when H binary32
// values fit (use_smem_acc; written to the workspace once at the end), else
// updated in the workspace with 16-byte read-modify-writes (the first row of
// the CTA initialises it).  Measured on GB300 at bf16 H = 32768: 1275 GB/s
// with per-element updates in global memory, 2455 with 16-byte ones, 3062
// in shared memory.
template <typename T, int VEC, bool DRES>
__global__ void __launch_bounds__(512) bwd_chunked_kernel(BwdArgs a) {
    using P = Pack<T, VEC>;
    constexpr int U = 2;
    __shared__ float red[64];
    // dx may be dy, x or dres itself (in-place calls): not restrict
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    const T *x = static_cast<const T *>(a.x);
    const T *__restrict__ w = static_cast<const T *>(a.w);
    T *dx = static_cast<T *>(a.dx);
    const int nvec = a.H / VEC;
    const float hf = (float)a.H;
    const float ih = 1.0f / hf;   // one division per CTA; exact for power-of-two H
    const int chunk = blockDim.x * U;
    float *prow = a.partial != nullptr ? a.partial + (int64_t)blockIdx.x * a.H : nullptr;
    extern __shared__ __align__(16) float sacc[];   // the CTA's partial row (H floats) when given
    const bool use_s = prow != nullptr && (VEC % 4 == 0) && a.use_smem_acc;
    if (use_s)
        for (int c = threadIdx.x; c < nvec; c += blockDim.x)   // each thread's own columns
#pragma unroll
            for (int j = 0; j < VEC; ++j) sacc[c * VEC + j] = 0.0f;

    int bank = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.stride;
        const float rr = __ldg(a.rrms + row);
        const bool first = row == blockIdx.x;
        float dot = 0.0f;
        for (int c0 = 0; c0 < nvec; c0 += chunk) {
            P gp[U], xp[U], wp[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    gp[u] = ld_plain<T, VEC>(dy + base + (int64_t)c * VEC);
                    xp[u] = ld_plain<T, VEC>(x + base + (int64_t)c * VEC);
                    wp[u] = a.has_w ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    float d[VEC], xv[VEC], wv[VEC];
                    unpack(gp[u], d);
                    unpack(xp[u], xv);
                    unpack(wp[u], wv);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) dot += (d[j] * wv[j]) * (xv[j] * rr);
                }
            }
        }
        const float c_row = block_sum(dot, red, bank) * ih;
        bank ^= 1;
        for (int c0 = 0; c0 < nvec; c0 += chunk) {
            P gp[U], xp[U], wp[U], rp[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    gp[u] = ld_stream<T, VEC>(dy + base + (int64_t)c * VEC);
                    xp[u] = ld_stream<T, VEC>(x + base + (int64_t)c * VEC);
                    wp[u] = a.has_w ? ld_cached<T, VEC>(w + (int64_t)c * VEC) : fill<T, VEC>(one<T>());
                    if constexpr (DRES) rp[u] = ld_stream<T, VEC>(dres + base + (int64_t)c * VEC);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                if (c < nvec) {
                    float d[VEC], xv[VEC], wv[VEC], o[VEC], rv[VEC];
                    unpack(gp[u], d);
                    unpack(xp[u], xv);
                    unpack(wp[u], wv);
                    if constexpr (DRES) unpack(rp[u], rv);
                    float pk[VEC];   // this row's dweight terms dy * xhat
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const float xh = xv[j] * rr;
                        o[j] = rr * (d[j] * wv[j] - xh * c_row);
                        if constexpr (DRES) o[j] += rv[j];
                        pk[j] = d[j] * xh;
                    }
                    st_global<T, VEC>(dx + base + (int64_t)c * VEC, pack<T, VEC>(o));
                    if (use_s) {
                        if constexpr (VEC % 4 == 0) {
#pragma unroll
                            for (int j = 0; j < VEC; j += 4) {
                                float4 *q = reinterpret_cast<float4 *>(sacc + c * VEC + j);
                                const float4 t = *q;
                                *q = make_float4(t.x + pk[j], t.y + pk[j + 1], t.z + pk[j + 2], t.w + pk[j + 3]);
                            }
                        }
                    } else if (prow != nullptr) {   // 16-byte read-modify-write of the CTA's own partial row
                        float *p = prow + (int64_t)c * VEC;
                        if constexpr (VEC % 4 == 0) {
#pragma unroll
                            for (int j = 0; j < VEC; j += 4) {
                                float4 *q = reinterpret_cast<float4 *>(p + j);
                                const float4 t = first ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : *q;
                                *q = make_float4(t.x + pk[j], t.y + pk[j + 1], t.z + pk[j + 2], t.w + pk[j + 3]);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < VEC; ++j) p[j] = first ? pk[j] : p[j] + pk[j];
                        }
                    }
                }
            }
        }
    }
    if (use_s)   // the partial, built in shared memory, written once
        for (int c = threadIdx.x; c < nvec; c += blockDim.x)
#pragma unroll
            for (int j = 0; j < VEC; j += 4)
                *reinterpret_cast<float4 *>(prow + (int64_t)c * VEC + j) =
                    *reinterpret_cast<const float4 *>(sacc + c * VEC + j);
    allow_dependent_launch();
}

// dweight_h = sum_{b = 0}^{G-1} partial[b][h].  A CTA covers 32 columns with
// S warps (S = blockDim.x / 32, at most kReduceSlices); warp k sums the
// contiguous slice of partial rows [k*G/S, (k+1)*G/S) in ascending order (up
// to kReduceBatch loads in flight, added one after another), then the slice
// sums are added in ascending k.  S depends only on G (reduce_slices), so the
// order, and the result, is reproducible.
constexpr int kReduceSlices = 32;
constexpr int kReduceBatch = 24;

// Warps per column block: about eight partial rows per slice, at most 32
// (the usual 300-600 partial rows of the ring backward take 32; the 20-80
// of the split backward a few, so fewer idle threads per column).
inline int reduce_slices(int G) {
    const int s = G / 8;
    return s < 1 ? 1 : (s > kReduceSlices ? kReduceSlices : s);
}

// SFIX > 0: the slice count as a compile-time constant (the ring backward's
// usual 32), so the final sum over the slices is unrolled -- its loads issue
// together instead of one load-add chain (measured 0.35 us less per call);
// SFIX = 0: S = blockDim.x / 32 at run time.  The order of the additions is
// the same either way.
template <int SFIX>
__global__ void __launch_bounds__(32 * kReduceSlices)
    dweight_reduce_kernel(const float *__restrict__ partial, int G, int H, float *__restrict__ dweight) {
    // launched as a programmatic dependent of the backward: its partials are
    // complete and visible only after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float part[kReduceSlices][33];
    const int S = SFIX > 0 ? SFIX : (int)(blockDim.x >> 5);
    const int col = threadIdx.x & 31, k = threadIdx.x >> 5;
    const int h = blockIdx.x * 32 + col;
    float s = 0.0f;
    if (h < H) {
        const int g0 = (int)((int64_t)G * k / S), g1 = (int)((int64_t)G * (k + 1) / S);
        // up to kReduceBatch loads in flight per thread: a slice of the
        // usual 304-608 partial rows is one round trip to L2 (summed in
        // ascending row order either way)
        for (int g = g0; g < g1; g += kReduceBatch) {
            float v[kReduceBatch];
#pragma unroll
            for (int u = 0; u < kReduceBatch; ++u)
                v[u] = g + u < g1 ? __ldg(partial + (int64_t)(g + u) * H + h) : 0.0f;
#pragma unroll
            for (int u = 0; u < kReduceBatch; ++u) s += v[u];
        }
    }
    part[k][col] = s;
    __syncthreads();
    if (k == 0 && h < H) {
        float t = 0.0f;
        if constexpr (SFIX > 0) {
#pragma unroll
            for (int q = 0; q < SFIX; ++q) t += part[q][col];
        } else {
            for (int q = 0; q < S; ++q) t += part[q][col];
        }
        dweight[h] = t;
    }
}

namespace {

constexpr int kRowMaxThreads = 512;
constexpr size_t kChunkedSmemAccBytes = 160 * 1024;   // largest shared partial row of the chunked backward
constexpr int kChunkThreads = 512;
constexpr int kVecNV[] = {1, 2};
constexpr int kScalarNV[] = {1, 2, 4, 8};

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

bool pick_row(int nvec, bool vec, int &threads, int &nv) {
    const int *set = vec ? kVecNV : kScalarNV;
    const int n = vec ? 2 : 4;
    for (int k = 0; k < n; ++k) {
        const int t = round_up((nvec + set[k] - 1) / set[k], 32);
        if (t <= kRowMaxThreads) {
            threads = t;
            nv = set[k];
            return true;
        }
    }
    return false;
}

template <typename T, int VEC, int NV, bool DRES>
const void *row_kernel() {
    return reinterpret_cast<const void *>(bwd_row_kernel<T, VEC, NV, DRES>);
}

template <typename T, bool DRES>
const void *row_kernel_for(bool vec, int nv) {
    constexpr int V = Vec16<T>::n;
    if (vec) {
        switch (nv) {
        case 1: return row_kernel<T, V, 1, DRES>();
        case 2: return row_kernel<T, V, 2, DRES>();
        }
    } else {
        switch (nv) {
        case 1: return row_kernel<T, 1, 1, DRES>();
        case 2: return row_kernel<T, 1, 2, DRES>();
        case 4: return row_kernel<T, 1, 4, DRES>();
        case 8: return row_kernel<T, 1, 8, DRES>();
        }
    }
    return nullptr;
}

template <typename T, bool DRES>
const void *chunked_kernel_for(bool vec) {
    constexpr int V = Vec16<T>::n;
    return vec ? reinterpret_cast<const void *>(bwd_chunked_kernel<T, V, DRES>)
               : reinterpret_cast<const void *>(bwd_chunked_kernel<T, 1, DRES>);
}

template <typename T>
const void *kernel_for_dt(const BwdPlan &p, bool vec) {
    if (p.dres) return p.kind == kBwdRow ? row_kernel_for<T, true>(vec, p.nv) : chunked_kernel_for<T, true>(vec);
    return p.kind == kBwdRow ? row_kernel_for<T, false>(vec, p.nv) : chunked_kernel_for<T, false>(vec);
}

const void *kernel_for(const BwdPlan &p, int dtype, bool vec) {
    if (p.kind == kBwdRing) return bwd_ring_kernel_for(dtype, p.nv, p.dres);
    if (p.kind == kBwdPhase) return bwd_phase_kernel_for(dtype, p.nv, p.dres);
    if (p.kind == kBwdRingPhase) return bwd_ring_phase_kernel_for(dtype, p.nv, p.dres);
    if (p.kind == kBwdSplit) return bwd_split_kernel_for(dtype, p.nv, p.dres);
    switch (dtype) {
    case kF32: return kernel_for_dt<float>(p, vec);
    case kF16: return kernel_for_dt<__half>(p, vec);
    case kBF16: return kernel_for_dt<__nv_bfloat16>(p, vec);
    }
    return nullptr;
}

}  // namespace

BwdPlan plan_bwd(int64_t M, int H, int dtype, bool vec, bool phased, bool dres, int sm_count) {
    BwdPlan p{};
    p.dres = dres;
    p.cs = 1;
    RingPlan rp{};
    SplitPlan sp{};
    if (vec && bwd_ring_geometry(H, dtype, dres, &rp)) {
        p.kind = kBwdRing;
        p.threads = rp.threads;
        p.nv = rp.nv;
        p.smem_bytes = rp.smem_bytes;
        p.ring = rp.shape;
    } else if (vec && split_geometry(H, dtype, dres ? 3 : 2, true, &sp) &&
               finish_split_plan(bwd_split_kernel_for(dtype, sp.nv, dres), M > 0 ? M : 1, sm_count, &sp)) {
        p.kind = kBwdSplit;   // a cluster per row (aligned rows of 32-256 KB)
        p.threads = sp.threads;
        p.nv = sp.nv;
        p.smem_bytes = sp.smem_bytes;
        p.split = sp.shape;
        p.cs = sp.cs;
        p.grid = sp.grid;
        p.partial_rows = sp.grid / sp.cs;
        return p;
    } else if (!vec && phased && bwd_ring_phase_geometry(H, dtype, dres, &rp)) {
        p.kind = kBwdRingPhase;   // misaligned rows at one phase of 2-32 KB: the ring in the row's frame
        p.threads = rp.threads;
        p.nv = rp.nv;
        p.smem_bytes = rp.smem_bytes;
        p.ring = rp.shape;
    } else if (!vec && phased && bwd_phase_pick(H, dtype, &p.threads, &p.nv)) {
        p.kind = kBwdPhase;   // misaligned rows at one phase: 128-bit accesses in the row's frame
    } else {
        const int nvec = vec ? H / vec_elems(dtype) : H;
        p.kind = pick_row(nvec, vec, p.threads, p.nv) ? kBwdRow : kBwdChunked;
        if (p.kind == kBwdChunked) {
            p.threads = kChunkThreads;
            p.nv = 0;
        }
    }
    const void *k = kernel_for(p, dtype, vec);
    int occ = 0;
    size_t smem_occ = p.smem_bytes;   // the chunked kernel's shared partial row counts toward occupancy
    if (p.kind == kBwdChunked && vec && (size_t)H * 4 <= kChunkedSmemAccBytes) smem_occ = (size_t)H * 4;
    if (k != nullptr && allow_dynamic_smem(k, smem_occ) == cudaSuccess)
        occ = occupancy(k, p.threads, smem_occ);
    int64_t cap = (int64_t)(occ > 0 ? occ : 1) * sm_count;
    // rows not 16-byte aligned: a grid that is a multiple of V (elements per
    // 16 bytes) gives every row of a CTA the same phase, which the kernels'
    // dweight registers need (rows G apart are a multiple of 16 bytes apart)
    const int V = vec_elems(dtype);
    if ((p.kind == kBwdPhase || p.kind == kBwdRingPhase) && M > cap && cap >= V) cap = cap / V * V;
    p.grid = (int)(M < cap ? (M > 0 ? M : 1) : cap);
    p.partial_rows = p.grid;
    return p;
}

size_t bwd_partial_bytes(const BwdPlan &p, int H) { return (size_t)p.partial_rows * (size_t)H * sizeof(float); }

cudaError_t launch_bwd(const BwdArgs &a, const BwdPlan &p, int dtype, bool vec, float *dweight,
                       cudaStream_t st) {
    const void *k = kernel_for(p, dtype, vec);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = allow_dynamic_smem(k, p.smem_bytes);
    if (e != cudaSuccess) return e;
    BwdArgs args = a;
    if (p.kind == kBwdSplit) {
        SplitPlan sp{};
        sp.cs = p.cs;
        sp.nv = p.nv;
        sp.threads = p.threads;
        sp.grid = p.grid;
        sp.smem_bytes = p.smem_bytes;
        sp.shape = p.split;
        SplitShape shape = p.split;
        void *params[] = {&args, &shape};
        e = launch_cluster(k, sp, params, st);
    } else {
        RingShape shape = p.ring;
        size_t smem = p.smem_bytes;
        if (p.kind == kBwdChunked && vec && a.partial != nullptr && (size_t)a.H * 4 <= kChunkedSmemAccBytes) {
            smem = (size_t)a.H * 4;
            args.use_smem_acc = 1;
            e = allow_dynamic_smem(k, smem);
            if (e != cudaSuccess) return e;
        }
        void *params[] = {&args, &shape};
        e = cudaLaunchKernel(k, dim3((unsigned)p.grid), dim3((unsigned)p.threads), params, smem, st);
    }
    if (e != cudaSuccess) return e;
    if (dweight != nullptr && a.partial != nullptr) {
        // a programmatic dependent of the backward: its CTAs are scheduled as
        // the backward's last CTAs finish (hiding the launch), and wait in
        // griddepcontrol.wait for the backward's completion (measured: 1 us
        // less per backward at bf16 16384 x 4096)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((a.H + 31) / 32));
        cfg.blockDim = dim3(32u * (unsigned)reduce_slices(p.partial_rows));
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const float *part = a.partial;
        const int G = p.partial_rows, H = a.H;
        e = reduce_slices(G) == kReduceSlices
                ? cudaLaunchKernelEx(&cfg, dweight_reduce_kernel<kReduceSlices>, part, G, H, dweight)
                : cudaLaunchKernelEx(&cfg, dweight_reduce_kernel<0>, part, G, H, dweight);
    }
    return e;
}

}  // namespace rmsn
