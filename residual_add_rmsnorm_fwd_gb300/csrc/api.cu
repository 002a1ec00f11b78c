// api.cu -- the extern "C" entry points of include/rmsnorm.h: argument
// validation (all of it before any launch), per-device limits, kernel choice
// and launch.
#include <cmath>
#include <cstring>
#include <initializer_list>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/rmsnorm.h"
#include "bulk.cuh"
#include "launch.h"

namespace rmsn {

// Device-side error word: bit kErrPipelineTimeout is set when a kernel's
// bounded wait on its bulk-copy pipeline gives up.  Read and cleared by
// rmsnorm_read_device_errors().
__device__ unsigned g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxH = int64_t(1) << 24;   // H is exact in binary32 up to 2^24
constexpr int kSmallH = 256;                  // warp-per-row kernel below this

struct DevInfo {
    bool checked = false;
    int status = RMSN_OK;
    int sm_count = 0;
    unsigned *err_word = nullptr;   // this device's copy of g_device_error
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
// Pipeline-wait settings copied into every launch: the poll limit, and the
// time-out test's held-back first copy (rmsnorm_debug_pipeline_timeout).
std::atomic<uint32_t> g_wait_polls{kWaitPolls};
std::atomic<int> g_hold_first{0};
std::map<std::tuple<int, const void *, int, size_t>, int> g_occ;
std::map<std::tuple<int, const void *, int, size_t, int>, int> g_cluster_occ;
std::map<std::pair<int, const void *>, size_t> g_smem_attr;


inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int round_up_to(int a, int b) { return ceil_div(a, b) * b; }

// Kernel image for sm_103 only: check the current device once.
int current_device(int *dev_out, int *sm_count) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RMSN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DevInfo &d = g_dev[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return RMSN_ERR_CUDA;
        }
        d.status = (major == 10 && minor == 3 && sms > 0) ? RMSN_OK : RMSN_ERR_UNSUPPORTED;
        d.sm_count = sms;
        if (d.status == RMSN_OK &&
            cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err_word), g_device_error) != cudaSuccess)
            return RMSN_ERR_CUDA;
        d.checked = true;
    }
    *dev_out = dev;
    *sm_count = d.sm_count;
    return d.status;
}

unsigned *device_error_word(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    return g_dev[dev].err_word;
}

bool aligned(const void *p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

struct Range {
    uintptr_t lo = 0, hi = 0;  // [lo, hi); empty when lo == hi
};

Range bytes_of(const void *p, size_t n) {
    Range r;
    if (p != nullptr && n > 0) {
        r.lo = reinterpret_cast<uintptr_t>(p);
        r.hi = r.lo + n;
    }
    return r;
}

Range matrix_of(const void *p, int64_t M, int64_t H, int64_t stride, int es) {
    if (M <= 0) return Range{};
    return bytes_of(p, (size_t)((M - 1) * stride + H) * (size_t)es);
}

bool overlap(const Range &a, const Range &b) {
    return a.lo != a.hi && b.lo != b.hi && a.lo < b.hi && b.lo < a.hi;
}

// Common shape checks; also rules out int64 overflow of the largest offset.
int check_shape(int64_t M, int64_t H, int64_t stride, int dtype) {
    if (dtype != RMSN_F32 && dtype != RMSN_F16 && dtype != RMSN_BF16) return RMSN_ERR_INVALID;
    if (M < 0 || H <= 0 || H > kMaxH || stride < H) return RMSN_ERR_INVALID;
    const int es = elem_bytes(dtype);
    if (M > 0 && (M - 1) > (INT64_MAX / es - H) / stride) return RMSN_ERR_INVALID;
    if (M > INT32_MAX) return RMSN_ERR_INVALID;  // grid arithmetic
    return RMSN_OK;
}

// The row matrices of a call (x, residual, outputs; nullptr = absent) start
// at one offset modulo 16 bytes: with their shared row stride, every row
// then has one alignment phase in all of them.
bool same_phase(std::initializer_list<const void *> ps) {
    const void *first = *ps.begin();
    for (const void *p : ps)
        if (p != nullptr && reinterpret_cast<uintptr_t>(p) % 16 != reinterpret_cast<uintptr_t>(first) % 16)
            return false;
    return true;
}

bool rows_vectorisable(int64_t H, int64_t stride, int dtype) {
    const int es = elem_bytes(dtype);
    return (H * es) % 16 == 0 && (stride * es) % 16 == 0;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? RMSN_OK : RMSN_ERR_CUDA; }

// Kernel family by row length and layout: lane groups below 256 elements
// (plain and residual-fused; AdaLN and LayerNorm take the register kernel
// there), a warp per aligned row of 512 B to 2 KB (plain, and AdaLN whose
// conditioning rows each serve 1024 rows or more), the bulk-copy ring for
// aligned rows of 4 KB (one input stream) or 8 KB and more up to 32 KB, the
// register kernel, a cluster of CTAs per aligned row of 32-256 KB, and the
// two-pass chunked kernel for the rest (longer or misaligned rows).  Rows
// that are not 16-byte aligned but whose matrices share one alignment phase
// (`phased`) take the register kernel in each row's aligned frame while the
// row fits it.
int dispatch_fwd(const FwdArgs &a, int dtype, int mode, bool vec, bool phased, int sms, cudaStream_t s) {
    if (a.H < kSmallH && (mode == kPlain || mode == kResid)) return to_status(launch_fwd_small(a, dtype, vec, sms, s));
    // AdaLN conditioning rows count as shared when each serves at least four
    // of a CTA's strides of rows, so a CTA rarely moves to a new one (below
    // that, staging them beside x, or the register kernel, measured 10-45%
    // faster: bf16 H = 4096 with 1024 rows per conditioning row, 4428 against
    // 4954 GB/s), or when one conditioning row serves every row
    if (vec && (mode == kPlain || (mode == kAdaln && a.rows_per_cond >= 1024)) && fwd_warp_fits(a.H, dtype))
        return to_status(launch_fwd_warp(a, dtype, mode, sms, s));
    RingPlan ring;
    if (vec && mode == kAdaln && plan_fwd_ring(a.M, a.H, dtype, kAdalnShared, sms, &ring)) {
        // few conditioning rows (at most one per four CTAs): one group of CTAs
        // per conditioning row, so each CTA reads a single one (bf16 12288 x
        // 2048, two rows: 20.1 -> 19.4 us per call); else the plain stride
        // when a conditioning row spans four of a CTA's strides of rows
        const int64_t n_cond = (a.M - 1) / a.rows_per_cond + 1;
        if (4 * n_cond <= (int64_t)ring.grid) {
            FwdArgs g = a;
            g.cond_groups = n_cond;
            return to_status(launch_fwd_ring(g, dtype, kAdalnShared, ring, s));
        }
        if (a.rows_per_cond >= 4 * (int64_t)ring.grid || a.rows_per_cond >= a.M)
            return to_status(launch_fwd_ring(a, dtype, kAdalnShared, ring, s));
    }
    if (vec && plan_fwd_ring(a.M, a.H, dtype, mode, sms, &ring))
        return to_status(launch_fwd_ring(a, dtype, mode, ring, s));
    if (!vec && phased) {
        if (plan_fwd_ring_phase(a.M, a.H, dtype, mode, sms, &ring))
            return to_status(launch_fwd_ring_phase(a, dtype, mode, ring, s));
        if (fwd_phase_fits(a.H, dtype)) return to_status(launch_fwd_phase(a, dtype, mode, sms, s));
    }
    if (fwd_row_fits(a.H, dtype, vec)) return to_status(launch_fwd_row(a, dtype, mode, vec, sms, s));
    // aligned rows above 32 KB: a cluster of CTAs per row (the same
    // shared-conditioning rule, with the cluster count as the row stride)
    SplitPlan split;
    if (vec && mode == kAdaln && plan_fwd_split(a.M, a.H, dtype, kAdalnShared, sms, &split) &&
        (a.rows_per_cond >= 4 * (int64_t)(split.grid / split.cs) || a.rows_per_cond >= a.M))
        return to_status(launch_fwd_split(a, dtype, kAdalnShared, split, s));
    if (vec && plan_fwd_split(a.M, a.H, dtype, mode, sms, &split))
        return to_status(launch_fwd_split(a, dtype, mode, split, s));
    return to_status(launch_fwd_chunked(a, dtype, mode, vec, sms, s));
}

int forward(const void *x, const void *residual, const void *weight, void *y, void *residual_out,
            float *rrms, int64_t row_stride, int64_t M, int64_t H, float eps, int dtype, int has_weight,
            void *stream, bool fused) {
    int st = check_shape(M, H, row_stride, dtype);
    if (st) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSN_ERR_INVALID;
    if (has_weight && weight == nullptr) return RMSN_ERR_INVALID;
    if (M > 0) {  // with no rows the matrix pointers are never used
        if (x == nullptr || y == nullptr) return RMSN_ERR_INVALID;
        if (fused && (residual == nullptr || residual_out == nullptr)) return RMSN_ERR_INVALID;
    }
    const int es = elem_bytes(dtype);
    const void *w = has_weight ? weight : nullptr;
    for (const void *p : {x, residual, w, static_cast<const void *>(y), static_cast<const void *>(residual_out)})
        if (p != nullptr && !aligned(p, es)) return RMSN_ERR_INVALID;
    if (rrms != nullptr && !aligned(rrms, 4)) return RMSN_ERR_INVALID;

    const Range rx = matrix_of(x, M, H, row_stride, es);
    const Range rr = fused ? matrix_of(residual, M, H, row_stride, es) : Range{};
    const Range rw = bytes_of(w, (size_t)H * es);
    const Range ry = matrix_of(y, M, H, row_stride, es);
    const Range rs = fused ? matrix_of(residual_out, M, H, row_stride, es) : Range{};
    const Range rq = bytes_of(rrms, (size_t)M * sizeof(float));
    const Range outs[] = {ry, rs, rq};
    const Range all[] = {rx, rr, rw, ry, rs, rq};
    // in place: y may be x itself and residual_out the residual itself
    // (every element is read before its thread writes it)
    const bool same[3][6] = {{y == x, false, false, false, false, false},
                             {false, fused && residual_out == residual, false, false, false, false},
                             {false, false, false, false, false, false}};
    for (int o = 0; o < 3; ++o)
        for (int k = 0; k < 6; ++k)
            if (k != 3 + o && !same[o][k] && overlap(outs[o], all[k])) return RMSN_ERR_ALIAS;

    if (M == 0) return RMSN_OK;
    int dev = 0, sms = 0;
    st = current_device(&dev, &sms);
    if (st) return st;

    bool vec = rows_vectorisable(H, row_stride, dtype);
    for (const void *p : {x, residual, w, static_cast<const void *>(y), static_cast<const void *>(residual_out)})
        if (p != nullptr && !aligned(p, 16)) vec = false;
    const bool phased = same_phase({x, fused ? residual : nullptr, y, fused ? residual_out : nullptr});

    FwdArgs a{};
    a.err = device_error_word(dev);
    a.wait_polls = g_wait_polls.load();
    a.hold_first = g_hold_first.load();
    a.x = x;
    a.r = fused ? residual : nullptr;
    a.w = w;
    a.y = y;
    a.s_out = fused ? residual_out : nullptr;
    a.rrms = rrms;
    a.stride = row_stride;
    a.M = M;
    a.H = (int)H;
    a.eps = eps;
    a.has_w = has_weight ? 1 : 0;
    return dispatch_fwd(a, dtype, fused ? kResid : kPlain, vec, phased, sms, static_cast<cudaStream_t>(stream));
}

// AdaLN forward: rows use conditioning row i / rows_per_cond of scale and
// shift (n_cond = ceil(M / rows_per_cond) rows of cond_stride elements).
int adaln_forward(const void *x, const void *weight, const void *scale, const void *shift, void *y, float *rrms,
                  int64_t row_stride, int64_t cond_stride, int64_t rows_per_cond, int64_t M, int64_t H, float eps,
                  int dtype, int has_weight, void *stream) {
    int st = check_shape(M, H, row_stride, dtype);
    if (st) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSN_ERR_INVALID;
    if (has_weight && weight == nullptr) return RMSN_ERR_INVALID;
    if (rows_per_cond < 1 || cond_stride < H) return RMSN_ERR_INVALID;
    const int64_t n_cond = M > 0 ? (M - 1) / rows_per_cond + 1 : 0;
    if ((st = check_shape(n_cond, H, cond_stride, dtype))) return st;
    if (M > 0 && (x == nullptr || y == nullptr || scale == nullptr || shift == nullptr)) return RMSN_ERR_INVALID;
    const int es = elem_bytes(dtype);
    const void *w = has_weight ? weight : nullptr;
    for (const void *p : {x, w, scale, shift, static_cast<const void *>(y)})
        if (p != nullptr && !aligned(p, es)) return RMSN_ERR_INVALID;
    if (rrms != nullptr && !aligned(rrms, 4)) return RMSN_ERR_INVALID;

    const Range rx = matrix_of(x, M, H, row_stride, es);
    const Range rw = bytes_of(w, (size_t)H * es);
    const Range rsc = matrix_of(scale, n_cond, H, cond_stride, es);
    const Range rsh = matrix_of(shift, n_cond, H, cond_stride, es);
    const Range ry = matrix_of(y, M, H, row_stride, es);
    const Range rq = bytes_of(rrms, (size_t)M * sizeof(float));
    const Range outs[] = {ry, rq};
    const Range all[] = {rx, rw, rsc, rsh, ry, rq};
    // in place: y may be x itself (scale and shift may be shared by rows,
    // so they are never overwritten)
    for (int o = 0; o < 2; ++o)
        for (int k = 0; k < 6; ++k)
            if (k != 4 + o && !(o == 0 && k == 0 && y == x) && overlap(outs[o], all[k])) return RMSN_ERR_ALIAS;

    if (M == 0) return RMSN_OK;
    int dev = 0, sms = 0;
    st = current_device(&dev, &sms);
    if (st) return st;

    bool vec = rows_vectorisable(H, row_stride, dtype) && (cond_stride * es) % 16 == 0;
    for (const void *p : {x, w, scale, shift, static_cast<const void *>(y)})
        if (p != nullptr && !aligned(p, 16)) vec = false;
    const bool phased = same_phase({x, y});

    FwdArgs a{};
    a.err = device_error_word(dev);
    a.wait_polls = g_wait_polls.load();
    a.hold_first = g_hold_first.load();
    a.x = x;
    a.w = w;
    a.y = y;
    a.rrms = rrms;
    a.stride = row_stride;
    a.M = M;
    a.H = (int)H;
    a.eps = eps;
    a.has_w = has_weight ? 1 : 0;
    a.scale = scale;
    a.shift = shift;
    a.cond_stride = cond_stride;
    a.rows_per_cond = rows_per_cond < M ? rows_per_cond : M;   // below 2^31, like M: 32-bit division
    return dispatch_fwd(a, dtype, kAdaln, vec, phased, sms, static_cast<cudaStream_t>(stream));
}

// Residual + LayerNorm forward: validation as for the RMSNorm forward, plus
// the bias and the saved mean.
int layernorm_forward(const void *x, const void *residual, const void *weight, const void *bias, void *y,
                      void *residual_out, float *mean, float *rstd, int64_t row_stride, int64_t M, int64_t H,
                      float eps, int dtype, int has_weight, int has_bias, void *stream, bool fused) {
    int st = check_shape(M, H, row_stride, dtype);
    if (st) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSN_ERR_INVALID;
    if ((has_weight && weight == nullptr) || (has_bias && bias == nullptr)) return RMSN_ERR_INVALID;
    if (M > 0) {
        if (x == nullptr || y == nullptr) return RMSN_ERR_INVALID;
        if (fused && (residual == nullptr || residual_out == nullptr)) return RMSN_ERR_INVALID;
    }
    const int es = elem_bytes(dtype);
    const void *w = has_weight ? weight : nullptr;
    const void *b = has_bias ? bias : nullptr;
    const void *r = fused ? residual : nullptr;
    void *so = fused ? residual_out : nullptr;
    for (const void *p : {x, r, w, b, static_cast<const void *>(y), static_cast<const void *>(so)})
        if (p != nullptr && !aligned(p, es)) return RMSN_ERR_INVALID;
    if ((rstd != nullptr && !aligned(rstd, 4)) || (mean != nullptr && !aligned(mean, 4))) return RMSN_ERR_INVALID;

    const Range rx = matrix_of(x, M, H, row_stride, es);
    const Range rr = matrix_of(r, M, H, row_stride, es);
    const Range rw = bytes_of(w, (size_t)H * es);
    const Range rb = bytes_of(b, (size_t)H * es);
    const Range ry = matrix_of(y, M, H, row_stride, es);
    const Range rs = matrix_of(so, M, H, row_stride, es);
    const Range rq = bytes_of(rstd, (size_t)M * sizeof(float));
    const Range rm = bytes_of(mean, (size_t)M * sizeof(float));
    const Range outs[] = {ry, rs, rq, rm};
    const Range all[] = {rx, rr, rw, rb, ry, rs, rq, rm};
    // in place: y may be x itself and residual_out the residual itself
    for (int o = 0; o < 4; ++o)
        for (int k = 0; k < 8; ++k) {
            const bool same = (o == 0 && k == 0 && y == x) || (o == 1 && k == 1 && so == r);
            if (k != 4 + o && !same && overlap(outs[o], all[k])) return RMSN_ERR_ALIAS;
        }

    if (M == 0) return RMSN_OK;
    int dev = 0, sms = 0;
    st = current_device(&dev, &sms);
    if (st) return st;

    bool vec = rows_vectorisable(H, row_stride, dtype);
    for (const void *p : {x, r, w, b, static_cast<const void *>(y), static_cast<const void *>(so)})
        if (p != nullptr && !aligned(p, 16)) vec = false;
    const bool phased = same_phase({x, r, y, so});

    FwdArgs a{};
    a.err = device_error_word(dev);
    a.wait_polls = g_wait_polls.load();
    a.hold_first = g_hold_first.load();
    a.x = x;
    a.r = r;
    a.w = w;
    a.b = b;
    a.y = y;
    a.s_out = so;
    a.rrms = rstd;
    a.mean = mean;
    a.stride = row_stride;
    a.M = M;
    a.H = (int)H;
    a.eps = eps;
    a.has_w = has_weight ? 1 : 0;
    return dispatch_fwd(a, dtype, fused ? kLnResid : kLn, vec, phased, sms, static_cast<cudaStream_t>(stream));
}

}  // namespace

cudaError_t allow_dynamic_smem(const void *func, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_pair(dev, func);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_smem_attr.find(key);
        if (it != g_smem_attr.end() && it->second >= bytes) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    size_t &v = g_smem_attr[key];
    if (bytes > v) v = bytes;
    return cudaSuccess;
}

namespace {

void finish_ring(RingPlan *p, int nv, int threads, int64_t row_bytes, int streams, int stages, int max_cps) {
    const uint32_t pitch = (uint32_t)round_up_to((int)row_bytes, 128);
    p->nv = nv;
    p->threads = threads;
    p->grid = 0;
    p->max_ctas_per_sm = max_cps;
    p->shape.stages = stages;
    p->shape.row_bytes = (uint32_t)row_bytes;
    p->shape.row_pitch = pitch;
    p->smem_bytes = kRingHeaderBytes + (size_t)stages * streams * pitch;
}

}  // namespace

// Forward ring geometry, measured on GB300 (bf16 unless noted, 100-540 MB
// per call).  Two 16-byte groups per thread (four above 1024 groups, and
// for LayerNorm from 8 KB, below).  The
// rule behind the table: about 64 KB of rows in flight per SM (stages x CTAs
// per SM x input rows per slot x row bytes) -- less leaves HBM idle, more
// loses DRAM efficiency -- with more CTAs per SM for short rows, whose fixed
// per-row cost (wait, barrier, reduction, rsqrt) is paid by every thread.
//   - One input row per slot (plain, LayerNorm, AdaLN with shared
//     conditioning rows), from 4 KB rows: 4-6 KB 2 stages x 8 CTAs (H = 2048:
//     5431 -> 5653 GB/s against the register kernel); 6-8 KB 4 x 4 (H = 3072:
//     5043 -> 6293 GB/s); 8-16 KB 2 x 4 (H = 4096: 4862 -> 6185 GB/s against
//     2 x 2; fp16 H = 6144: 6226 against 6106 at 2 x 3); from 16 KB 2 x 2
//     (H = 8192: 5826 -> 6515 GB/s against 3 x 4; fp32 H = 4096: 5493 -> 6592).
//   - Two input rows per slot (residual-fused, LayerNorm fused), from 8 KB
//     rows: 8-12 KB 2 x 2 (deeper or wider measured slower); 12-16 KB 3 x 1
//     (fp16 H = 6144: 5914 -> 6580 GB/s against 2 x 2); from 16 KB 2 x 1
//     (H = 8192: 5941 -> 6319 GB/s; fp32 H = 4096: 5930 -> 6309 GB/s).
//     Fused LayerNorm at 8-12 KB: 1 x 4 (6146 -> 6310 GB/s; its second
//     reduction per row favours more CTAs with one row each in flight).
//   - Three input rows per slot (AdaLN with per-token conditioning), from
//     8 KB rows: 8-12 KB 2 x 3 (6510 -> 6742 GB/s against 2 x 2); longer 2 x 1.
// Below these lengths the register and warp kernels were as fast or faster.
bool fwd_ring_geometry(int H, int dtype, int mode, RingPlan *p) {
    const int64_t row_bytes = (int64_t)H * elem_bytes(dtype);
    // x (+ residual | scale, shift)
    const int streams = mode == kAdaln ? 3 : ((mode == kResid || mode == kLnResid) ? 2 : 1);
    if (row_bytes % 16 != 0 || row_bytes < (streams == 1 ? 4096 : 8192)) return false;
    const int nvec = (int)(row_bytes / 16);
    constexpr int64_t KB = 1024;
    int nv = nvec <= 1024 ? 2 : 4;
    int stages = 2, cps = 2;
    if (streams == 1) {
        if (row_bytes < 6 * KB) cps = 8;
        else if (row_bytes < 8 * KB) stages = 4, cps = 4;
        else if (row_bytes < 16 * KB) cps = 4;
        // four groups per thread for plain LayerNorm from 8 KB, where the
        // per-row work every thread repeats (two reductions) dominates (bf16
        // H = 4096: 53.3 -> 49.5 us per 16384 rows).  At 4 KB rows four
        // groups with three stages helped only the weighted bf16 norm (18.0
        // -> 17.4 us per 12288 rows) and cost the unweighted, fp32 and f16
        // ones 1-3%, and shared-conditioning AdaLN 7%: two stay there
        if (mode == kLn && row_bytes >= 8 * KB) nv = 4;
    } else if (streams == 2) {
        if (row_bytes >= 16 * KB) cps = 1;
        else if (row_bytes >= 12 * KB) stages = 3, cps = 1;
        else if (mode == kLnResid) stages = 1, cps = 4;   // two reductions per row: more CTAs, one row each
        // fused LayerNorm takes plain LayerNorm's four groups per thread from
        // 8 KB (measured equal: 85.7 against 85.3 us at bf16 16384 x 4096), so
        // the two forms sum a row in the same order and give the same bits
        // for the same s
        if (mode == kLnResid && row_bytes >= 8 * KB) nv = 4;
    } else {
        cps = row_bytes < 12 * KB ? 3 : 1;
    }
    const int threads = round_up_to(ceil_div(nvec, nv), 32);
    if (threads > 512) return false;
    if (stages > kRingMaxStages) return false;   // one mbarrier per stage in the ring header
    if (kRingHeaderBytes + (size_t)stages * streams * round_up_to((int)row_bytes, 128) > 200 * 1024) return false;
    finish_ring(p, nv, threads, row_bytes, streams, stages, cps);
    return true;
}

// Backward: bfloat16 and binary32 rows take two 16-byte groups per thread up
// to 768 groups per row and four above (H = 4096 bf16: 256 threads; 6144:
// 384; 8192: 256); binary16 rows take four (its widening runs on the FP32
// pipe, and the longer per-thread chains measured faster: H = 6144 f16, 205
// against 245 us), or three where that fills whole warps (182 us at 6144).
// Two stages, as many CTAs per SM as fit -- the backward
// profits from every resident warp.  Measured on GB300 at H = 4096-8192.
bool bwd_ring_geometry(int H, int dtype, bool dres, RingPlan *p) {
    const int64_t row_bytes = (int64_t)H * elem_bytes(dtype);
    if (row_bytes % 16 != 0 || row_bytes < 2048) return false;
    const int nvec = (int)(row_bytes / 16);
    int nv = (dtype != kF16 && nvec <= 768) ? 2 : 4;
    // binary16 rows of 768-1536 groups that split evenly into warps of three
    // groups per thread: three (f16 H = 6144: 205.8 -> 182.2 us per 32768 rows)
    if (dtype == kF16 && nvec >= 768 && nvec <= 1536 && nvec % 96 == 0) nv = 3;
    const int threads = round_up_to(ceil_div(nvec, nv), 32);
    if (threads > 512) return false;
    const int stages = kBwdRingStages;
    const int streams = dres ? 3 : 2;
    const size_t smem = kRingHeaderBytes + (size_t)stages * streams * round_up_to((int)row_bytes, 128);
    if (smem > 200 * 1024) return false;
    finish_ring(p, nv, threads, row_bytes, streams, stages, 0);
    return true;
}

// Split-row rule: the longest segment (16-byte groups) a CTA takes, the
// ring stages per CTA and the CTAs per SM (0 = as many as fit), by kernel.
struct SplitRule {
    int max_seg;
    int stages;
    int cps;
};

SplitRule split_rule(int streams, bool backward) {
    if (backward) return SplitRule{2048, kBwdRingStages, 0};
    return SplitRule{2048, 2, 0};
}

// Split-row geometry, for aligned rows above 32 KB (which one CTA's
// registers and ring no longer hold) up to 256 KB: the smallest cluster of
// 2, 4 or 8 CTAs whose segments fit the rule's longest segment, else eight
// CTAs with segments up to 2048 groups (32 KB).  Groups per thread as in the
// ring kernels for rows of the segment's length; stages from the rule,
// fewer if the ring would exceed 200 KB of shared memory.
bool split_geometry(int H, int dtype, int streams, bool backward, SplitPlan *p) {
    const int64_t row_bytes = (int64_t)H * elem_bytes(dtype);
    if (row_bytes % 16 != 0) return false;
    const int nvec = (int)(row_bytes / 16);
    if (nvec <= 2048) return false;   // one CTA holds the row
    const SplitRule rule = split_rule(streams, backward);
    int cs = 0;
    for (int c : {2, 4, 8})
        if (ceil_div(nvec, c) <= rule.max_seg) {
            cs = c;
            break;
        }
    if (cs == 0) {
        if (ceil_div(nvec, 8) > 2048) return false;
        cs = 8;
    }
    // seg >= 257 groups and cs * seg - nvec < cs, so the last segment is not empty
    const int seg = ceil_div(nvec, cs);
    const int nv = backward ? ((dtype != kF16 && seg <= 768) ? 2 : 4) : (seg <= 1024 ? 2 : 4);
    const uint32_t pitch = (uint32_t)round_up_to(seg * 16, 128);
    int stages = rule.stages;
    while (stages > 2 && kRingHeaderBytes + (size_t)stages * streams * pitch > 200 * 1024) --stages;
    const size_t smem = kRingHeaderBytes + (size_t)stages * streams * pitch;
    if (smem > 200 * 1024 || stages > kRingMaxStages) return false;
    p->cs = cs;
    p->nv = nv;
    p->threads = round_up_to(ceil_div(seg, nv), 32);
    p->grid = 0;
    p->max_ctas_per_sm = rule.cps;
    p->smem_bytes = smem;
    p->shape.stages = stages;
    p->shape.seg_groups = seg;
    p->shape.seg_pitch = pitch;
    return true;
}

namespace {

// Clusters of `cs` CTAs of `func` that can be resident on the device at once.
int cluster_occupancy(const void *func, int threads, size_t smem, int cs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(dev, func, threads, smem, cs);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_cluster_occ.find(key);
        if (it != g_cluster_occ.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    g_cluster_occ[key] = n;
    return n;
}

}  // namespace

bool finish_split_plan(const void *k, int64_t M, int sm_count, SplitPlan *p) {
    if (allow_dynamic_smem(k, p->smem_bytes) != cudaSuccess) return false;
    int64_t nc = cluster_occupancy(k, p->threads, p->smem_bytes, p->cs);
    if (nc <= 0) return false;
    if (p->max_ctas_per_sm > 0) {
        const int64_t cap = (int64_t)p->max_ctas_per_sm * sm_count / p->cs;
        if (cap >= 1 && cap < nc) nc = cap;
    }
    if (nc > M) nc = M;
    p->grid = (int)(nc * p->cs);
    return true;
}

cudaError_t launch_cluster(const void *k, const SplitPlan &p, void **params, cudaStream_t st) {
    cudaError_t e = allow_dynamic_smem(k, p.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, k, params);
}

int occupancy(const void *func, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(dev, func, threads, smem);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    g_occ[key] = n;
    return n;
}

namespace {

int backward(const void *dy, const void *dres, const void *x, const void *weight, const float *rrms, void *dx,
             float *dweight, void *workspace, size_t workspace_bytes, int64_t row_stride, int64_t M, int64_t H,
             int dtype, int has_weight, void *stream, bool fused) {
    int st = check_shape(M, H, row_stride, dtype);
    if (st) return st;
    if (has_weight && weight == nullptr) return RMSN_ERR_INVALID;
    if (M > 0 && (dy == nullptr || x == nullptr || rrms == nullptr || dx == nullptr || (fused && dres == nullptr)))
        return RMSN_ERR_INVALID;  // with no rows the row pointers are never used
    const int es = elem_bytes(dtype);
    const void *w = has_weight ? weight : nullptr;
    float *dw = has_weight ? dweight : nullptr;
    const void *dr = fused ? dres : nullptr;
    for (const void *p : {dy, dr, x, w, static_cast<const void *>(dx)})
        if (p != nullptr && !aligned(p, es)) return RMSN_ERR_INVALID;
    if ((rrms != nullptr && !aligned(rrms, 4)) || (dw != nullptr && !aligned(dw, 4))) return RMSN_ERR_INVALID;

    if (M == 0) {
        // no rows: dweight is an empty sum
        if (dw != nullptr) return to_status(cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float),
                                                            static_cast<cudaStream_t>(stream)));
        return RMSN_OK;
    }
    int dev = 0, sms = 0;
    st = current_device(&dev, &sms);
    if (st) return st;

    bool vec = rows_vectorisable(H, row_stride, dtype);
    for (const void *p : {dy, dr, x, w, static_cast<const void *>(dx)})
        if (p != nullptr && !aligned(p, 16)) vec = false;
    const bool phased = same_phase({x, dy, dr, dx});
    const BwdPlan plan = plan_bwd(M, (int)H, dtype, vec, phased, fused, sms);
    const size_t part_bytes = dw != nullptr ? bwd_partial_bytes(plan, (int)H) : 0;
    if (dw != nullptr) {
        if (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < part_bytes)
            return RMSN_ERR_WORKSPACE;
    }

    const Range rdy = matrix_of(dy, M, H, row_stride, es);
    const Range rx = matrix_of(x, M, H, row_stride, es);
    const Range rw = bytes_of(w, (size_t)H * es);
    const Range rq = bytes_of(rrms, (size_t)M * sizeof(float));
    const Range rdr = matrix_of(dr, M, H, row_stride, es);
    const Range rdx = matrix_of(dx, M, H, row_stride, es);
    const Range rdw = bytes_of(dw, (size_t)H * sizeof(float));
    const Range rws = bytes_of(dw != nullptr ? workspace : nullptr, part_bytes);
    const Range outs[] = {rdx, rdw, rws};
    const Range all[] = {rdy, rx, rw, rq, rdr, rdx, rdw, rws};
    // in place: dx may be dy, x or dresidual_out itself (each element of a
    // row is read before its thread writes dx there; the row's reduction
    // completes before any dx of the row is written)
    const bool same_dx[8] = {dx == dy, dx == x, false, false, dr != nullptr && dx == dr, false, false, false};
    for (int o = 0; o < 3; ++o)
        for (int k = 0; k < 8; ++k)
            if (k != 5 + o && !(o == 0 && same_dx[k]) && overlap(outs[o], all[k])) return RMSN_ERR_ALIAS;

    BwdArgs a{};
    a.err = device_error_word(dev);
    a.wait_polls = g_wait_polls.load();
    a.hold_first = g_hold_first.load();
    a.dy = dy;
    a.dres = dr;
    a.x = x;
    a.w = w;
    a.rrms = rrms;
    a.dx = dx;
    a.partial = dw != nullptr ? static_cast<float *>(workspace) : nullptr;
    a.stride = row_stride;
    a.M = M;
    a.H = (int)H;
    a.has_w = has_weight ? 1 : 0;
    return to_status(launch_bwd(a, plan, dtype, vec, dw, static_cast<cudaStream_t>(stream)));
}

}  // namespace

}  // namespace rmsn

using namespace rmsn;

// the library is built with hidden visibility; only the C ABI is exported
#define RMSN_API __attribute__((visibility("default")))

extern "C" {

RMSN_API int rmsnorm_fwd(const void *x, const void *weight, void *y, float *rrms, int64_t row_stride, int64_t M,
                int64_t H, float eps, int dtype, int has_weight, void *stream) {
    return forward(x, nullptr, weight, y, nullptr, rrms, row_stride, M, H, eps, dtype, has_weight, stream, false);
}

RMSN_API int rmsnorm_fwd_residual(const void *x, const void *residual, const void *weight, void *y, void *residual_out,
                         float *rrms, int64_t row_stride, int64_t M, int64_t H, float eps, int dtype,
                         int has_weight, void *stream) {
    return forward(x, residual, weight, y, residual_out, rrms, row_stride, M, H, eps, dtype, has_weight, stream,
                   true);
}

RMSN_API int rmsnorm_adaln_fwd(const void *x, const void *weight, const void *scale, const void *shift, void *y,
                               float *rrms, int64_t row_stride, int64_t cond_stride, int64_t rows_per_cond,
                               int64_t M, int64_t H, float eps, int dtype, int has_weight, void *stream) {
    return adaln_forward(x, weight, scale, shift, y, rrms, row_stride, cond_stride, rows_per_cond, M, H, eps, dtype,
                         has_weight, stream);
}

RMSN_API int layernorm_fwd(const void *x, const void *weight, const void *bias, void *y, float *mean, float *rstd,
                           int64_t row_stride, int64_t M, int64_t H, float eps, int dtype, int has_weight,
                           int has_bias, void *stream) {
    return layernorm_forward(x, nullptr, weight, bias, y, nullptr, mean, rstd, row_stride, M, H, eps, dtype,
                             has_weight, has_bias, stream, false);
}

RMSN_API int layernorm_fwd_residual(const void *x, const void *residual, const void *weight, const void *bias,
                                    void *y, void *residual_out, float *mean, float *rstd, int64_t row_stride,
                                    int64_t M, int64_t H, float eps, int dtype, int has_weight, int has_bias,
                                    void *stream) {
    return layernorm_forward(x, residual, weight, bias, y, residual_out, mean, rstd, row_stride, M, H, eps, dtype,
                             has_weight, has_bias, stream, true);
}

RMSN_API int rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H, int dtype, size_t *bytes) {
    if (bytes == nullptr) return RMSN_ERR_INVALID;
    *bytes = 0;
    int st = check_shape(M, H, H, dtype);
    if (st) return st;
    if (M == 0) return RMSN_OK;
    int dev = 0, sms = 0;
    st = current_device(&dev, &sms);
    if (st) return st;
    // the largest of the variants rmsnorm_bwd and rmsnorm_bwd_residual may pick
    size_t need = 0;
    for (int layout = 0; layout < 3; ++layout) {   // 16-byte aligned rows, rows at one phase, other rows
        const bool vec = layout == 0, phased = layout == 1;
        if (vec && (H * elem_bytes(dtype)) % 16 != 0) continue;
        for (int dres = 0; dres < 2; ++dres) {
            const size_t v = bwd_partial_bytes(plan_bwd(M, (int)H, dtype, vec, phased, dres != 0, sms), (int)H);
            need = v > need ? v : need;
        }
    }
    *bytes = need;
    return RMSN_OK;
}

RMSN_API int rmsnorm_bwd(const void *dy, const void *x, const void *weight, const float *rrms, void *dx, float *dweight,
                         void *workspace, size_t workspace_bytes, int64_t row_stride, int64_t M, int64_t H, int dtype,
                         int has_weight, void *stream) {
    return backward(dy, nullptr, x, weight, rrms, dx, dweight, workspace, workspace_bytes, row_stride, M, H, dtype,
                    has_weight, stream, false);
}

RMSN_API int rmsnorm_bwd_residual(const void *dy, const void *dresidual_out, const void *x, const void *weight,
                                  const float *rrms, void *dx, float *dweight, void *workspace,
                                  size_t workspace_bytes, int64_t row_stride, int64_t M, int64_t H, int dtype,
                                  int has_weight, void *stream) {
    return backward(dy, dresidual_out, x, weight, rrms, dx, dweight, workspace, workspace_bytes, row_stride, M, H,
                    dtype, has_weight, stream, true);
}

RMSN_API int rmsnorm_read_device_errors(unsigned *flags) {
    if (flags == nullptr) return RMSN_ERR_INVALID;
    *flags = 0;
    int dev = 0, sms = 0;
    int st = current_device(&dev, &sms);
    if (st) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return RMSN_ERR_CUDA;
    unsigned *word = device_error_word(dev);
    unsigned zero = 0;
    if (cudaMemcpy(flags, word, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(word, &zero, sizeof(unsigned), cudaMemcpyHostToDevice) != cudaSuccess)
        return RMSN_ERR_CUDA;
    return RMSN_OK;
}

RMSN_API int rmsnorm_debug_pipeline_timeout(unsigned polls, int hold_first_copy) {
    if (polls == 0 && hold_first_copy == 0) {   // normal operation
        g_wait_polls.store(kWaitPolls);
        g_hold_first.store(0);
        return RMSN_OK;
    }
    if (polls == 0 || polls > kWaitPolls || (hold_first_copy != 0 && hold_first_copy != 1)) return RMSN_ERR_INVALID;
    g_wait_polls.store(polls);
    g_hold_first.store(hold_first_copy);
    return RMSN_OK;
}

RMSN_API const char *rmsnorm_status_string(int status) {
    switch (status) {
    case RMSN_OK: return "ok";
    case RMSN_ERR_INVALID: return "invalid argument (pointer, size, stride, eps, dtype or alignment)";
    case RMSN_ERR_ALIAS: return "an output overlaps another argument";
    case RMSN_ERR_WORKSPACE: return "backward workspace missing, misaligned or too small";
    case RMSN_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case RMSN_ERR_UNSUPPORTED: return "no usable sm_103 device is current";
    }
    return "unknown status";
}

}  // extern "C"
