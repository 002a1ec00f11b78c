"""GPU parity: every kernel path of the library against the fp64 oracle,
element by element, on seeded inputs, with guard bands around every buffer.

Tolerances: forward fp32 within 1e-5 relative per element; forward f16/bf16
within 1 ulp of the oracle's value rounded to the storage type; residual
write-back bit-exact with the oracle's sum rounded to the storage type;
backward dx within 1e-5 (fp32) or 2e-2 (f16/bf16) of max(|ref|, row rms of
ref, dx_scale) where dx_scale is the size of the two terms whose difference
forms dx; dweight within the same rtol times sum_i |dy * xhat| per column.

Kernel paths (chosen by H, dtype and layout): the lane-group kernel for
H < 256, a warp per aligned row of 512 B to 2 KB (plain forward), the
register-resident row kernel, the bulk-copy ring for aligned rows of 4-8 KB
up to 32 KB, a thread-block cluster per aligned row of 32-256 KB (H = 32768
bf16/f16 and f32 H = 16384 here; tests/test_split_gpu.py covers that path in
depth), the chunked two-pass kernel for misaligned rows above the register
budget; the lane-group, row and chunked kernels each in a 128-bit variant
(16-byte aligned rows) and a scalar one.
"""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import (Guarded, bwd_rtol, check_dweight, check_fwd_values, check_dx, device_vec,
                     f32_buffer)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]
# small-H lane groups, register rows, 4097 (scalar tail), 10001 (scalar, chunked), split rows
H_FWD = [1, 7, 8, 64, 100, 255, 256, 1000, 1024, 2048, 4096, 4097, 6144, 8192, 10001, 16384, 32768]
H_BWD = [1, 7, 64, 255, 256, 1000, 2048, 4096, 4097, 6144, 8192, 10001, 16384]


def rows_for(H, cap=400_000):
    return int(max(3, min(257, cap // H))) | 1   # odd row counts leave ragged grid tails


def run_fwd(oracle, dtype, M, H, stride=None, residual=False, weight=True, save_rrms=True, offset=0,
            eps=1e-5, seed=0, x_np=None, r_np=None, w_np=None, w_offset=None):
    """w_offset: the weight's own element offset (default: offset)."""
    stride = H if stride is None else stride
    w_offset = offset if w_offset is None else w_offset
    rng = wl.rng_for(seed)
    x = wl.matrix(rng, M, H, dtype, stride) if x_np is None else x_np
    r = (wl.matrix(rng, M, H, dtype, stride) if r_np is None else r_np) if residual else None
    w = (wl.weight(rng, H, dtype) if w_np is None else w_np) if weight else None
    gx = Guarded(M, H, stride, dtype, offset).upload(x)
    gy = Guarded(M, H, stride, dtype, offset)
    gr = Guarded(M, H, stride, dtype, offset).upload(r) if residual else None
    gs = Guarded(M, H, stride, dtype, offset) if residual else None
    wd = device_vec(w, dtype, w_offset) if weight else None
    rrms = f32_buffer(M, offset) if save_rrms else None
    if residual:
        rn.rmsnorm_fwd_residual(gx.t, gr.t, wd, gy.t, gs.t, rrms, eps=eps)
    else:
        rn.rmsnorm_fwd(gx.t, wd, gy.t, rrms, eps=eps)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_fwd(x[:, :H], w, eps, dtype, residual=None if r is None else r[:, :H])
    res = {"y": check_fwd_values(gy.host(), ref["y"], dtype, oracle)}
    assert gy.untouched_outside() and gx.untouched_outside()
    if residual:
        want_s = oracle.encode(ref["s"], dtype)
        got_s = gs.host()
        res["s_mismatch"] = int(np.sum(got_s.view(np.uint32 if dtype == "f32" else np.uint16)
                                       != want_s.view(np.uint32 if dtype == "f32" else np.uint16)))
        assert gs.untouched_outside() and gr.untouched_outside()
    if save_rrms:
        got = rrms.cpu().numpy().astype(np.float64)
        res["rrms_bad"] = int(np.sum(~(np.abs(got - ref["rrms"]) <= 1e-5 * ref["rrms"])))
    res.update(gy=gy, gs=gs, rrms=rrms, ref=ref, x=x, r=r, w=w)
    return res


def assert_fwd_ok(res):
    assert res["y"]["failed"] == 0, f"y: {res['y']['failed']} failed elements, max err {res['y']['max_err']}"
    assert res.get("s_mismatch", 0) == 0, f"residual_out: {res['s_mismatch']} elements not bit-exact"
    assert res.get("rrms_bad", 0) == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", H_FWD)
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("weight", [True, False])
def test_fwd_paths(oracle, dtype, H, residual, weight):
    res = run_fwd(oracle, dtype, rows_for(H), H, residual=residual, weight=weight, seed=H)
    assert_fwd_ok(res)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,stride,offset", [
    (64, 72, 0), (64, 67, 0), (1000, 1003, 0), (4096, 4096, 1), (4096, 4160, 0), (6144, 6272, 0),
    (2048, 2049, 1), (200, 200, 3), (16384, 16392, 0), (16384, 16385, 1), (512, 520, 0), (1024, 1032, 0),
    (768, 776, 0)])
def test_fwd_strides_and_misalignment(oracle, dtype, H, stride, offset):
    for residual in (False, True):
        res = run_fwd(oracle, dtype, rows_for(H, 200_000), H, stride=stride, residual=residual,
                      offset=offset, seed=stride + offset)
        assert_fwd_ok(res)


@pytest.mark.parametrize("dtype,H,M", [("bf16", 64, 50001), ("bf16", 1024, 5001), ("f16", 8, 70001),
                                       ("f32", 4096, 1201), ("bf16", 32768, 401)])
def test_fwd_grid_stride(oracle, dtype, H, M):
    """More rows than resident CTAs/warps: every CTA handles several rows."""
    assert_fwd_ok(run_fwd(oracle, dtype, M, H, residual=True, seed=M))


@pytest.mark.parametrize("dtype,H,M", [("bf16", 1024, 40001), ("f16", 512, 90001), ("f32", 256, 70001),
                                       ("bf16", 4096, 20001), ("bf16", 8192, 6001), ("f32", 4096, 9001)])
def test_fwd_plain_grid_stride(oracle, dtype, H, M):
    """The plain forward over many rows per warp (512 B - 2 KB rows) or per ring CTA."""
    assert_fwd_ok(run_fwd(oracle, dtype, M, H, residual=False, seed=M + 1))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 1024, 4097, 32768])
def test_no_weight_is_bitwise_unit_weight(oracle, dtype, H):
    M = rows_for(H)
    a = run_fwd(oracle, dtype, M, H, weight=False, seed=3)
    ones = wl.to_storage(np.ones(H, np.float32), dtype)
    b = run_fwd(oracle, dtype, M, H, weight=True, w_np=ones, x_np=a["x"], seed=3)
    assert torch.equal(a["gy"].t, b["gy"].t)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 4096, 32768])
def test_residual_fusion_equals_add_then_norm(oracle, dtype, H):
    """With sums exact in the storage type, fusing the add changes nothing (bitwise)."""
    M = rows_for(H)
    rng = np.random.default_rng(H)
    xv = rng.integers(-60, 60, (M, H)).astype(np.float32)
    rv = rng.integers(-60, 60, (M, H)).astype(np.float32)
    x, r = wl.to_storage(xv, dtype), wl.to_storage(rv, dtype)
    s = wl.to_storage(xv + rv, dtype)
    fused = run_fwd(oracle, dtype, M, H, residual=True, x_np=x, r_np=r, seed=1)
    plain = run_fwd(oracle, dtype, M, H, residual=False, x_np=s, w_np=fused["w"], seed=1)
    assert torch.equal(fused["gy"].t, plain["gy"].t)
    assert torch.equal(fused["rrms"], plain["rrms"])


@pytest.mark.parametrize("H", [64, 2048, 32768])
def test_fp16_outliers_need_fp32_accumulation(oracle, H):
    """|x| up to 300: x^2 exceeds the fp16 maximum (65504); the result stays finite and exact."""
    M = rows_for(H)
    x = wl.matrix(wl.rng_for(5), M, H, "f16", outlier_frac=0.05)
    res = run_fwd(oracle, "f16", M, H, residual=True, x_np=x, seed=5)
    assert_fwd_ok(res)
    assert bool(torch.isfinite(res["gy"].t).all())


@pytest.mark.parametrize("dtype", DTYPES)
def test_zero_rows_and_eps(oracle, dtype):
    H, M = 1024, 5
    x = wl.to_storage(np.zeros((M, H), np.float32), dtype)
    res = run_fwd(oracle, dtype, M, H, x_np=x, eps=1e-6)
    assert_fwd_ok(res)
    assert bool((res["gy"].t == 0).all())
    np.testing.assert_allclose(res["rrms"].cpu().numpy(), 1 / np.sqrt(np.float32(1e-6)), rtol=1e-6)
    # eps = 0 on nonzero rows is valid and exact to the same tolerance
    assert_fwd_ok(run_fwd(oracle, dtype, 33, 512, eps=0.0, seed=9))


def test_rrms_optional_and_single_row(oracle):
    assert_fwd_ok(run_fwd(oracle, "bf16", 1, 4096, residual=True, save_rrms=False))
    assert_fwd_ok(run_fwd(oracle, "bf16", 1, 64, save_rrms=False))


def test_zero_rows_no_launch():
    x = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    rn.rmsnorm_fwd(x, None, torch.empty_like(x))
    dw = torch.full((64,), 7.0, device="cuda")
    rn.rmsnorm_bwd(x, x.clone(), torch.ones(64, device="cuda", dtype=torch.bfloat16),
                   torch.empty(0, device="cuda"), torch.empty_like(x), dw, None)
    torch.cuda.synchronize()
    assert bool((dw == 0).all())   # the empty sum


# ---------------------------------------------------------------- backward --

def run_bwd(oracle, dtype, M, H, stride=None, weight=True, offset=0, eps=1e-5, seed=0, want_dw=True,
            fused=False, w_offset=None):
    stride = H if stride is None else stride
    w_offset = offset if w_offset is None else w_offset
    rng = wl.rng_for(seed)
    fwd = run_fwd(oracle, dtype, M, H, stride=stride, residual=fused, weight=weight, offset=offset,
                  eps=eps, seed=seed, w_offset=w_offset)
    assert_fwd_ok(fwd)
    # the input the backward sees: x, or residual_out for the fused forward
    xin = fwd["gs"] if fused else None
    x_np = xin.host() if fused else fwd["x"][:, :H]
    dy = wl.matrix(rng, M, H, dtype, stride)
    gdy = Guarded(M, H, stride, dtype, offset).upload(dy)
    if fused:
        gx = xin
    else:
        gx = Guarded(M, H, stride, dtype, offset).upload(fwd["x"])
    gdx = Guarded(M, H, stride, dtype, offset)
    w = fwd["w"]
    wd = device_vec(w, dtype, w_offset) if weight else None
    dw = f32_buffer(H) if (weight and want_dw) else None
    nbytes = rn.rmsnorm_bwd_workspace_bytes(M, H, dtype=wl.torch_dtype(dtype))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda") if dw is not None else None
    rn.rmsnorm_bwd(gdy.t, gx.t, wd, fwd["rrms"], gdx.t, dw, ws)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_bwd(dy[:, :H], x_np, w, eps, dtype)
    got_dx = oracle.decode(gdx.host(), dtype) if dtype != "f32" else gdx.host().astype(np.float64)
    out = {"dx": check_dx(got_dx, ref["dx"], ref["dx_scale"], bwd_rtol(dtype))}
    if dw is not None:
        out["dw"] = check_dweight(dw.cpu().numpy(), ref["dweight"], ref["dweight_abs"], bwd_rtol(dtype))
    assert gdx.untouched_outside() and gdy.untouched_outside()
    out.update(dw_t=dw, gdx=gdx, ws=ws)
    return out


def run_bwd_residual(oracle, dtype, M, H, stride=None, weight=True, offset=0, eps=1e-5, seed=0, w_offset=None):
    """Fused forward, then the fused backward with an incoming residual-stream gradient."""
    stride = H if stride is None else stride
    w_offset = offset if w_offset is None else w_offset
    rng = wl.rng_for(seed + 1000)
    fwd = run_fwd(oracle, dtype, M, H, stride=stride, residual=True, weight=weight, offset=offset, eps=eps,
                  seed=seed, w_offset=w_offset)
    assert_fwd_ok(fwd)
    s_np = fwd["gs"].host()
    dy = wl.matrix(rng, M, H, dtype, stride)
    dres = wl.matrix(rng, M, H, dtype, stride)
    gdy = Guarded(M, H, stride, dtype, offset).upload(dy)
    gdr = Guarded(M, H, stride, dtype, offset).upload(dres)
    gdx = Guarded(M, H, stride, dtype, offset)
    w = fwd["w"]
    wd = device_vec(w, dtype, w_offset) if weight else None
    dw = f32_buffer(H) if weight else None
    nbytes = rn.rmsnorm_bwd_workspace_bytes(M, H, wl.torch_dtype(dtype))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda") if dw is not None else None
    rn.rmsnorm_bwd_residual(gdy.t, gdr.t, fwd["gs"].t, wd, fwd["rrms"], gdx.t, dw, ws)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_bwd(dy[:, :H], s_np, w, eps, dtype, dres=dres[:, :H])
    got_dx = oracle.decode(gdx.host(), dtype) if dtype != "f32" else gdx.host().astype(np.float64)
    out = {"dx": check_dx(got_dx, ref["dx"], ref["dx_scale"], bwd_rtol(dtype))}
    if dw is not None:
        out["dw"] = check_dweight(dw.cpu().numpy(), ref["dweight"], ref["dweight_abs"], bwd_rtol(dtype))
    assert gdx.untouched_outside() and gdy.untouched_outside() and gdr.untouched_outside()
    return out


def assert_bwd_ok(out):
    assert out["dx"]["failed"] == 0, f"dx: {out['dx']['failed']} failed, max rel {out['dx']['max_rel']}"
    if "dw" in out:
        assert out["dw"]["failed"] == 0, f"dweight: {out['dw']['failed']} failed, max rel {out['dw']['max_rel']}"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", H_BWD)
@pytest.mark.parametrize("weight", [True, False])
def test_bwd_paths(oracle, dtype, H, weight):
    assert_bwd_ok(run_bwd(oracle, dtype, rows_for(H), H, weight=weight, seed=H + 1))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,stride,offset", [(64, 67, 0), (4096, 4096, 1), (6144, 6272, 0), (1000, 1001, 1),
                                             (16384, 16400, 0)])
def test_bwd_strides_and_misalignment(oracle, dtype, H, stride, offset):
    assert_bwd_ok(run_bwd(oracle, dtype, rows_for(H, 200_000), H, stride=stride, offset=offset, seed=stride))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 4096, 6144])
def test_bwd_after_fused_forward(oracle, dtype, H):
    """Backward of the fused forward: x := residual_out, saved rrms from the unrounded sum."""
    assert_bwd_ok(run_bwd(oracle, dtype, rows_for(H), H, fused=True, seed=H + 7))


@pytest.mark.parametrize("dtype,H,M", [("bf16", 4096, 3001), ("f16", 64, 20001), ("f32", 16384, 301)])
def test_bwd_grid_stride(oracle, dtype, H, M):
    assert_bwd_ok(run_bwd(oracle, dtype, M, H, seed=M))


def test_bwd_without_dweight(oracle):
    assert_bwd_ok(run_bwd(oracle, "bf16", 129, 4096, want_dw=False))


@pytest.mark.parametrize("dtype,H", [("bf16", 8192), ("f16", 6144), ("f32", 1000), ("bf16", 16384)])
def test_dweight_deterministic(oracle, dtype, H):
    a = run_bwd(oracle, dtype, 1001, H, seed=4)
    b = run_bwd(oracle, dtype, 1001, H, seed=4)
    assert torch.equal(a["dw_t"], b["dw_t"])
    assert torch.equal(a["gdx"].t, b["gdx"].t)


def test_workspace_too_small():
    M, H = 256, 4096
    x = torch.randn(M, H, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    rrms = torch.ones(M, device="cuda")
    need = rn.rmsnorm_bwd_workspace_bytes(M, H, torch.bfloat16)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_bwd(x, x.clone(), w, rrms, torch.empty_like(x), torch.empty(H, device="cuda"), ws)
    assert e.value.status == 3
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_bwd(x, x.clone(), w, rrms, torch.empty_like(x), torch.empty(H, device="cuda"), None)
    assert e.value.status == 3


def test_partial_overlap_rejected():
    x = torch.randn(64, 1024, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_fwd(x[:, :1000], None, x[:, 8:1008])
    assert e.value.status == 2


def check_in_place(oracle, dtype, M, H, offset, eps=1e-5):
    """In-place calls on one kernel path, each checked against the oracle
    element by element and bit for bit against the same call with separate
    outputs: the fused forward with y over x and residual_out over the
    residual; the backward with dx over dy, over x, and (fused backward) over
    dresidual_out.  Guard bands and padding stay untouched."""
    rng = wl.rng_for(H + offset)
    xs, rs = wl.matrix(rng, M, H, dtype), wl.matrix(rng, M, H, dtype)
    w_np = wl.weight(rng, H, dtype)
    w = device_vec(w_np, dtype, offset)
    dys, drs = wl.matrix(rng, M, H, dtype), wl.matrix(rng, M, H, dtype)
    G = lambda a=None: Guarded(M, H, H, dtype, offset) if a is None else Guarded(M, H, H, dtype, offset).upload(a)
    # forward, out of place
    x, r, y, so = G(xs), G(rs), G(), G()
    rr = f32_buffer(M, offset)
    rn.rmsnorm_fwd_residual(x.t, r.t, w, y.t, so.t, rr, eps=eps)
    # forward, in place
    xi, ri = G(xs), G(rs)
    rri = f32_buffer(M, offset)
    rn.rmsnorm_fwd_residual(xi.t, ri.t, w, xi.t, ri.t, rri, eps=eps)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_fwd(xs, w_np, eps, dtype, residual=rs)
    c = check_fwd_values(xi.host(), ref["y"], dtype, oracle)
    assert c["failed"] == 0, f"in-place y: {c['failed']} failed elements"
    want_s = oracle.encode(ref["s"], dtype)
    assert np.array_equal(ri.host().view(want_s.dtype), want_s), "in-place residual_out not bit-exact"
    got_rr = rri.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_rr - ref["rrms"]) <= 1e-5 * ref["rrms"])
    assert torch.equal(xi.t, y.t) and torch.equal(ri.t, so.t) and torch.equal(rri, rr)
    assert xi.untouched_outside() and ri.untouched_outside()

    # backward on the fused forward's residual_out: dx over dy, over x, over dresidual_out
    s_np = so.host()
    nbytes = rn.rmsnorm_bwd_workspace_bytes(M, H, wl.torch_dtype(dtype))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    dy, dx, dw = G(dys), G(), f32_buffer(H)
    rn.rmsnorm_bwd(dy.t, so.t, w, rr, dx.t, dw, ws)
    dyi, dwi = G(dys), f32_buffer(H)
    rn.rmsnorm_bwd(dyi.t, so.t, w, rr, dyi.t, dwi, ws)              # dx over dy
    sx, dwx = G(s_np), f32_buffer(H)
    rn.rmsnorm_bwd(dy.t, sx.t, w, rr, sx.t, dwx, ws)                # dx over x
    dr, dx2, dw2 = G(drs), G(), f32_buffer(H)
    rn.rmsnorm_bwd_residual(dy.t, dr.t, so.t, w, rr, dx2.t, dw2, ws)
    dri, dw2i = G(drs), f32_buffer(H)
    rn.rmsnorm_bwd_residual(dy.t, dri.t, so.t, w, rr, dri.t, dw2i, ws)   # dx over dresidual_out
    torch.cuda.synchronize()
    rtol = bwd_rtol(dtype)
    refb = oracle.rmsnorm_bwd(dys, s_np, w_np, eps, dtype)
    refr = oracle.rmsnorm_bwd(dys, s_np, w_np, eps, dtype, dres=drs)
    dec = (lambda b: b.astype(np.float64)) if dtype == "f32" else (lambda b: oracle.decode(b, dtype))
    for name, got, want, dwt in (("dx over dy", dyi, refb, dwi), ("dx over x", sx, refb, dwx),
                                 ("dx over dresidual_out", dri, refr, dw2i)):
        c = check_dx(dec(got.host()), want["dx"], want["dx_scale"], rtol)
        assert c["failed"] == 0, f"{name}: {c['failed']} failed, max rel {c['max_rel']}"
        c = check_dweight(dwt.cpu().numpy(), want["dweight"], want["dweight_abs"], rtol)
        assert c["failed"] == 0, f"{name}: dweight {c['failed']} failed"
        assert got.untouched_outside()
    assert torch.equal(dyi.t, dx.t) and torch.equal(dwi, dw)
    assert torch.equal(sx.t, dx.t) and torch.equal(dwx, dw)
    assert torch.equal(dri.t, dx2.t) and torch.equal(dw2i, dw2)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,offset", [(64, 0), (255, 0), (1000, 0), (2048, 0), (4096, 0), (4097, 0), (8192, 0),
                                      (32768, 0), (4096, 1)])
def test_in_place(oracle, dtype, H, offset):
    """In place on the lane-group, register-row, ring, split-row (H = 32768)
    and scalar-access paths."""
    check_in_place(oracle, dtype, rows_for(H, 200_000), H, offset)


@pytest.mark.parametrize("dtype,H,offset,M", [
    ("bf16", 10001, 1, 37),     # misaligned rows above the register budget: chunked forward and backward
    ("f16", 10001, 0, 21),
    ("f32", 65540, 0, 9),       # aligned rows above 256 KB: chunked, 16-byte accesses
    ("bf16", 131080, 0, 7),
    ("f32", 16384, 0, 33),      # split-row kernels (cluster per row)
])
def test_in_place_long_rows(oracle, dtype, H, offset, M):
    """In place on the kernels for rows longer than one CTA holds, where a
    row is read twice (chunked) or split over a cluster."""
    check_in_place(oracle, dtype, M, H, offset)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("H,offset", [(4096, 0), (4096, 1), (64, 0), (8192, 0)])
def test_storage_widening_exhaustive(dtype, H, offset):
    """Every 16-bit pattern passes through the kernels' widening exactly:
    with residual = -0, residual_out = x + (-0) must reproduce x bit for bit
    (NaNs as NaNs), through the 128-bit path (offset 0) and the scalar path."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    M = 65536 // H
    x = pats.reshape(M, H)
    r = np.full((M, H), 0x8000, np.uint16)
    gx = Guarded(M, H, H, dtype, offset).upload(x)
    gr = Guarded(M, H, H, dtype, offset).upload(r)
    gy, gs = Guarded(M, H, H, dtype, offset), Guarded(M, H, H, dtype, offset)
    rn.rmsnorm_fwd_residual(gx.t, gr.t, None, gy.t, gs.t, None, eps=1e-5)
    torch.cuda.synchronize()
    got = gs.host()
    isnan = ((x & 0x7FFF) > (0x7C00 if dtype == "f16" else 0x7F80))
    assert np.array_equal(got[~isnan], x[~isnan])
    nan_exp = 0x7C00 if dtype == "f16" else 0x7F80
    assert np.all(((got[isnan] & nan_exp) == nan_exp) & ((got[isnan] & (0x3FF if dtype == "f16" else 0x7F)) != 0))
    assert gs.untouched_outside() and gy.untouched_outside()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [1, 64, 255, 1000, 2048, 4096, 4097, 6144, 8192, 16384])
@pytest.mark.parametrize("weight", [True, False])
def test_bwd_residual_paths(oracle, dtype, H, weight):
    """Backward of the fused forward with the residual stream's gradient, every kernel path."""
    assert_bwd_ok(run_bwd_residual(oracle, dtype, rows_for(H), H, weight=weight, seed=H + 3))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,stride,offset", [(4096, 4096, 1), (6144, 6272, 0), (1000, 1001, 1)])
def test_bwd_residual_strides(oracle, dtype, H, stride, offset):
    assert_bwd_ok(run_bwd_residual(oracle, dtype, rows_for(H, 200_000), H, stride=stride, offset=offset,
                                   seed=stride))


def test_bwd_residual_dweight_matches_plain_backward(oracle):
    """The residual stream's gradient does not reach dweight: rmsnorm_bwd_residual's
    dweight equals rmsnorm_bwd's up to summation order (the two entry points may run
    different grids, hence different partial sums), i.e. within 1e-5 of sum |dy * xhat|."""
    M, H = 513, 4096
    rng = wl.rng_for(31)
    x_np, w_np = wl.matrix(rng, M, H, "bf16"), wl.weight(rng, H, "bf16")
    dy_np = wl.matrix(rng, M, H, "bf16")
    x, w = wl.to_torch(x_np, "bf16").cuda(), wl.to_torch(w_np, "bf16").cuda()
    dy = wl.to_torch(dy_np, "bf16").cuda()
    dres = wl.to_torch(wl.matrix(rng, M, H, "bf16"), "bf16").cuda()
    rrms = torch.empty(M, device="cuda")
    rn.rmsnorm_fwd(x, w, torch.empty_like(x), rrms, eps=1e-5)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, torch.bfloat16), dtype=torch.uint8, device="cuda")
    dw1, dw2 = torch.empty(H, device="cuda"), torch.empty(H, device="cuda")
    dx1, dx2 = torch.empty_like(x), torch.empty_like(x)
    rn.rmsnorm_bwd(dy, x, w, rrms, dx1, dw1, ws)
    rn.rmsnorm_bwd_residual(dy, dres, x, w, rrms, dx2, dw2, ws)
    torch.cuda.synchronize()
    scale = oracle.rmsnorm_bwd(dy_np, x_np, w_np, 1e-5, "bf16", want_dx=False)["dweight_abs"]
    diff = np.abs(dw1.cpu().numpy().astype(np.float64) - dw2.cpu().numpy())
    assert np.all(diff <= 1e-5 * scale)
    assert not torch.equal(dx1, dx2)
