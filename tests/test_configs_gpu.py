"""GPU parity on the five named workloads (and the long-row and odd-row cases) at full size, through the same
binding calls the benchmark times.  The oracle checks every row element by element (in blocks of
rows, to bound host memory): y within the forward tolerance, residual_out bit-exact, rrms within
1e-5, dx within the backward tolerance, and the full dweight (an fp64 sum over every row); plus
whole-tensor properties: every output finite, padding columns and guard regions untouched."""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import Guarded, bwd_rtol, check_dweight, check_fwd_values, check_dx, device_vec, f32_buffer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BLOCK_ELEMS = 1 << 25   # rows per oracle block: about 32 M elements (a few hundred MB of fp64 results)


def row_blocks(M, H):
    step = max(1, BLOCK_ELEMS // H)
    for r0 in range(0, M, step):
        yield r0, min(M, r0 + step)


def fwd_check(oracle, cfg, x, r, w, gy, gs, rrms, has_weight=True):
    dt, H, eps, M = cfg["dtype"], cfg["H"], cfg["eps"], cfg["M"]
    got_y = gy.host()
    got_s = gs.host() if r is not None else None
    got_rr = rrms.cpu().numpy().astype(np.float64) if rrms is not None else None
    for r0, r1 in row_blocks(M, H):
        ref = oracle.rmsnorm_fwd(np.ascontiguousarray(x[r0:r1, :H]), w if has_weight else None, eps, dt,
                                 residual=None if r is None else np.ascontiguousarray(r[r0:r1, :H]))
        c = check_fwd_values(got_y[r0:r1], ref["y"], dt, oracle)
        assert c["failed"] == 0, f"y rows {r0}-{r1}: {c['failed']} failed elements"
        if r is not None:
            want = oracle.encode(ref["s"], dt)
            assert np.array_equal(got_s[r0:r1].view(want.dtype), want), f"residual_out rows {r0}-{r1} not bit-exact"
        if got_rr is not None:
            assert np.all(np.abs(got_rr[r0:r1] - ref["rrms"]) <= 1e-5 * ref["rrms"]), f"rrms rows {r0}-{r1}"
    assert bool(torch.isfinite(gy.t).all())
    assert gy.untouched_outside()
    if r is not None:
        assert gs.untouched_outside()


def bwd_check(oracle, cfg, dy, xin, w, gdx, dw):
    dt, H, eps, M = cfg["dtype"], cfg["H"], cfg["eps"], cfg["M"]
    got = gdx.host()
    for r0, r1 in row_blocks(M, H):
        ref = oracle.rmsnorm_bwd(np.ascontiguousarray(dy[r0:r1, :H]), np.ascontiguousarray(xin[r0:r1, :H]),
                                 w, eps, dt, want_dweight=False)
        g = got[r0:r1]
        got64 = g.astype(np.float64) if dt == "f32" else oracle.decode(g, dt)
        c = check_dx(got64, ref["dx"], ref["dx_scale"], bwd_rtol(dt))
        assert c["failed"] == 0, f"dx rows {r0}-{r1}: {c['failed']} failed, max rel {c['max_rel']}"
    assert bool(torch.isfinite(gdx.t).all())
    assert gdx.untouched_outside()
    full = oracle.rmsnorm_bwd(dy[:, :H], xin[:, :H], w, eps, dt, want_dx=False)
    c = check_dweight(dw.cpu().numpy(), full["dweight"], full["dweight_abs"], bwd_rtol(dt))
    assert c["failed"] == 0, f"dweight: {c['failed']} failed, max rel {c['max_rel']}"


def test_config1_fwd_f32(oracle):
    cfg = wl.CONFIGS[1]
    d = wl.generate(1)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    gx = Guarded(M, H, S, dt).upload(d["x"])
    gy = Guarded(M, H, S, dt)
    rn.rmsnorm_fwd(gx.t, device_vec(d["w"], dt), gy.t, None, eps=cfg["eps"])
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], None, d["w"], gy, None, None)


def test_config2_fused_fwd_bf16(oracle):
    cfg = wl.CONFIGS[2]
    d = wl.generate(2)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    gx, gr = Guarded(M, H, S, dt).upload(d["x"]), Guarded(M, H, S, dt).upload(d["residual"])
    gy, gs = Guarded(M, H, S, dt), Guarded(M, H, S, dt)
    rn.rmsnorm_fwd_residual(gx.t, gr.t, device_vec(d["w"], dt), gy.t, gs.t, None, eps=cfg["eps"])
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, None)


def test_config3_dit_mix_bf16(oracle):
    cfg = wl.CONFIGS[3]
    d = wl.generate(3)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    wd = device_vec(d["w"], dt)
    for k, weighted in ((0, True), (1, False)):
        gx, gy = Guarded(M, H, S, dt).upload(d["xs"][k]), Guarded(M, H, S, dt)
        rn.rmsnorm_fwd(gx.t, wd if weighted else None, gy.t, None, eps=cfg["eps"])
        torch.cuda.synchronize()
        fwd_check(oracle, cfg, d["xs"][k], None, d["w"], gy, None, None, has_weight=weighted)
    hcfg = dict(cfg, M=cfg["head_M"], H=cfg["head_H"], stride=cfg["head_H"])
    hM, hH = hcfg["M"], hcfg["H"]
    gx, gy = Guarded(hM, hH, hH, dt).upload(d["head_x"]), Guarded(hM, hH, hH, dt)
    rn.rmsnorm_fwd(gx.t, device_vec(d["head_w"], dt), gy.t, None, eps=cfg["eps"])
    torch.cuda.synchronize()
    fwd_check(oracle, hcfg, d["head_x"], None, d["head_w"], gy, None, None)


def test_config4_fwd_bwd_bf16(oracle):
    cfg = wl.CONFIGS[4]
    d = wl.generate(4)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    gx, gy = Guarded(M, H, S, dt).upload(d["x"]), Guarded(M, H, S, dt)
    wd = device_vec(d["w"], dt)
    rrms = f32_buffer(M)
    rn.rmsnorm_fwd(gx.t, wd, gy.t, rrms, eps=cfg["eps"])
    gdy, gdx = Guarded(M, H, S, dt).upload(d["dy"]), Guarded(M, H, S, dt)
    dw = f32_buffer(H)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, wl.torch_dtype(dt)), dtype=torch.uint8, device="cuda")
    rn.rmsnorm_bwd(gdy.t, gx.t, wd, rrms, gdx.t, dw, ws)
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], None, d["w"], gy, None, rrms)
    bwd_check(oracle, cfg, d["dy"], d["x"], d["w"], gdx, dw)


def test_config5_fused_fwd_bwd_f16_padded(oracle):
    cfg = wl.CONFIGS[5]
    d = wl.generate(5)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    assert S == 6272 and H == 6144
    gx, gr = Guarded(M, H, S, dt).upload(d["x"]), Guarded(M, H, S, dt).upload(d["residual"])
    gy, gs = Guarded(M, H, S, dt), Guarded(M, H, S, dt)
    wd = device_vec(d["w"], dt)
    rrms = f32_buffer(M)
    rn.rmsnorm_fwd_residual(gx.t, gr.t, wd, gy.t, gs.t, rrms, eps=cfg["eps"])
    gdy, gdx = Guarded(M, H, S, dt).upload(d["dy"]), Guarded(M, H, S, dt)
    dw = f32_buffer(H)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, wl.torch_dtype(dt)), dtype=torch.uint8, device="cuda")
    rn.rmsnorm_bwd(gdy.t, gs.t, wd, rrms, gdx.t, dw, ws)
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, rrms)
    assert gx.untouched_outside() and gr.untouched_outside()
    s_host = np.full((M, S), 0, np.uint16)
    s_host[:, :H] = gs.host()
    bwd_check(oracle, cfg, d["dy"], s_host, d["w"], gdx, dw)


def test_long_rows_fused_fwd_bwd_bf16(oracle):
    """The long-row measurement case (bf16 4096 x 32768, 64 KB rows: the
    split-row kernels) at full size, as the benchmark's long_rows step runs it."""
    cfg = wl.CONFIGS[6]
    d = wl.generate(6)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    gx, gr = Guarded(M, H, S, dt).upload(d["x"]), Guarded(M, H, S, dt).upload(d["residual"])
    gy, gs = Guarded(M, H, S, dt), Guarded(M, H, S, dt)
    wd = device_vec(d["w"], dt)
    rrms = f32_buffer(M)
    rn.rmsnorm_fwd_residual(gx.t, gr.t, wd, gy.t, gs.t, rrms, eps=cfg["eps"])
    gdy, gdx = Guarded(M, H, S, dt).upload(d["dy"]), Guarded(M, H, S, dt)
    dw = f32_buffer(H)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, wl.torch_dtype(dt)), dtype=torch.uint8, device="cuda")
    rn.rmsnorm_bwd(gdy.t, gs.t, wd, rrms, gdx.t, dw, ws)
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, rrms)
    bwd_check(oracle, cfg, d["dy"], gs.host(), d["w"], gdx, dw)


def test_odd_rows_fused_fwd_bwd_bf16(oracle):
    """The misaligned-row measurement case (bf16 16384 x 4095, rows contiguous,
    so they start at every element offset within 16 bytes: the aligned-frame
    kernels) at full size, as the benchmark's odd_rows step runs it."""
    cfg = wl.CONFIGS[7]
    d = wl.generate(7)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    gx, gr = Guarded(M, H, S, dt).upload(d["x"]), Guarded(M, H, S, dt).upload(d["residual"])
    gy, gs = Guarded(M, H, S, dt), Guarded(M, H, S, dt)
    wd = device_vec(d["w"], dt)
    rrms = f32_buffer(M)
    rn.rmsnorm_fwd_residual(gx.t, gr.t, wd, gy.t, gs.t, rrms, eps=cfg["eps"])
    gdy, gdx = Guarded(M, H, S, dt).upload(d["dy"]), Guarded(M, H, S, dt)
    dw = f32_buffer(H)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, wl.torch_dtype(dt)), dtype=torch.uint8, device="cuda")
    rn.rmsnorm_bwd(gdy.t, gs.t, wd, rrms, gdx.t, dw, ws)
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, rrms)
    assert gx.untouched_outside() and gr.untouched_outside()
    bwd_check(oracle, cfg, d["dy"], gs.host(), d["w"], gdx, dw)
