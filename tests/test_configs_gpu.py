"""GPU parity on the five named workloads (and the long-row case) at full size, through the same
binding calls the benchmark times.  The oracle checks sampled rows (first,
last and 509 seeded random rows) element by element, the full dweight (an
fp64 sum over every row), and whole-tensor properties: every output finite,
padding columns and guard regions untouched."""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import Guarded, bwd_rtol, check_dweight, check_fwd_values, check_dx, device_vec, f32_buffer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def sample_rows(M, n=509, seed=77):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, M - 2, M - 1], rng.integers(0, M, n)]))


def fwd_check(oracle, cfg, x, r, w, gy, gs, rrms, rows, has_weight=True):
    dt, H, eps = cfg["dtype"], cfg["H"], cfg["eps"]
    ref = oracle.rmsnorm_fwd(np.ascontiguousarray(x[rows, :H]), w if has_weight else None, eps, dt,
                             residual=None if r is None else np.ascontiguousarray(r[rows, :H]))
    got = gy.host()[rows]
    c = check_fwd_values(got, ref["y"], dt, oracle)
    assert c["failed"] == 0, f"y: {c['failed']} failed elements of {got.size}"
    assert bool(torch.isfinite(gy.t).all())
    assert gy.untouched_outside()
    if r is not None:
        want = oracle.encode(ref["s"], dt)
        assert np.array_equal(gs.host()[rows].view(want.dtype), want), "residual_out not bit-exact"
        assert gs.untouched_outside()
    if rrms is not None:
        g = rrms.cpu().numpy()[rows].astype(np.float64)
        assert np.all(np.abs(g - ref["rrms"]) <= 1e-5 * ref["rrms"])
    return ref


def bwd_check(oracle, cfg, dy, xin, w, gdx, dw, rows):
    dt, H, eps = cfg["dtype"], cfg["H"], cfg["eps"]
    ref_rows = oracle.rmsnorm_bwd(np.ascontiguousarray(dy[rows, :H]), np.ascontiguousarray(xin[rows, :H]),
                                  w, eps, dt, want_dweight=False)
    got = gdx.host()[rows]
    got64 = got.astype(np.float64) if dt == "f32" else oracle.decode(got, dt)
    c = check_dx(got64, ref_rows["dx"], ref_rows["dx_scale"], bwd_rtol(dt))
    assert c["failed"] == 0, f"dx: {c['failed']} failed, max rel {c['max_rel']}"
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
    fwd_check(oracle, cfg, d["x"], None, d["w"], gy, None, None, np.arange(M))


def test_config2_fused_fwd_bf16(oracle):
    cfg = wl.CONFIGS[2]
    d = wl.generate(2)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    gx, gr = Guarded(M, H, S, dt).upload(d["x"]), Guarded(M, H, S, dt).upload(d["residual"])
    gy, gs = Guarded(M, H, S, dt), Guarded(M, H, S, dt)
    rn.rmsnorm_fwd_residual(gx.t, gr.t, device_vec(d["w"], dt), gy.t, gs.t, None, eps=cfg["eps"])
    torch.cuda.synchronize()
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, None, sample_rows(M))


def test_config3_dit_mix_bf16(oracle):
    cfg = wl.CONFIGS[3]
    d = wl.generate(3)
    M, H, S, dt = cfg["M"], cfg["H"], cfg["stride"], cfg["dtype"]
    wd = device_vec(d["w"], dt)
    for k, weighted in ((0, True), (1, False)):
        gx, gy = Guarded(M, H, S, dt).upload(d["xs"][k]), Guarded(M, H, S, dt)
        rn.rmsnorm_fwd(gx.t, wd if weighted else None, gy.t, None, eps=cfg["eps"])
        torch.cuda.synchronize()
        fwd_check(oracle, cfg, d["xs"][k], None, d["w"], gy, None, None, sample_rows(M, seed=k),
                  has_weight=weighted)
    hcfg = dict(cfg, M=cfg["head_M"], H=cfg["head_H"], stride=cfg["head_H"])
    hM, hH = hcfg["M"], hcfg["H"]
    gx, gy = Guarded(hM, hH, hH, dt).upload(d["head_x"]), Guarded(hM, hH, hH, dt)
    rn.rmsnorm_fwd(gx.t, device_vec(d["head_w"], dt), gy.t, None, eps=cfg["eps"])
    torch.cuda.synchronize()
    fwd_check(oracle, hcfg, d["head_x"], None, d["head_w"], gy, None, None, sample_rows(hM, 2045))


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
    rows = sample_rows(M)
    fwd_check(oracle, cfg, d["x"], None, d["w"], gy, None, rrms, rows)
    bwd_check(oracle, cfg, d["dy"], d["x"], d["w"], gdx, dw, rows)


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
    rows = sample_rows(M)
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, rrms, rows)
    assert gx.untouched_outside() and gr.untouched_outside()
    s_host = np.full((M, S), 0, np.uint16)
    s_host[:, :H] = gs.host()
    bwd_check(oracle, cfg, d["dy"], s_host, d["w"], gdx, dw, rows)


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
    rows = sample_rows(M)
    fwd_check(oracle, cfg, d["x"], d["residual"], d["w"], gy, gs, rrms, rows)
    bwd_check(oracle, cfg, d["dy"], gs.host(), d["w"], gdx, dw, rows)
