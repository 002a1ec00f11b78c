"""GPU parity of layernorm_fwd and layernorm_fwd_residual against the fp64
oracle: every kernel path (the register kernel for H < 256, for rows up to the
register budget and for unaligned rows; the bulk-copy ring for aligned rows
of 4 KB and more (8 KB fused) up to 32 KB; a cluster of CTAs per aligned row
of 32-256 KB; the chunked kernel for unaligned rows above the budget), with and
without weight and bias, padded and misaligned layouts, in place, with guard
bands around every buffer.

Tolerances: y is formed by a mean subtraction and a bias add that can cancel,
so each element is compared against y_scale = (|s| + mean|s|) * rstd * |w| +
|b| from the oracle: fp32 within 1e-5 * y_scale; f16/bf16 within 1 ulp of the
oracle rounded to the storage type, or within 1e-5 * y_scale.  residual_out
bit-exact with the oracle's sum rounded; mean within 1e-6 * mean|s| (absolute,
the sum's condition); rstd within 1e-5 relative.
"""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import Guarded, check_scaled_values, device_vec, f32_buffer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]
H_LN = [1, 7, 64, 255, 256, 1000, 1024, 2048, 3072, 4096, 4097, 6144, 8192, 10001, 16384, 32768]


def rows_for(H, cap=300_000):
    return int(max(3, min(257, cap // H))) | 1


def run_ln(oracle, dtype, M, H, residual=False, weight=True, bias=True, stride=None, offset=0, eps=1e-5, seed=0,
           in_place=False, x_np=None, r_np=None, w_np=None, b_np=None, shift=0.0, w_offset=None):
    """w_offset: the weight's and bias's own element offset (default: offset)."""
    stride = H if stride is None else stride
    w_offset = offset if w_offset is None else w_offset
    rng = wl.rng_for(seed)
    if x_np is None:
        x = wl.matrix(rng, M, H, dtype, stride)
        if shift:   # rows with a large common offset: the mean matters
            x = wl.to_storage(oracle.decode(x, dtype).astype(np.float32) + np.float32(shift), dtype)
    else:
        x = x_np
    r = (wl.matrix(rng, M, H, dtype, stride) if r_np is None else r_np) if residual else None
    w = (wl.weight(rng, H, dtype) if w_np is None else w_np) if weight else None
    b = (wl.conditioning(rng, 1, H, dtype)[0] if b_np is None else b_np) if bias else None
    gx = Guarded(M, H, stride, dtype, offset).upload(x)
    gr = Guarded(M, H, stride, dtype, offset).upload(r) if residual else None
    gy = gx if in_place else Guarded(M, H, stride, dtype, offset)
    gs = (gr if in_place else Guarded(M, H, stride, dtype, offset)) if residual else None
    wd = device_vec(w, dtype, w_offset) if weight else None
    bd = device_vec(b, dtype, w_offset) if bias else None
    mean = f32_buffer(M, offset)
    rstd = f32_buffer(M, offset)
    if residual:
        rn.layernorm_fwd_residual(gx.t, gr.t, wd, bd, gy.t, gs.t, mean, rstd, eps=eps)
    else:
        rn.layernorm_fwd(gx.t, wd, bd, gy.t, mean, rstd, eps=eps)
    torch.cuda.synchronize()
    ref = oracle.layernorm_fwd(x[:, :H], w, b, eps, dtype, residual=None if r is None else r[:, :H])
    res = {"y": check_scaled_values(gy.host(), ref["y"], ref["y_scale"], dtype, oracle)}
    assert gy.untouched_outside()
    if residual:
        want_s = oracle.encode(ref["s"], dtype)
        view = np.uint32 if dtype == "f32" else np.uint16
        res["s_mismatch"] = int(np.sum(gs.host().view(view) != want_s.view(view)))
        assert gs.untouched_outside()
    mean_abs = np.abs(ref["s"]).mean(axis=1)
    got_m = mean.cpu().numpy().astype(np.float64)
    res["mean_bad"] = int(np.sum(~(np.abs(got_m - ref["mean"]) <= 1e-6 * mean_abs + 1e-30)))
    got_r = rstd.cpu().numpy().astype(np.float64)
    res["rstd_bad"] = int(np.sum(~(np.abs(got_r - ref["rstd"]) <= 1e-5 * ref["rstd"])))
    res.update(gy=gy, gs=gs, x=x, r=r, w=w, b=b, mean=mean, rstd=rstd)
    return res


def assert_ok(res):
    assert res["y"]["failed"] == 0, f"y: {res['y']['failed']} failed, max rel {res['y']['max_rel']}"
    assert res.get("s_mismatch", 0) == 0, f"residual_out: {res['s_mismatch']} elements not bit-exact"
    assert res["mean_bad"] == 0 and res["rstd_bad"] == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", H_LN)
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("affine", [True, False])
def test_layernorm_paths(oracle, dtype, H, residual, affine):
    assert_ok(run_ln(oracle, dtype, rows_for(H), H, residual=residual, weight=affine, bias=affine, seed=H + 7))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 1024, 4096, 32768])
def test_layernorm_offset_rows(oracle, dtype, H):
    """Rows with a large common offset (mean >> spread): the mean subtraction cancels."""
    assert_ok(run_ln(oracle, dtype, rows_for(H), H, residual=True, seed=H, shift=24.0))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,stride,offset", [
    (64, 72, 0), (64, 67, 0), (1000, 1003, 0), (1024, 1032, 0), (2048, 2049, 1), (4096, 4160, 0),
    (4096, 4096, 1), (6144, 6272, 0), (200, 200, 3), (16384, 16392, 0), (16384, 16385, 1)])
def test_layernorm_strides_and_misalignment(oracle, dtype, H, stride, offset):
    for residual in (False, True):
        assert_ok(run_ln(oracle, dtype, rows_for(H, 150_000), H, residual=residual, stride=stride, offset=offset,
                         seed=stride + offset))


@pytest.mark.parametrize("dtype,H,M", [("bf16", 1024, 40001), ("bf16", 4096, 20001), ("f16", 64, 70001),
                                       ("f32", 2048, 9001), ("bf16", 32768, 401), ("f32", 8192, 3001)])
def test_layernorm_grid_stride(oracle, dtype, H, M):
    for residual in (False, True):
        assert_ok(run_ln(oracle, dtype, M, H, residual=residual, seed=M))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 1024, 4096, 32768])
def test_layernorm_absent_affine_is_bitwise_ones_and_zeros(oracle, dtype, H):
    M = rows_for(H)
    a = run_ln(oracle, dtype, M, H, weight=False, bias=False, seed=3)
    ones = wl.to_storage(np.ones(H, np.float32), dtype)
    zeros = wl.to_storage(np.zeros(H, np.float32), dtype)
    b = run_ln(oracle, dtype, M, H, x_np=a["x"], w_np=ones, b_np=zeros, seed=3)
    assert torch.equal(a["gy"].t, b["gy"].t)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 1024, 4096, 32768])
def test_layernorm_residual_fusion_equals_add_then_norm(oracle, dtype, H):
    """With sums exact in the storage type, fusing the add changes nothing (bitwise)."""
    M = rows_for(H)
    rng = np.random.default_rng(H)
    xv = rng.integers(-60, 60, (M, H)).astype(np.float32)
    rv = rng.integers(-60, 60, (M, H)).astype(np.float32)
    x, r = wl.to_storage(xv, dtype), wl.to_storage(rv, dtype)
    s = wl.to_storage(xv + rv, dtype)
    fused = run_ln(oracle, dtype, M, H, residual=True, x_np=x, r_np=r, seed=1)
    plain = run_ln(oracle, dtype, M, H, residual=False, x_np=s, w_np=fused["w"], b_np=fused["b"], seed=1)
    assert torch.equal(fused["gy"].t, plain["gy"].t)
    assert torch.equal(fused["rstd"], plain["rstd"]) and torch.equal(fused["mean"], plain["mean"])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 1024, 4096, 8192, 32768])
@pytest.mark.parametrize("residual", [False, True])
def test_layernorm_in_place_matches_out_of_place(oracle, dtype, H, residual):
    a = run_ln(oracle, dtype, rows_for(H), H, residual=residual, seed=17)
    b = run_ln(oracle, dtype, rows_for(H), H, residual=residual, x_np=a["x"], r_np=a["r"], w_np=a["w"],
               b_np=a["b"], in_place=True, seed=17)
    assert_ok(b)
    assert torch.equal(a["gy"].t, b["gy"].t)
    if residual:
        assert torch.equal(a["gs"].t, b["gs"].t)


def test_layernorm_fp16_outliers(oracle):
    """|s| up to 300: s^2 exceeds the fp16 maximum; binary32 accumulation keeps the result finite."""
    H = 4096
    M = rows_for(H)
    x = wl.matrix(wl.rng_for(5), M, H, "f16", outlier_frac=0.05)
    res = run_ln(oracle, "f16", M, H, residual=True, x_np=x, seed=5)
    assert_ok(res)
    assert bool(torch.isfinite(res["gy"].t).all())
