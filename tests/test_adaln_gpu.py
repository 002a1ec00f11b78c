"""GPU parity of rmsnorm_adaln_fwd against the fp64 oracle: every kernel path
(register rows for H < 256 and up to the register budget, a warp per aligned
row of 512 B to 2 KB when conditioning rows serve 1024 rows or more, the
bulk-copy ring for aligned rows -- conditioning staged beside x, or held in
registers when each conditioning row spans four of a CTA's row strides -- a
cluster of CTAs per aligned row of 32-256 KB, and the chunked two-pass kernel
for unaligned rows above the budget), per-token and broadcast conditioning rows,
padded and misaligned layouts, in place, with guard bands around every
buffer.

Tolerance: y = t + shift may cancel, so each element is compared against
y_scale = |t| + |shift| from the oracle: fp32 within 1e-5 * y_scale; f16 and
bf16 within 1 ulp of the oracle's value rounded to the storage type, or
within 1e-5 * y_scale of it.  rrms within 1e-5 relative.
"""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import Guarded, check_scaled_values, device_vec, f32_buffer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]
H_ADALN = [1, 7, 64, 255, 256, 1000, 1152, 2048, 3072, 4096, 4097, 6144, 8192, 10001, 16384, 32768]


def rows_for(H, cap=300_000):
    return int(max(3, min(257, cap // H))) | 1


def run_adaln(oracle, dtype, M, H, rows_per_cond=1, stride=None, cond_stride=None, weight=True,
              offset=0, cond_offset=0, eps=1e-6, seed=0, in_place=False, x_np=None, sc_np=None, sh_np=None,
              w_np=None):
    stride = H if stride is None else stride
    cond_stride = H if cond_stride is None else cond_stride
    n_cond = -(-M // rows_per_cond)
    rng = wl.rng_for(seed)
    x = wl.matrix(rng, M, H, dtype, stride) if x_np is None else x_np
    sc = wl.conditioning(rng, n_cond, H, dtype, cond_stride) if sc_np is None else sc_np
    sh = wl.conditioning(rng, n_cond, H, dtype, cond_stride) if sh_np is None else sh_np
    w = (wl.weight(rng, H, dtype) if w_np is None else w_np) if weight else None
    gx = Guarded(M, H, stride, dtype, offset).upload(x)
    gsc = Guarded(n_cond, H, cond_stride, dtype, cond_offset).upload(sc)
    gsh = Guarded(n_cond, H, cond_stride, dtype, cond_offset).upload(sh)
    gy = gx if in_place else Guarded(M, H, stride, dtype, offset)
    wd = device_vec(w, dtype, offset) if weight else None
    rrms = f32_buffer(M, offset)
    rn.rmsnorm_adaln_fwd(gx.t, wd, gsc.t, gsh.t, gy.t, rows_per_cond=rows_per_cond, rrms=rrms, eps=eps)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_adaln_fwd(x[:, :H], w, sc[:, :H], sh[:, :H], eps, dtype, rows_per_cond=rows_per_cond)
    res = {"y": check_scaled_values(gy.host(), ref["y"], ref["y_scale"], dtype, oracle)}
    got = rrms.cpu().numpy().astype(np.float64)
    res["rrms_bad"] = int(np.sum(~(np.abs(got - ref["rrms"]) <= 1e-5 * ref["rrms"])))
    assert gy.untouched_outside() and gsc.untouched_outside() and gsh.untouched_outside()
    if not in_place:
        assert gx.untouched_outside()
        assert torch.equal(gx.flat.view(torch.int16 if dtype != "f32" else torch.int32),
                           gx.initial.view(torch.int16 if dtype != "f32" else torch.int32))
    res.update(gy=gy, x=x, sc=sc, sh=sh, w=w, rrms=rrms)
    return res


def assert_ok(res):
    assert res["y"]["failed"] == 0, f"y: {res['y']['failed']} failed, max rel {res['y']['max_rel']}"
    assert res["rrms_bad"] == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", H_ADALN)
@pytest.mark.parametrize("rows_per_cond", [1, 5, 64])
def test_adaln_paths(oracle, dtype, H, rows_per_cond):
    assert_ok(run_adaln(oracle, dtype, rows_for(H), H, rows_per_cond=rows_per_cond, seed=H + rows_per_cond))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 2048, 4096, 32768])
def test_adaln_without_weight(oracle, dtype, H):
    assert_ok(run_adaln(oracle, dtype, rows_for(H), H, weight=False, seed=7))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,stride,cond_stride,offset,cond_offset", [
    (1152, 1160, 1152, 0, 0), (4096, 4160, 4104, 0, 0), (4096, 4096, 4096, 0, 1), (4096, 4096, 4097, 0, 0),
    (4096, 4096, 4096, 1, 0), (3072, 3075, 3072, 0, 0), (64, 72, 80, 0, 0), (16384, 16392, 16400, 0, 0),
    (8192, 8192, 12288, 0, 0)])
def test_adaln_strides_and_misalignment(oracle, dtype, H, stride, cond_stride, offset, cond_offset):
    """Padded rows, a conditioning stride of its own, and layouts that leave
    the 128-bit path (misaligned scale/shift, odd strides) or the ring."""
    for rpc in (1, 4):
        assert_ok(run_adaln(oracle, dtype, rows_for(H, 150_000), H, rows_per_cond=rpc, stride=stride,
                            cond_stride=cond_stride, offset=offset, cond_offset=cond_offset, seed=stride + rpc))


@pytest.mark.parametrize("dtype,H,M,rpc", [("bf16", 1152, 20001, 4096), ("bf16", 4096, 6001, 1000),
                                           ("f16", 3072, 9001, 1), ("f32", 4096, 3001, 3001),
                                           ("bf16", 64, 50001, 7), ("bf16", 1024, 30001, 512),
                                           ("f32", 512, 20001, 64), ("f16", 256, 70001, 9),
                                           ("bf16", 1024, 30001, 2048), ("f16", 512, 40001, 4096),
                                           ("bf16", 2048, 20001, 5000)])
def test_adaln_grid_stride(oracle, dtype, H, M, rpc):
    """More rows than resident CTAs; conditioning rows shared by many rows,
    a ragged last sequence, and a single conditioning row for all rows."""
    assert_ok(run_adaln(oracle, dtype, M, H, rows_per_cond=rpc, seed=M))


@pytest.mark.parametrize("dtype,H,M,rpc", [("bf16", 2048, 12289, 6144), ("bf16", 2048, 12288, 6144),
                                           ("f16", 4096, 20001, 1000), ("bf16", 2048, 9001, 37),
                                           ("f32", 2048, 8191, 2000), ("bf16", 8192, 4099, 1024)])
def test_adaln_conditioning_groups(oracle, dtype, H, M, rpc):
    """Few conditioning rows on the bulk-copy ring: each gets its own group of
    CTAs, sized by its rows (a ragged last row gets a small group), every
    row of x processed once with its own conditioning row."""
    assert_ok(run_adaln(oracle, dtype, M, H, rows_per_cond=rpc, seed=M + rpc))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 2048, 4096, 8192, 32768])
def test_adaln_broadcast_is_bitwise_repeated_rows(oracle, dtype, H):
    """rows_per_cond = S gives the same bits as the conditioning rows repeated S times."""
    S = 6
    M = (rows_for(H, 100_000) // S + 1) * S - 2          # ragged last sequence
    n = -(-M // S)
    rng = wl.rng_for(11)
    sc = wl.conditioning(rng, n, H, dtype)
    sh = wl.conditioning(rng, n, H, dtype)
    a = run_adaln(oracle, dtype, M, H, rows_per_cond=S, sc_np=sc, sh_np=sh, seed=11)
    b = run_adaln(oracle, dtype, M, H, rows_per_cond=1, x_np=a["x"], w_np=a["w"],
                  sc_np=np.repeat(sc, S, axis=0)[:M], sh_np=np.repeat(sh, S, axis=0)[:M], seed=11)
    assert_ok(a)
    assert torch.equal(a["gy"].t, b["gy"].t)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [1024, 2048, 3072, 4096, 32768])
def test_adaln_zero_conditioning_is_bitwise_rmsnorm(oracle, dtype, H):
    """scale = shift = 0: y * (1 + 0) + 0 = y exactly, so the result equals
    rmsnorm_fwd's bit for bit.  One conditioning row serves every row, which
    takes the same kernel family as the plain forward from H = 256 up (below
    that the plain forward reduces a row in a lane group instead; a warp per
    row needs conditioning rows serving 1024 rows, hence M >= 1025)."""
    M = max(rows_for(H), 1025)
    z = wl.to_storage(np.zeros((1, H), np.float32), dtype)
    a = run_adaln(oracle, dtype, M, H, rows_per_cond=M, sc_np=z, sh_np=z, seed=13)
    assert_ok(a)
    xd = wl.to_torch(a["x"], dtype).cuda()
    wd = wl.to_torch(a["w"], dtype).cuda()
    y = torch.empty_like(xd)
    q = torch.empty(M, device="cuda")
    rn.rmsnorm_fwd(xd, wd, y, q, eps=1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a["gy"].t, y)
    assert torch.equal(a["rrms"], q)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [64, 1152, 4096, 8192, 32768])
def test_adaln_in_place_matches_out_of_place(oracle, dtype, H):
    a = run_adaln(oracle, dtype, rows_for(H), H, rows_per_cond=3, seed=17)
    b = run_adaln(oracle, dtype, rows_for(H), H, rows_per_cond=3, x_np=a["x"], sc_np=a["sc"], sh_np=a["sh"],
                  w_np=a["w"], in_place=True, seed=17)
    assert_ok(b)
    assert torch.equal(a["gy"].t, b["gy"].t)


def test_adaln_rejects_bad_conditioning(oracle):
    x = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    sc = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rn.RmsnormError):   # shift overlapping y
        rn.rmsnorm_adaln_fwd(x, None, sc, y, y)
    with pytest.raises(ValueError):        # wrong number of conditioning rows
        rn.rmsnorm_adaln_fwd(x, None, sc[:3], sc[:3], y, rows_per_cond=2)
