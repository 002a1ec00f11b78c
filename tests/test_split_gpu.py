"""GPU parity of the split-row kernels (a thread-block cluster per aligned row
of 32-256 KB, one column segment per CTA, the row's sums exchanged through
distributed shared memory) against the fp64 oracle, and of the two-pass
chunked kernels that still take aligned rows above 256 KB.

Row lengths are chosen for the segment arithmetic: 16392 bf16 (32784 B,
2049 groups: four CTAs of 513, 513, 513 and 510 groups), 24576 and 32768
(four CTAs), 40000 (eight CTAs of 625), 65536 (eight of 1024), 131072 (eight
of 2048, four groups per thread), 131080 (16385 groups: the chunked kernel);
binary32 8196, 12288, 16384, 32768, 65536 and 65540 likewise.  Tolerances are
those of the other parity tests (forward within 1 ulp / 1e-5, residual_out
bit-exact, dx and dweight within the backward's bounds).
"""
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from test_adaln_gpu import assert_ok as assert_adaln_ok
from test_adaln_gpu import run_adaln
from test_layernorm_gpu import assert_ok as assert_ln_ok
from test_layernorm_gpu import run_ln
from test_parity_gpu import assert_bwd_ok, assert_fwd_ok, run_bwd, run_bwd_residual, run_fwd

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

H_SPLIT = {"bf16": [16392, 24576, 32768, 40000, 65536, 131072, 131080],
           "f16": [16392, 32768, 40000, 131072],
           "f32": [8196, 12288, 16384, 32768, 65536, 65540]}
CASES = [(dt, H) for dt, hs in H_SPLIT.items() for H in hs]


def rows_for(H, cap=600_000):
    return int(max(3, min(65, cap // H))) | 1


@pytest.mark.parametrize("dtype,H", CASES)
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("weight", [True, False])
def test_split_fwd(oracle, dtype, H, residual, weight):
    assert_fwd_ok(run_fwd(oracle, dtype, rows_for(H), H, residual=residual, weight=weight, seed=H + residual))


@pytest.mark.parametrize("dtype,H,M", [("bf16", 32768, 401), ("f32", 65536, 97), ("f16", 40000, 203),
                                       ("bf16", 131072, 61)])
@pytest.mark.parametrize("residual", [False, True])
def test_split_fwd_grid_stride(oracle, dtype, H, M, residual):
    """More rows than resident clusters: every cluster takes several rows."""
    assert_fwd_ok(run_fwd(oracle, dtype, M, H, residual=residual, seed=M))


@pytest.mark.parametrize("dtype,H,stride", [("bf16", 32768, 32776), ("f32", 16384, 16388), ("f16", 24576, 25600)])
def test_split_fwd_padded_rows(oracle, dtype, H, stride):
    """Row strides above H (16-byte multiples): the segments start at row * stride."""
    for residual in (False, True):
        assert_fwd_ok(run_fwd(oracle, dtype, rows_for(H), H, stride=stride, residual=residual, seed=stride))


@pytest.mark.parametrize("dtype,H", CASES)
@pytest.mark.parametrize("weight", [True, False])
def test_split_bwd(oracle, dtype, H, weight):
    assert_bwd_ok(run_bwd(oracle, dtype, rows_for(H), H, weight=weight, seed=H + 2))


@pytest.mark.parametrize("dtype,H", [("bf16", 32768), ("f16", 40000), ("f32", 16384), ("bf16", 131072)])
def test_split_bwd_residual(oracle, dtype, H):
    """Backward of the fused forward with the residual stream's gradient added."""
    assert_bwd_ok(run_bwd_residual(oracle, dtype, rows_for(H), H, seed=H + 3))


@pytest.mark.parametrize("dtype,H,M", [("bf16", 32768, 401), ("f32", 65536, 97), ("f16", 40000, 203)])
def test_split_bwd_grid_stride(oracle, dtype, H, M):
    assert_bwd_ok(run_bwd(oracle, dtype, M, H, seed=M + 5))


@pytest.mark.parametrize("dtype,H", [("bf16", 32768), ("f32", 65536)])
def test_split_dweight_deterministic(oracle, dtype, H):
    a = run_bwd(oracle, dtype, 301, H, seed=8)
    b = run_bwd(oracle, dtype, 301, H, seed=8)
    assert torch.equal(a["dw_t"], b["dw_t"])
    assert torch.equal(a["gdx"].t, b["gdx"].t)


@pytest.mark.parametrize("dtype,H", [("bf16", 32768), ("bf16", 40000), ("f32", 16384), ("f16", 131072),
                                     ("bf16", 131080)])
@pytest.mark.parametrize("residual", [False, True])
def test_split_layernorm(oracle, dtype, H, residual):
    """Two cluster reductions per row (the sum, then the centred sum of squares)."""
    assert_ln_ok(run_ln(oracle, dtype, rows_for(H), H, residual=residual, seed=H + residual))
    assert_ln_ok(run_ln(oracle, dtype, rows_for(H), H, residual=residual, seed=H + 7, shift=40.0))


@pytest.mark.parametrize("dtype,H", [("bf16", 32768), ("f32", 16384), ("f16", 65536), ("bf16", 131080)])
@pytest.mark.parametrize("rows_per_cond", [1, 5, 10_000])
def test_split_adaln(oracle, dtype, H, rows_per_cond):
    """Per-token conditioning staged beside x, and conditioning shared by many rows."""
    M = rows_for(H)
    assert_adaln_ok(run_adaln(oracle, dtype, M, H, rows_per_cond=rows_per_cond, seed=H + rows_per_cond))


def test_split_adaln_shared_grid_stride(oracle):
    """Conditioning rows shared by 4 x the cluster count: the cluster's rows
    cross conditioning-row boundaries while their w * (1 + scale) is cached."""
    assert_adaln_ok(run_adaln(oracle, "bf16", 2049, 32768, rows_per_cond=500, seed=11))


@pytest.mark.parametrize("dtype,H", [("bf16", 32768), ("f32", 32768)])
def test_split_in_place(dtype, H):
    """y over x and residual_out over the residual: the bits of separate outputs."""
    M = rows_for(H)
    rng = wl.rng_for(H)
    dt = wl.torch_dtype(dtype)
    x = wl.to_torch(wl.matrix(rng, M, H, dtype), dtype).cuda()
    r = wl.to_torch(wl.matrix(rng, M, H, dtype), dtype).cuda()
    w = wl.to_torch(wl.weight(rng, H, dtype), dtype).cuda()
    y, s = torch.empty_like(x), torch.empty_like(x)
    rn.rmsnorm_fwd_residual(x, r, w, y, s, None, eps=1e-5)
    xi, ri = x.clone(), r.clone()
    rn.rmsnorm_fwd_residual(xi, ri, w, xi, ri, None, eps=1e-5)
    torch.cuda.synchronize()
    assert xi.dtype == dt and torch.equal(xi, y) and torch.equal(ri, s)
