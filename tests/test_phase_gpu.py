"""GPU parity of the kernels for rows that are not 16-byte aligned but whose
matrices share one alignment phase (odd hidden sizes, strides that are not a
multiple of 16 bytes, views starting between 16-byte boundaries): 128-bit
accesses in each row's own aligned frame, the first and last frame vectors
masked, the weight (bias, conditioning rows) cut out of its own aligned
vectors by the row's shift, and -- in the backward -- the dweight terms moved
back to a fixed column frame by warp shuffles.

Every case is checked against the fp64 oracle with the tolerances of the
aligned paths (tests/test_parity_gpu.py, test_layernorm_gpu.py,
test_adaln_gpu.py), with guard bands around every buffer, so a masked
element written or a shifted weight off by one column fails.

Layouts: contiguous odd H (the phase changes from row to row and cycles
through every value), a padded odd stride, an aligned stride with the base
offset (one phase for all rows), each storage type; the weight at its own
phase (different from the rows'); the longest rows the frame kernels take
(2048 frame vectors); and, as a control, outputs at a phase different from
the inputs' (the scalar path).
"""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import Guarded, check_fwd_values, device_vec, f32_buffer
from test_adaln_gpu import assert_ok as adaln_ok
from test_adaln_gpu import run_adaln
from test_layernorm_gpu import assert_ok as ln_ok
from test_layernorm_gpu import run_ln
from test_parity_gpu import (assert_bwd_ok, assert_fwd_ok, check_in_place, run_bwd, run_bwd_residual,
                             run_fwd)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

V = {"f32": 4, "f16": 8, "bf16": 8}

# (H, stride, offset, w_offset): contiguous odd H (the phase moves every row),
# padded odd strides, aligned strides with a misaligned base, and the weight
# at a phase of its own
LAYOUTS = {
    "bf16": [(257, 257, 0, 0), (1001, 1001, 0, 0), (2047, 2047, 3, 0), (4095, 4095, 0, 5), (4096, 4096, 1, 1),
             (4096, 4096, 7, 2), (3000, 3003, 5, 0), (6143, 6143, 0, 0), (8191, 8195, 1, 6), (16377, 16377, 0, 0)],
    "f16": [(257, 257, 0, 0), (1999, 1999, 0, 3), (4096, 4096, 3, 3), (6143, 6149, 2, 0), (16377, 16379, 7, 1)],
    "f32": [(257, 257, 0, 0), (1023, 1023, 1, 0), (2048, 2048, 1, 3), (4095, 4101, 2, 2), (8189, 8189, 3, 1)],
}
CASES = [(dt, *lay) for dt, lays in LAYOUTS.items() for lay in lays]


def rows_for(H, cap=300_000):
    return int(max(5, min(203, cap // H))) | 1


@pytest.mark.parametrize("dtype,H,stride,offset,w_offset", CASES)
@pytest.mark.parametrize("residual", [False, True])
def test_phase_forward(oracle, dtype, H, stride, offset, w_offset, residual):
    for weight in (True, False):
        res = run_fwd(oracle, dtype, rows_for(H), H, stride=stride, residual=residual, weight=weight,
                      offset=offset, w_offset=w_offset, seed=H + stride + offset + 2 * residual)
        assert_fwd_ok(res)


@pytest.mark.parametrize("dtype,H,stride,offset,w_offset", CASES)
def test_phase_backward(oracle, dtype, H, stride, offset, w_offset):
    assert_bwd_ok(run_bwd(oracle, dtype, rows_for(H), H, stride=stride, offset=offset, w_offset=w_offset,
                          seed=H + offset))
    assert_bwd_ok(run_bwd_residual(oracle, dtype, rows_for(H), H, stride=stride, offset=offset,
                                   w_offset=w_offset, seed=H + offset + 1))


@pytest.mark.parametrize("dtype,H,stride,offset,w_offset", [c for c in CASES if c[1] in (1001, 1999, 4096, 4095)])
def test_phase_backward_without_weight(oracle, dtype, H, stride, offset, w_offset):
    assert_bwd_ok(run_bwd(oracle, dtype, rows_for(H), H, stride=stride, offset=offset, weight=False, seed=H))


@pytest.mark.parametrize("dtype,H,M", [("bf16", 4095, 9001), ("f16", 2047, 12001), ("f32", 1023, 20001)])
def test_phase_grid_stride(oracle, dtype, H, M):
    """More rows than the persistent grid: CTAs stride over rows of every
    phase, the weight windows reloaded as the phase changes, and the
    backward's per-CTA dweight columns summed over many rows."""
    assert_fwd_ok(run_fwd(oracle, dtype, M, H, residual=True, seed=M))
    assert_bwd_ok(run_bwd(oracle, dtype, M, H, seed=M + 1))


@pytest.mark.parametrize("dtype,H,stride,offset,w_offset", [c for c in CASES if c[1] in (257, 2047, 4096, 4095, 1023)])
@pytest.mark.parametrize("residual", [False, True])
def test_phase_layernorm(oracle, dtype, H, stride, offset, w_offset, residual):
    ln_ok(run_ln(oracle, dtype, rows_for(H, 150_000), H, residual=residual, stride=stride, offset=offset,
                 w_offset=w_offset, seed=H + offset))
    ln_ok(run_ln(oracle, dtype, rows_for(H, 150_000), H, residual=residual, stride=stride, offset=offset,
                 w_offset=w_offset, seed=H + offset + 1, shift=24.0))


@pytest.mark.parametrize("dtype,H,stride,cond_stride,offset,cond_offset", [
    ("bf16", 4095, 4095, 4095, 0, 0), ("bf16", 4096, 4096, 4096, 3, 5), ("f16", 2047, 2049, 2051, 1, 0),
    ("f32", 1023, 1023, 1025, 2, 1), ("bf16", 8191, 8191, 8193, 0, 3)])
def test_phase_adaln(oracle, dtype, H, stride, cond_stride, offset, cond_offset):
    for rpc in (1, 4, 1000):
        adaln_ok(run_adaln(oracle, dtype, rows_for(H, 150_000), H, rows_per_cond=rpc, stride=stride,
                           cond_stride=cond_stride, offset=offset, cond_offset=cond_offset, seed=H + rpc))


@pytest.mark.parametrize("dtype,H,offset", [("bf16", 4095, 0), ("bf16", 4096, 3), ("f16", 1001, 0),
                                            ("f32", 2047, 1)])
def test_phase_in_place(oracle, dtype, H, offset):
    """y over x, residual_out over the residual, dx over dy / x / dresidual_out:
    the masked first and last vectors read and write only their own columns."""
    check_in_place(oracle, dtype, rows_for(H), H, offset)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_outputs_at_another_phase(oracle, dtype):
    """y at a different alignment phase from x: no frame is shared, so the
    call takes the scalar path, which must still match the oracle."""
    M, H = 37, 3001
    rng = wl.rng_for(5)
    x, w = wl.matrix(rng, M, H, dtype), wl.weight(rng, H, dtype)
    gx = Guarded(M, H, H, dtype, 1).upload(x)
    gy = Guarded(M, H, H, dtype, 2)
    rrms = f32_buffer(M)
    rn.rmsnorm_fwd(gx.t, device_vec(w, dtype), gy.t, rrms, eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_fwd(x, w, 1e-5, dtype)
    assert check_fwd_values(gy.host(), ref["y"], dtype, oracle)["failed"] == 0
    assert gy.untouched_outside() and gx.untouched_outside()
    got = rrms.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref["rrms"]) <= 1e-5 * ref["rrms"])


@pytest.mark.parametrize("dtype,H,offset", [("bf16", 4095, 0), ("f16", 2047, 5), ("f32", 1023, 1)])
def test_phase_dweight_deterministic(oracle, dtype, H, offset):
    """The column-frame dweight partials and their reduction give the same
    bits on every call."""
    out1 = run_bwd(oracle, dtype, 4001, H, offset=offset, seed=3)
    assert_bwd_ok(out1)
    first = out1["dw_t"].clone()
    out2 = run_bwd(oracle, dtype, 4001, H, offset=offset, seed=3)
    assert torch.equal(first, out2["dw_t"])
