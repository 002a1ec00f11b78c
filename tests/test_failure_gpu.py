"""Failure detection on the GPU without a fault: the kernels' bounded
pipeline waits.  Every wait on a bulk-copy barrier is bounded; a wait that
runs out sets RMSN_DEVERR_PIPELINE_TIMEOUT in the library's device error
word, the kernel finishes with no copy left in flight, and
rmsnorm_read_device_errors() reports the flag and clears it.

The waits are made to run out on purpose with the library's diagnostic
setting (rmsnorm_debug_pipeline_timeout): a short poll limit, and each ring
CTA's issuing thread waiting for its first row before it has issued any
copy.  Nothing faults, traps or hangs: the issuing thread still confirms
every copy it issued before it re-arms a stage or exits.  After the setting
is cleared, the same calls give the oracle's results again and the error
word stays clear."""
import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl
from helpers import bwd_rtol, check_dx, check_fwd_values

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TIMEOUT = 1   # RMSN_DEVERR_PIPELINE_TIMEOUT


@pytest.fixture
def timeout_test_mode():
    def enable(polls, hold):
        rn.rmsnorm_debug_pipeline_timeout(polls, hold)
    yield enable
    rn.rmsnorm_debug_pipeline_timeout(0, False)
    torch.cuda.synchronize()
    rn.rmsnorm_read_device_errors()   # flags a test left set are its own


def _inputs(M, H, dtype="bf16", seed=0):
    rng = wl.rng_for(seed)
    x, r, w, dy = (wl.matrix(rng, M, H, dtype), wl.matrix(rng, M, H, dtype), wl.weight(rng, H, dtype),
                   wl.matrix(rng, M, H, dtype))
    return (x, r, w, dy), tuple(wl.to_torch(a, dtype).cuda() for a in (x, r, w, dy))


def _fused(tx, tr, tw):
    y, s = torch.empty_like(tx), torch.empty_like(tx)
    rr = torch.empty(tx.shape[0], device="cuda")
    rn.rmsnorm_fwd_residual(tx, tr, tw, y, s, rr, eps=1e-5)
    return y, s, rr


def _bwd(tdy, s, tw, rr):
    M, H = s.shape
    dx, dw = torch.empty_like(s), torch.empty(H, device="cuda")
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, s.dtype), dtype=torch.uint8, device="cuda")
    rn.rmsnorm_bwd(tdy, s, tw, rr, dx, dw, ws)
    return dx, dw


@pytest.mark.parametrize("M", [1, 613])
def test_held_first_copy_sets_the_flag_then_clears(oracle, timeout_test_mode, M):
    """Fused forward (8 KB bf16 rows: the ring kernel) and backward (the
    backward ring) with every CTA's first wait running out: the call
    returns, the flag is set, one read clears it; then normal calls match
    the oracle with the flag clear."""
    (x, r, w, dy), (tx, tr, tw, tdy) = _inputs(M, 4096, seed=M)
    timeout_test_mode(256, True)
    y, s, rr = _fused(tx, tr, tw)
    _bwd(tdy, s, tw, rr)
    torch.cuda.synchronize()
    assert rn.rmsnorm_read_device_errors() & TIMEOUT
    assert rn.rmsnorm_read_device_errors() == 0, "reading the error word clears it"

    rn.rmsnorm_debug_pipeline_timeout(0, False)
    y, s, rr = _fused(tx, tr, tw)
    dx, dw = _bwd(tdy, s, tw, rr)
    torch.cuda.synchronize()
    assert rn.rmsnorm_read_device_errors() == 0
    ref = oracle.rmsnorm_fwd(x, w, 1e-5, "bf16", residual=r)
    assert check_fwd_values(wl.from_torch(y, "bf16"), ref["y"], "bf16", oracle)["failed"] == 0
    s_np = wl.from_torch(s, "bf16")
    assert np.array_equal(s_np, oracle.encode(ref["s"], "bf16"))
    refb = oracle.rmsnorm_bwd(dy, s_np, w, 1e-5, "bf16")
    got = oracle.decode(wl.from_torch(dx, "bf16"), "bf16")
    assert check_dx(got, refb["dx"], refb["dx_scale"], bwd_rtol("bf16"))["failed"] == 0


def test_plain_ring_forward_flag(timeout_test_mode):
    """The one-input ring forward (4 KB bf16 rows) reports its held wait too."""
    _, (tx, _, tw, _) = _inputs(4099, 2048, seed=3)
    timeout_test_mode(64, True)
    rn.rmsnorm_fwd(tx, tw, torch.empty_like(tx), None, eps=1e-6)
    torch.cuda.synchronize()
    assert rn.rmsnorm_read_device_errors() & TIMEOUT
    assert rn.rmsnorm_read_device_errors() == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("H", [4096, 32768])
def test_one_poll_limit_finishes(oracle, timeout_test_mode, dtype, H):
    """A one-poll limit with nothing held.  The f16 kernels take their wait
    limit from the call: their threads whose waits run out carry on with the
    shortened limit while each CTA's issuing thread (and, on the split-row
    kernels, the thread that arms the cluster exchange) waits for every copy
    and partial sum it armed.  The bf16 kernels poll against the full limit
    until a wait has run out, so the setting leaves them as they are.  Either
    way the calls finish, whether or not a wait ran out this time, and normal
    calls afterwards match the oracle."""
    M = 2049 if H == 4096 else 129
    (x, r, w, dy), (tx, tr, tw, tdy) = _inputs(M, H, dtype, seed=H)
    timeout_test_mode(1, False)
    for _ in range(3):
        y, s, rr = _fused(tx, tr, tw)
        _bwd(tdy, s, tw, rr)
    torch.cuda.synchronize()
    rn.rmsnorm_read_device_errors()

    rn.rmsnorm_debug_pipeline_timeout(0, False)
    y, s, rr = _fused(tx, tr, tw)
    torch.cuda.synchronize()
    assert rn.rmsnorm_read_device_errors() == 0
    ref = oracle.rmsnorm_fwd(x, w, 1e-5, dtype, residual=r)
    assert check_fwd_values(wl.from_torch(y, dtype), ref["y"], dtype, oracle)["failed"] == 0


def test_debug_setting_validation():
    with pytest.raises(rn.RmsnormError):
        rn.rmsnorm_debug_pipeline_timeout((1 << 22) + 1, False)
    with pytest.raises(rn.RmsnormError):
        rn.rmsnorm_debug_pipeline_timeout(0, True)
    rn.rmsnorm_debug_pipeline_timeout(0, False)
