"""rmsnorm_bwd_noalloc: the backward for callers that cannot allocate device
memory (engines that reserve all memory up front, plugin interfaces that
only pass inputs and outputs, hot paths where cudaMalloc is not allowed).
It must give the same dx and dweight as rmsnorm_bwd with a caller-allocated
workspace, on consecutive calls that share its fixed scratch array.  This
file is collected last so a failure here leaves every other test run."""
import ctypes

import numpy as np
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn
import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(dtype, M, H, seed):
    rng = wl.rng_for(seed)
    dt = wl.torch_dtype(dtype)
    x = wl.to_torch(wl.matrix(rng, M, H, dtype), dtype).cuda()
    w = wl.to_torch(wl.weight(rng, H, dtype), dtype).cuda()
    dy = wl.to_torch(wl.matrix(rng, M, H, dtype), dtype).cuda()
    rrms = torch.empty(M, device="cuda")
    rn.rmsnorm_fwd(x, w, torch.empty_like(x), rrms, eps=1e-5)
    return x, w, dy, rrms, dt


def _noalloc_raw(dy, x, w, rrms, dx, dw, dtype_code):
    """Call the entry point through the C ABI with raw pointers."""
    M, H = x.shape
    return rn.lib().rmsnorm_bwd_noalloc(
        dy.data_ptr(), x.data_ptr(), w.data_ptr(), rrms.data_ptr(), dx.data_ptr(), dw.data_ptr(),
        H, M, H, dtype_code, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,M,H", [("bf16", 4099, 4096), ("f16", 2051, 6144), ("f32", 1025, 1000),
                                       ("bf16", 3001, 64), ("bf16", 301, 32768)])
def test_noalloc_matches_workspace_backward_on_consecutive_calls(dtype, M, H):
    x, w, dy, rrms, dt = _inputs(dtype, M, H, seed=M)
    ref_dx, ref_dw = torch.empty_like(x), torch.empty(H, device="cuda")
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, H, dt), dtype=torch.uint8, device="cuda")
    rn.rmsnorm_bwd(dy, x, w, rrms, ref_dx, ref_dw, ws)
    for call in range(2):    # the second call reuses the scratch the first one left behind
        dx, dw = torch.full_like(x, float("nan")), torch.full((H,), float("nan"), device="cuda")
        status = _noalloc_raw(dy, x, w, rrms, dx, dw, rn.dtype_code(dt))
        assert status == 0, rn.rmsnorm_status_string(status)
        torch.cuda.synchronize()
        # same kernels, same fixed reduction order: identical bits (stricter
        # than the backward tolerance used elsewhere)
        assert torch.equal(dx, ref_dx), f"dx differs on call {call}"
        assert torch.equal(dw, ref_dw), f"dweight differs on call {call}"


def test_noalloc_rejects_oversized_partials():
    # 131080 bf16 columns (rows above 256 KB take the chunked kernel, one
    # partial row per CTA): 64 partial rows exceed the 16 MiB array
    M, H = 64, (1 << 17) + 8
    x = torch.zeros(M, H, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    rrms = torch.ones(M, device="cuda")
    assert rn.rmsnorm_bwd_workspace_bytes(M, H, torch.bfloat16) > 16 << 20
    dx, dw = torch.empty_like(x), torch.empty(H, device="cuda")
    status = _noalloc_raw(x, x.clone(), w, rrms, dx, dw, rn.RMSN_BF16)
    assert status == 3   # RMSN_ERR_WORKSPACE, before any launch


@pytest.mark.parametrize("has_weight,want_dw", [(0, True), (1, False)])
def test_noalloc_without_dweight(has_weight, want_dw):
    """No weight, or no dweight wanted: the call needs no scratch (it is not
    looked up) and gives rmsnorm_bwd's dx, bit for bit."""
    M, H = 1031, 4096
    x, w, dy, rrms, dt = _inputs("bf16", M, H, seed=7)
    ref_dx = torch.empty_like(x)
    rn.rmsnorm_bwd(dy, x, w if has_weight else None, rrms, ref_dx, None, None)
    dx = torch.full_like(x, float("nan"))
    dw = torch.full((H,), 7.0, device="cuda")
    status = rn.lib().rmsnorm_bwd_noalloc(
        dy.data_ptr(), x.data_ptr(), w.data_ptr() if has_weight else None, rrms.data_ptr(), dx.data_ptr(),
        dw.data_ptr() if want_dw else None, H, M, H, rn.dtype_code(dt), has_weight,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0, rn.rmsnorm_status_string(status)
    torch.cuda.synchronize()
    assert torch.equal(dx, ref_dx)
    assert bool((dw == 7.0).all()), "dweight is not written when there is no weight or none is asked for"


def test_noalloc_zero_rows_zeroes_dweight():
    """M = 0: dweight is the empty sum (zeros); nothing else is touched."""
    H = 4096
    w = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    dw = torch.full((H,), 7.0, device="cuda")
    status = rn.lib().rmsnorm_bwd_noalloc(None, None, w.data_ptr(), None, None, dw.data_ptr(), H, 0, H,
                                          rn.RMSN_BF16, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0, rn.rmsnorm_status_string(status)
    torch.cuda.synchronize()
    assert bool((dw == 0).all())
