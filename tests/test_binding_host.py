"""The Python binding's argument marshalling (no GPU): the (M, H, row stride)
it derives from torch tensors, the one-row-stride rule of the ABI, dtype
codes, and the checks that fail before anything reaches the library."""
import pytest

import residual_add_rmsnorm_fwd_gb300 as rn

torch = pytest.importorskip("torch")


def test_rows_of_contiguous_and_padded_views():
    x = torch.zeros(7, 100)
    assert rn._rows(x, "x") == (7, 100, 100)
    padded = torch.zeros(7, 104)[:, :100]          # padded rows: the stride is the allocation's
    assert rn._rows(padded, "x") == (7, 100, 104)
    one = torch.zeros(1, 104)[:, :100]             # a single row: the stride is at least H
    assert rn._rows(one, "x") == (1, 100, 104)


def test_rows_rejects_other_layouts():
    with pytest.raises(ValueError, match="2-D"):
        rn._rows(torch.zeros(2, 3, 4), "x")
    with pytest.raises(ValueError, match="contiguous"):
        rn._rows(torch.zeros(8, 6).t(), "x")       # columns strided: not rows of the ABI


def test_shared_stride_requires_one_shape_and_one_stride():
    buf = torch.zeros(5, 72)
    x, y = buf[:, :64], torch.zeros(5, 72)[:, :64]
    assert rn._shared_stride([(x, "x"), (y, "y")]) == (5, 64, 72)
    with pytest.raises(ValueError, match="shape"):
        rn._shared_stride([(x, "x"), (torch.zeros(5, 63), "y")])
    with pytest.raises(ValueError, match="row stride"):
        rn._shared_stride([(x, "x"), (torch.zeros(5, 64), "y")])


def test_dtype_codes():
    assert rn.dtype_code(torch.float32) == rn.RMSN_F32
    assert rn.dtype_code(torch.float16) == rn.RMSN_F16
    assert rn.dtype_code(torch.bfloat16) == rn.RMSN_BF16
    with pytest.raises(TypeError):
        rn.dtype_code(torch.float64)


def test_adaln_conditioning_rows_are_checked_before_the_call():
    x, y = torch.zeros(10, 32), torch.zeros(10, 32)
    with pytest.raises(ValueError, match="rows"):          # 10 rows at 4 per conditioning row need 3
        rn.rmsnorm_adaln_fwd(x, None, torch.zeros(2, 32), torch.zeros(2, 32), y, rows_per_cond=4)
    with pytest.raises(ValueError, match="columns"):
        rn.rmsnorm_adaln_fwd(x, None, torch.zeros(10, 16), torch.zeros(10, 16), y)
    with pytest.raises(ValueError, match="rows"):
        rn.rmsnorm_adaln_fwd(x, None, torch.zeros(10, 32), torch.zeros(10, 32), y, rows_per_cond=0)


def test_workspace_bytes_of_no_rows_needs_no_device():
    assert rn.rmsnorm_bwd_workspace_bytes(0, 4096, torch.bfloat16) == 0
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_bwd_workspace_bytes(4, 0, torch.bfloat16)   # H = 0 is invalid
    assert e.value.status == 1


def test_status_text_of_every_code():
    for code in range(6):
        assert rn.rmsnorm_status_string(code) and rn.rmsnorm_status_string(code) != "unknown status"
    assert rn.rmsnorm_status_string(99) == "unknown status"
