"""The GPU parity tests' tolerance checks, on the host: each accepts what its
stated bound allows and rejects one step beyond it, NaN and infinity, so a
kernel that is off by two ulp or writes NaN cannot pass a parity test."""
import numpy as np
import pytest

from helpers import bwd_rtol, check_dweight, check_dx, check_fwd_values, check_scaled_values, ordinal


def test_ordinal_orders_bit_patterns_like_values():
    bits = np.array([0x8002, 0x8001, 0x8000, 0x0000, 0x0001, 0x0002, 0x3F80, 0x3F81], np.uint16)
    o = ordinal(bits)
    assert list(o) == [-2, -1, 0, 0, 1, 2, 0x3F80, 0x3F81]   # +0 and -0 coincide


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_forward_check_allows_one_ulp_and_no_more(oracle, dtype):
    ref = np.array([[1.0, -2.5, 3.25e-3, 100.0]])
    want = oracle.encode(ref, dtype)
    assert check_fwd_values(want, ref, dtype, oracle)["failed"] == 0
    up1 = (want.astype(np.int64) + 1).astype(np.uint16)          # one ulp away from zero
    assert check_fwd_values(up1, ref, dtype, oracle)["failed"] == 0
    up2 = (want.astype(np.int64) + 2).astype(np.uint16)
    assert check_fwd_values(up2, ref, dtype, oracle)["failed"] == 4
    nan = want.copy()
    nan[0, 0] = 0x7E00 if dtype == "f16" else 0x7FC0
    assert check_fwd_values(nan, ref, dtype, oracle)["failed"] == 1


def test_forward_check_fp32_relative_bound(oracle):
    ref = np.array([[1.0, -3.0, 1e-3]])
    ok = (ref * (1 + 0.9e-5)).astype(np.float32)
    assert check_fwd_values(ok, ref, "f32", oracle)["failed"] == 0
    bad = (ref * (1 + 3e-5)).astype(np.float32)
    assert check_fwd_values(bad, ref, "f32", oracle)["failed"] == 3
    assert check_fwd_values(np.array([[np.nan, -3.0, 1e-3]], np.float32), ref, "f32", oracle)["failed"] == 1


def test_dx_check_scales_with_the_row_and_the_terms():
    ref = np.array([[1.0, -1.0, 0.0, 0.0]])                   # row rms 1/sqrt(2)
    scale = np.array([[1.0, 1.0, 0.0, 8.0]])
    rtol = bwd_rtol("bf16")
    got = ref + np.array([[0.019, -0.019, 0.014, 0.15]])     # inside: |ref|, row rms, dx_scale
    assert check_dx(got, ref, scale, rtol)["failed"] == 0
    got = ref + np.array([[0.021, 0.0, 0.015, 0.17]])        # each beyond its bound
    assert check_dx(got, ref, scale, rtol)["failed"] == 3
    assert check_dx(np.array([[np.inf, -1.0, 0.0, 0.0]]), ref, scale, rtol)["failed"] == 1


def test_dweight_check_is_relative_to_the_absolute_sum():
    ref, ref_abs = np.array([0.0, 10.0]), np.array([100.0, 10.0])
    assert check_dweight(np.array([1.9, 10.19]), ref, ref_abs, 2e-2)["failed"] == 0
    assert check_dweight(np.array([2.1, 10.21]), ref, ref_abs, 2e-2)["failed"] == 2
    assert check_dweight(np.array([np.nan, 10.0]), ref, ref_abs, 2e-2)["failed"] == 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scaled_check_for_cancelling_sums(oracle, dtype):
    # y = t + shift cancels to 1e-3 while its terms are of size 2: the bound is 1e-5 * 2
    ref = np.array([[1e-3, 0.5]])
    y_scale = np.array([[2.0, 0.5]])
    within = oracle.encode(ref + np.array([[1.5e-5, 0.0]]), dtype)
    assert check_scaled_values(within, ref, y_scale, dtype, oracle)["failed"] == 0
    beyond = oracle.encode(ref + np.array([[1e-3, 0.0]]), dtype)
    assert check_scaled_values(beyond, ref, y_scale, dtype, oracle)["failed"] == 1
    nan = oracle.encode(np.array([[np.nan, 0.5]]), dtype)
    assert check_scaled_values(nan, ref, y_scale, dtype, oracle)["failed"] == 1
