"""Test-side plumbing: guarded device buffers, tolerance checks, oracle calls."""
from __future__ import annotations

import numpy as np

import workloads as wl

GUARD = 64  # sentinel elements before and after every device buffer


def ordinal(bits: np.ndarray) -> np.ndarray:
    """f16/bf16 bit patterns -> integers ordered like the values they encode
    (adjacent representable values differ by 1; +0 and -0 both map to 0)."""
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


class Guarded:
    """A device matrix (M, H) with row stride `stride`, inside a flat buffer
    whose padding columns and head/tail guard regions hold a NaN sentinel."""

    def __init__(self, M, H, stride, dtype, offset_elems=0, device="cuda"):
        import torch
        self.M, self.H, self.stride, self.dtype = M, H, stride, dtype
        self.offset = GUARD + offset_elems
        n = self.offset + M * stride + GUARD
        host = wl.sentinel_fill((n,), dtype)
        self.flat = wl.to_torch(host, dtype).to(device)
        self.initial = self.flat.clone()
        body = self.flat[self.offset:self.offset + M * stride]
        self.full = body.view(M, stride) if M > 0 else body.view(0, stride)
        self.t = self.full[:, :H]
        self._torch = torch

    def upload(self, storage: np.ndarray):
        """Write an (M, >=H) storage array into the first H columns."""
        src = wl.to_torch(np.ascontiguousarray(storage[:, :self.H]), self.dtype).to(self.t.device)
        self.t.copy_(src)
        self.initial = self.flat.clone()
        return self

    def host(self) -> np.ndarray:
        return wl.from_torch(self.t, self.dtype)

    def untouched_outside(self) -> bool:
        """Guard regions and padding columns still hold what they held."""
        torch = self._torch
        a = self.flat.view(torch.int32 if self.dtype == "f32" else torch.int16)
        b = self.initial.view(torch.int32 if self.dtype == "f32" else torch.int16)
        mask = torch.ones_like(a, dtype=torch.bool)
        body = mask[self.offset:self.offset + self.M * self.stride].view(self.M, self.stride) \
            if self.M > 0 else None
        if body is not None:
            body[:, :self.H] = False
        return bool(torch.equal(a[mask], b[mask]))


def device_vec(storage: np.ndarray, dtype: str, offset_elems=0):
    """1-D device tensor (weight), optionally at a misaligned offset."""
    t = wl.to_torch(np.concatenate([np.zeros(offset_elems, storage.dtype), storage]) if offset_elems
                    else storage, dtype).cuda()
    return t[offset_elems:]


def f32_buffer(n, offset=0):
    import torch
    return torch.full((n + offset + 2 * GUARD,), float("nan"), device="cuda")[GUARD + offset:GUARD + offset + n]


def check_fwd_values(got_bits: np.ndarray, ref64: np.ndarray, dtype: str, oracle) -> dict:
    """Forward tolerance: fp32 within 1e-5 relative per element; f16/bf16
    within 1 ulp of the oracle's value rounded to the storage type."""
    if dtype == "f32":
        err = np.abs(got_bits.astype(np.float64) - ref64)
        bad = ~(err <= 1e-5 * np.abs(ref64))
    else:
        want = oracle.encode(ref64, dtype)
        d = np.abs(ordinal(got_bits) - ordinal(want))
        bad = ~(d <= 1)
        err = d
    return {"failed": int(bad.sum()), "max_err": float(err.max()) if err.size else 0.0, "bad": bad}


def check_dx(got: np.ndarray, ref: np.ndarray, scale: np.ndarray, rtol: float) -> dict:
    """Backward dx tolerance per element:
    |got - ref| <= rtol * max(|ref|, rms of the ref row, dx_scale), where
    dx_scale is the oracle's size of the two terms whose difference is dx
    (rounding error of any binary32 evaluation is proportional to it)."""
    row_rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    denom = np.maximum(np.maximum(np.abs(ref), row_rms), scale)
    err = np.abs(got - ref)
    bad = ~(err <= rtol * denom)
    return {"failed": int(bad.sum()), "max_rel": float((err / np.where(denom > 0, denom, 1)).max())
            if err.size else 0.0}


def check_dweight(got: np.ndarray, ref: np.ndarray, ref_abs: np.ndarray, rtol: float) -> dict:
    """Per column: |got - ref| <= rtol * sum_i |dy_ih * xhat_ih| (the sum's condition scale)."""
    err = np.abs(got.astype(np.float64) - ref)
    bad = ~(err <= rtol * ref_abs)
    return {"failed": int(bad.sum()), "max_rel": float((err / np.where(ref_abs > 0, ref_abs, 1)).max())}


def bwd_rtol(dtype: str) -> float:
    return 1e-5 if dtype == "f32" else 2e-2


def check_scaled_values(got_bits: np.ndarray, ref64: np.ndarray, y_scale: np.ndarray, dtype: str, oracle) -> dict:
    """Tolerance per element for outputs formed by sums that can cancel
    (AdaLN's + shift; LayerNorm's - mean and + bias): the binary32 evaluation
    error is relative to y_scale, the oracle's size of the terms y is formed
    from, not to |y|: fp32 within 1e-5 * y_scale; f16/bf16 within 1 ulp of the
    oracle's value rounded to the storage type, or within 1e-5 * y_scale."""
    got = oracle.decode(got_bits, dtype)
    err = np.abs(got - ref64)
    ok = err <= 1e-5 * y_scale
    if dtype != "f32":
        want = oracle.encode(ref64, dtype)
        ok |= np.abs(ordinal(got_bits) - ordinal(want)) <= 1
    bad = ~ok
    rel = err / np.where(y_scale > 0, y_scale, 1)
    return {"failed": int(bad.sum()), "max_rel": float(rel.max()) if rel.size else 0.0, "bad": bad}
