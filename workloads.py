"""Seeded synthetic inputs for RMSNorm, shared by the tests, the smoke check and
the benchmark.  This module holds no RMSNorm arithmetic: it only draws random
numbers and rounds them to a storage format.

Recipe (for every matrix): a ``numpy.random.Generator(PCG64(seed))`` draws
binary32 samples; the samples are rounded to the storage format with
round-to-nearest-even (numpy for fp16, torch for bf16, identity for fp32).
Each config draws its tensors in a fixed order: x, residual, weight, dy.
A weight is ``1 + 0.1 * N(0, 1)`` rounded to the storage format.  Padding
columns of a strided matrix (``stride > H``) hold a NaN sentinel, so a kernel
that reads them poisons its result and one that writes them is caught by the
guard-band checks.

Arrays are numpy arrays in the raw storage format: float32 for f32, uint16
bit patterns for f16 and bf16.  ``to_torch`` views them as torch tensors.

The five workloads mirror the shapes and value distributions of the pages'
LLM and DiT/video use (hidden sizes 2048-8192, the LTX-Video norm mix with
168 norm modules of which 112 have no weight, fp16 activations large enough
that squaring them would overflow binary16).
"""
from __future__ import annotations

import numpy as np

STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
# NaN bit patterns used to fill padding columns and guard regions
SENTINEL = {"f32": np.uint32(0x7FA5A5A5), "f16": np.uint16(0x7E5A), "bf16": np.uint16(0x7FA5)}


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def to_storage(a32: np.ndarray, dtype: str) -> np.ndarray:
    """binary32 samples -> storage array, round to nearest even."""
    a32 = np.asarray(a32, dtype=np.float32)
    if dtype == "f32":
        return a32.copy()
    if dtype == "f16":
        with np.errstate(over="ignore"):
            return a32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(a32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def sentinel_fill(shape, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.full(shape, SENTINEL["f32"], np.uint32).view(np.float32)
    return np.full(shape, SENTINEL[dtype], np.uint16)


def matrix(rng, M: int, H: int, dtype: str, stride: int | None = None,
           row_lognormal: bool = False, outlier_frac: float = 0.0,
           outlier_range=(200.0, 300.0)) -> np.ndarray:
    """An (M, stride) storage array whose first H columns hold the samples.

    Samples are N(0, 1).  ``row_lognormal``: every row is multiplied by
    exp(N(0, 1)) (one LogNormal(0, 1) factor per row, drawn after the
    normals).  ``outlier_frac``: that fraction of entries (Bernoulli mask) is
    replaced by a random sign times U(outlier_range) (mask, then magnitudes,
    then signs).
    """
    stride = H if stride is None else stride
    a = rng.standard_normal((M, H), dtype=np.float32)
    if row_lognormal:
        a *= np.exp(rng.standard_normal((M, 1), dtype=np.float32))
    if outlier_frac > 0:
        mask = rng.random((M, H), dtype=np.float32) < outlier_frac
        k = int(mask.sum())
        mags = rng.uniform(outlier_range[0], outlier_range[1], k).astype(np.float32)
        signs = np.where(rng.random(k) < 0.5, -1.0, 1.0).astype(np.float32)
        a[mask] = mags * signs
    body = to_storage(a, dtype)
    if stride == H:
        return body
    out = sentinel_fill((M, stride), dtype)
    out.view(body.dtype)[:, :H] = body
    return out.view(STORAGE[dtype])


def conditioning(rng, n: int, H: int, dtype: str, stride: int | None = None, sigma: float = 0.5) -> np.ndarray:
    """An (n, stride) storage array of AdaLN conditioning rows (scale or
    shift): sigma * N(0, 1) in the first H columns, sentinels in the padding.
    (In a DiT block these come out of the timestep-embedding MLP; zero-mean
    values of moderate size stand in for them.)"""
    stride = H if stride is None else stride
    body = to_storage(sigma * rng.standard_normal((n, H), dtype=np.float32), dtype)
    if stride == H:
        return body
    out = sentinel_fill((n, stride), dtype)
    out.view(body.dtype)[:, :H] = body
    return out.view(STORAGE[dtype])


def weight(rng, H: int, dtype: str) -> np.ndarray:
    """1 + 0.1 * N(0, 1), rounded to the storage format."""
    return to_storage(1.0 + 0.1 * rng.standard_normal(H, dtype=np.float32), dtype)


def to_torch(a: np.ndarray, dtype: str):
    """Storage array -> CPU torch tensor of the storage dtype (shares memory)."""
    import torch
    a = np.ascontiguousarray(a)
    if dtype == "f32":
        return torch.from_numpy(a.view(np.float32))
    return torch.from_numpy(a.view(np.int16)).view(torch_dtype(dtype))


def from_torch(t, dtype: str) -> np.ndarray:
    """CPU or CUDA torch tensor of the storage dtype -> numpy storage array."""
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

CONFIGS = {
    1: dict(name="fwd_f32_64x1024", dtype="f32", M=64, H=1024, stride=1024, eps=1e-6,
            seed=0, residual=False, weight=True, backward=False, save_rrms=False),
    2: dict(name="fused_fwd_bf16_16384x4096", dtype="bf16", M=16384, H=4096, stride=4096,
            eps=1e-5, seed=1, residual=True, weight=True, backward=False, save_rrms=False),
    3: dict(name="dit_mix_bf16", dtype="bf16", M=12288, H=2048, stride=2048, eps=1e-6,
            seed=2, residual=False, weight=True, backward=False, save_rrms=False,
            calls_weighted=56, calls_unweighted=112, head_M=393216, head_H=64, buffer_sets=4),
    4: dict(name="fwd_bwd_bf16_16384x8192", dtype="bf16", M=16384, H=8192, stride=8192,
            eps=1e-5, seed=3, residual=False, weight=True, backward=True, save_rrms=True),
    5: dict(name="fused_fwd_bwd_f16_32768x6144_stride6272", dtype="f16", M=32768, H=6144,
            stride=6272, eps=1e-5, seed=4, residual=True, weight=True, backward=True,
            save_rrms=True, outlier_frac=0.01),
    # rows longer than one CTA holds (64 KB): the split-row (cluster) kernels;
    # a measurement case beside the five configurations above
    6: dict(name="fused_fwd_bwd_bf16_4096x32768", dtype="bf16", M=4096, H=32768, stride=32768, eps=1e-5,
            seed=5, residual=True, weight=True, backward=True, save_rrms=True),
    # rows that are not 16-byte aligned: an odd hidden size, rows contiguous,
    # so a row starts at each of the 8 element offsets within 16 bytes in turn
    # (the aligned-frame kernels); a measurement case beside the five above
    7: dict(name="fused_fwd_bwd_bf16_16384x4095", dtype="bf16", M=16384, H=4095, stride=4095, eps=1e-5,
            seed=6, residual=True, weight=True, backward=True, save_rrms=True),
}


def generate(cfg_id: int, with_dy: bool | None = None, M: int | None = None) -> dict:
    """Inputs of workload ``cfg_id`` as storage arrays.

    Keys: x, residual (if fused), w, dy (if backward, or ``with_dy``).  For
    the DiT mix: xs (list of buffer sets), w, head_x, head_w.  ``M`` overrides
    the row count (a smaller sample of the same distribution and seed).
    """
    c = CONFIGS[cfg_id]
    rng = rng_for(c["seed"])
    dt, H, stride = c["dtype"], c["H"], c["stride"]
    rows = c["M"] if M is None else M
    out = {}
    if cfg_id == 3:
        out["xs"] = [matrix(rng, rows, H, dt, stride, row_lognormal=True)
                     for _ in range(c["buffer_sets"])]
        out["w"] = weight(rng, H, dt)
        head_rows = c["head_M"] if M is None else M
        out["head_x"] = matrix(rng, head_rows, c["head_H"], dt, row_lognormal=True)
        out["head_w"] = weight(rng, c["head_H"], dt)
        return out
    out["x"] = matrix(rng, rows, H, dt, stride, outlier_frac=c.get("outlier_frac", 0.0))
    if c["residual"]:
        out["residual"] = matrix(rng, rows, H, dt, stride)
    out["w"] = weight(rng, H, dt)
    if c["backward"] if with_dy is None else with_dy:
        out["dy"] = matrix(rng, rows, H, dt, stride)
    return out
