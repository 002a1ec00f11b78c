"""Pins for the oracle's storage codec (IEEE 754 binary16; bfloat16 = the top
16 bits of binary32), checked against independent implementations: numpy's
float16 conversions, torch's bfloat16 conversions, and a brute-force search
for the nearest representable value."""
import numpy as np
import pytest
import torch

ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _same(a, b):
    """Equal, with NaN == NaN."""
    return np.array_equal(a, b, equal_nan=True)


def test_decode_f16_exhaustive(oracle):
    ref = ALL16.view(np.float16).astype(np.float64)
    assert _same(oracle.decode(ALL16, "f16"), ref)


def test_decode_bf16_exhaustive(oracle):
    ref = torch.from_numpy(ALL16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(oracle.decode(ALL16, "bf16"), ref)


def test_roundtrip_exhaustive(oracle):
    for dt in ("f16", "bf16"):
        v = oracle.decode(ALL16, dt)
        back = oracle.encode(v, dt)
        finite = np.isfinite(v)
        assert np.array_equal(back[finite], ALL16[finite])
        assert np.all(np.isnan(oracle.decode(back[np.isnan(v)], dt)))
        # infinities keep their sign
        inf = np.isinf(v)
        assert np.array_equal(back[inf], ALL16[inf])


def _edge_values(dt):
    if dt == "f16":
        tiny, big, maxv = 2.0 ** -24, 2.0 ** 15, 65504.0
    else:
        tiny, big, maxv = 2.0 ** -133, 2.0 ** 127, float(np.float32(3.3895313892515355e38))
    vals = [0.0, -0.0, tiny, tiny / 2, tiny * 1.5, tiny * 2.5, tiny / 2 * 1.0000001,
            maxv, maxv * (1 + 2 ** -12), maxv * (1 + 2 ** -9), np.inf, -np.inf,
            big, 1.0, 1.0 + 2 ** -11, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -3.0 - 2 ** -10]
    if dt == "f16":
        vals += [65519.99, 65520.0, 2.0 ** -14, 2.0 ** -14 - 2 ** -25, 2.0 ** -14 - 2 ** -26]
    return np.array(vals, np.float64)


def test_encode_f16_vs_numpy(oracle):
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(200000) * np.exp2(rng.integers(-30, 18, 200000)),
        _edge_values("f16"),
        rng.standard_normal(1000).astype(np.float32).astype(np.float64),
    ])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode(v, "f16"), ref)


def test_encode_bf16_vs_torch(oracle):
    """Values exact in binary32 (torch rounds binary32 -> bfloat16 once)."""
    rng = np.random.default_rng(6)
    v32 = np.concatenate([
        (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 120, 200000))).astype(np.float32),
        rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    v32 = v32[np.isfinite(v32)]
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.encode(v32.astype(np.float64), "bf16"), ref)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_encode_nearest_brute_force(oracle, dt):
    """Round to nearest, ties to the even pattern, against a search over all
    finite patterns (binary64 inputs that are not exact in binary32 included)."""
    dec = oracle.decode(ALL16, dt)
    pos = (ALL16 < 0x8000) & np.isfinite(dec)
    vals, pats = dec[pos], ALL16[pos]
    order = np.argsort(vals, kind="stable")
    vals, pats = vals[order], pats[order]
    rng = np.random.default_rng(7)
    top = 16 if dt == "f16" else 128
    mags = np.concatenate([
        np.exp2(rng.uniform(-26 if dt == "f16" else -135, top - 0.01, 50000)),
        (vals[1:] + vals[:-1]) / 2,                        # every exact tie
    ])
    got = oracle.encode(mags, dt)
    idx = np.clip(np.searchsorted(vals, mags), 1, len(vals) - 1)
    lo, hi = vals[idx - 1], vals[idx]
    plo, phi = pats[idx - 1], pats[idx]
    dlo, dhi = mags - lo, hi - mags
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (phi % 2 == 0))
    want = np.where(pick_hi, phi, plo)
    assert np.array_equal(got, want)
    # negative values mirror the positive ones
    assert np.array_equal(oracle.encode(-mags, dt), want | np.uint16(0x8000))


def test_encode_special(oracle):
    for dt, inf_bits in (("f16", 0x7C00), ("bf16", 0x7F80)):
        out = oracle.encode(np.array([np.nan, np.inf, -np.inf, 0.0, -0.0]), dt)
        assert np.isnan(oracle.decode(out[:1], dt))[0]
        assert out[1] == inf_bits and out[2] == (inf_bits | 0x8000)
        assert out[3] == 0 and out[4] == 0x8000
    assert oracle.encode(np.array([65520.0]), "f16")[0] == 0x7C00       # tie above max -> inf
    assert oracle.encode(np.array([65519.0]), "f16")[0] == 0x7BFF       # max finite
    assert oracle.encode(np.array([2.0 ** -25]), "f16")[0] == 0         # tie to even zero
    assert oracle.encode(np.array([3 * 2.0 ** -25]), "f16")[0] == 2     # tie to even 2
