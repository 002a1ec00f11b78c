"""The seeded input generators (no GPU): reproducibility, the distributions
the workload recipe states, storage rounding, and the sentinels in padding
columns.  Statistical bounds are several standard errors wide, so they hold
for these fixed seeds and would catch a wrong scale, offset or fraction."""
import numpy as np
import pytest

import workloads as wl


def decode(a, dtype):
    """Storage array -> float64, for the checks here (numpy for f16, bit
    shift for bf16, which is the upper half of a binary32)."""
    with np.errstate(invalid="ignore"):   # the NaN sentinels widen quietly
        if dtype == "f32":
            return np.asarray(a, np.float32).astype(np.float64)
        if dtype == "f16":
            return a.view(np.float16).astype(np.float64)
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_same_seed_same_bits_other_seed_other_bits(dtype):
    a = wl.matrix(wl.rng_for(7), 33, 257, dtype)
    b = wl.matrix(wl.rng_for(7), 33, 257, dtype)
    c = wl.matrix(wl.rng_for(8), 33, 257, dtype)
    assert a.tobytes() == b.tobytes()
    assert a.tobytes() != c.tobytes()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_matrix_is_standard_normal_rounded_to_storage(dtype):
    x = decode(wl.matrix(wl.rng_for(1), 256, 1024, dtype), dtype)
    n = x.size
    assert abs(x.mean()) < 5 / np.sqrt(n)
    assert abs(x.std() - 1.0) < 0.01
    assert abs(np.mean(np.abs(x) > 1.96) - 0.05) < 0.005   # two-sided 5% tail
    # the storage values are the binary32 draws rounded once (not, say, truncated)
    raw = wl.rng_for(1).standard_normal((256, 1024), dtype=np.float32)
    want = wl.to_storage(raw, dtype)
    assert np.array_equal(wl.matrix(wl.rng_for(1), 256, 1024, dtype), want)


def test_bf16_rounding_is_to_nearest_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even (1)
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to even (1 + 2^-6)
    v = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, 1 + 2.0**-8 + 2.0**-20], np.float32)
    got = decode(wl.to_storage(v, "bf16"), "bf16")
    assert list(got) == [1.0, 1 + 2.0**-6, 1 + 2.0**-7]


def test_weight_is_one_plus_a_tenth_normal():
    w = decode(wl.weight(wl.rng_for(2), 65536, "f32"), "f32")
    assert abs(w.mean() - 1.0) < 5 * 0.1 / np.sqrt(w.size)
    assert abs(w.std() - 0.1) < 0.002


def test_conditioning_scale():
    c = decode(wl.conditioning(wl.rng_for(3), 64, 1024, "f32", sigma=0.5), "f32")
    assert abs(c.mean()) < 5 * 0.5 / np.sqrt(c.size)
    assert abs(c.std() - 0.5) < 0.01


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_padding_columns_hold_the_sentinel(dtype):
    a = wl.matrix(wl.rng_for(4), 5, 100, dtype, stride=104)
    assert a.shape == (5, 104)
    pad = a[:, 100:].view(np.uint32 if dtype == "f32" else np.uint16)
    assert np.all(pad == wl.SENTINEL[dtype])
    assert np.all(np.isnan(decode(a[:, 100:], dtype)))
    body = wl.matrix(wl.rng_for(4), 5, 100, dtype)
    assert np.array_equal(a[:, :100], body)   # padding does not change the samples


def test_outliers_fraction_and_range():
    """1% of entries replaced by +-U(200, 300), as in the padded fp16 workload."""
    x = decode(wl.matrix(wl.rng_for(5), 256, 4096, "f16", outlier_frac=0.01), "f16")
    big = np.abs(x) >= 200
    frac = big.mean()
    assert abs(frac - 0.01) < 5 * np.sqrt(0.01 * 0.99 / x.size)
    assert np.all(np.abs(x[big]) <= 300)
    assert abs(np.mean(x[big] > 0) - 0.5) < 0.05
    assert np.all(np.abs(x[~big]) < 10)
    assert np.all(np.isfinite(x)) and np.max(x**2) > 65504   # squares overflow binary16


def test_row_lognormal_scales_whole_rows():
    """The DiT mix: one exp(N(0, 1)) factor per row."""
    x = decode(wl.matrix(wl.rng_for(6), 4096, 2048, "f32", row_lognormal=True), "f32")
    log_rms = np.log(np.sqrt(np.mean(x**2, axis=1)))
    assert abs(log_rms.mean()) < 0.1
    assert abs(log_rms.std() - 1.0) < 0.05


def test_generate_draw_order_and_override():
    """Tensors of a workload are drawn x, residual, weight, dy from the config's seed;
    M overrides the row count with the same recipe."""
    c = wl.CONFIGS[5]
    d = wl.generate(5, M=8)
    rng = wl.rng_for(c["seed"])
    x = wl.matrix(rng, 8, c["H"], "f16", c["stride"], outlier_frac=0.01)
    r = wl.matrix(rng, 8, c["H"], "f16", c["stride"])
    w = wl.weight(rng, c["H"], "f16")
    dy = wl.matrix(rng, 8, c["H"], "f16", c["stride"])
    for got, want in ((d["x"], x), (d["residual"], r), (d["w"], w), (d["dy"], dy)):
        assert np.array_equal(got, want)
    assert d["x"].shape == (8, 6272)
