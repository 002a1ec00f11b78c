"""Pins for the fp64 CPU oracle: facts fixed by the pages and by mathematics.

Each test ties the oracle to something other than itself: the worked example
(tests/golden/worked_example.txt), closed forms of the forward definition
("Skill: Write a Triton RMSNorm Kernel", Purpose and Required reasoning 5-8),
invariants of the function, and central finite differences of the forward
for the backward formulas (Required reasoning 12).  A dropped term, a wrong
sign or index, eps outside the square root, a row-indexed weight, a mean over
the wrong count or a transposed reduction each fails at least one of them.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(v) for v in nums])
    return vals


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


# ---------------------------------------------------------------- forward --

@pytest.mark.parametrize("dtype", ["f64", "f32"])
def test_worked_example(oracle, dtype):
    g = _read_golden("worked_example.txt")
    st = np.float64 if dtype == "f64" else np.float32
    x = g["x"].astype(st)[None, :]
    w = g["w"].astype(st)
    out = oracle.rmsnorm_fwd(x, w, float(g["eps"][0]), dtype)
    np.testing.assert_allclose(out["y"][0], g["y"], rtol=0, atol=5e-5)
    # the same numbers in closed form: x / sqrt(12.5)
    np.testing.assert_allclose(out["y"][0], np.array([3.0, 4.0]) / np.sqrt(12.5), rtol=1e-15)
    assert out["rrms"][0] == pytest.approx(1 / np.sqrt(12.5), rel=1e-15)


def test_mean_square_of_output(oracle):
    """With w = 1: mean_h(y^2) = ms / (ms + eps)."""
    rng = np.random.default_rng(11)
    for H in (1, 5, 64, 1000):
        x = rng.standard_normal((6, H)) * rng.uniform(0.01, 10, (6, 1))
        eps = 1e-3
        e = oracle.eps_as_f32(eps)
        out = oracle.rmsnorm_fwd(_f64(x), np.ones(H), eps, "f64")
        ms = np.array([np.sum(r * r) / H for r in x])
        lhs = np.mean(out["y"] ** 2, axis=1)
        np.testing.assert_allclose(lhs, ms / (ms + e), rtol=1e-12)


def test_scale_invariance(oracle):
    """y_eps(c x) = y_{eps / c^2}(x) exactly; y(c x) -> y(x) as eps -> 0."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((4, 37))
    w = 1 + 0.1 * rng.standard_normal(37)
    c = 4.0                                   # power of two: scaling is exact
    eps = 1e-2                                # eps / 16 is also exact in binary32
    a = oracle.rmsnorm_fwd(_f64(c * x), w, eps, "f64")["y"]
    b = oracle.rmsnorm_fwd(_f64(x), w, eps / (c * c), "f64")["y"]
    np.testing.assert_allclose(a, b, rtol=1e-14)
    a0 = oracle.rmsnorm_fwd(_f64(3.0 * x), w, 0.0, "f64")["y"]
    b0 = oracle.rmsnorm_fwd(_f64(x), w, 0.0, "f64")["y"]
    np.testing.assert_allclose(a0, b0, rtol=1e-14)


def test_single_column(oracle):
    """H = 1: y = x * w / sqrt(x^2 + eps)."""
    x = np.array([[3.0], [-0.5], [1e-3], [250.0]])
    w = np.array([0.75])
    eps = 1e-4
    e = oracle.eps_as_f32(eps)
    out = oracle.rmsnorm_fwd(x, w, eps, "f64")
    np.testing.assert_allclose(out["y"][:, 0], x[:, 0] * 0.75 / np.sqrt(x[:, 0] ** 2 + e), rtol=1e-15)


def test_constant_row_with_per_column_weight(oracle):
    """x = c on a row: y_h = c * w_h / sqrt(c^2 + eps); the weight follows the column."""
    H = 9
    w = np.linspace(0.5, 1.5, H)
    x = np.array([[2.0] * H, [-7.0] * H, [0.25] * H])
    eps = 1e-5
    e = oracle.eps_as_f32(eps)
    y = oracle.rmsnorm_fwd(x, w, eps, "f64")["y"]
    for i, c in enumerate(x[:, 0]):
        np.testing.assert_allclose(y[i], c * w / np.sqrt(c * c + e), rtol=1e-15)


def test_zero_row(oracle):
    """A zero row with eps > 0 gives y = 0 and rrms = 1 / sqrt(eps)."""
    eps = 1e-6
    out = oracle.rmsnorm_fwd(np.zeros((2, 16)), np.ones(16), eps, "f64")
    assert np.all(out["y"] == 0)
    np.testing.assert_allclose(out["rrms"], 1 / np.sqrt(oracle.eps_as_f32(eps)), rtol=1e-15)


def test_mean_over_full_row_length(oracle):
    """Zero entries count in the mean: [a, b, 0, 0] uses (a^2 + b^2) / 4."""
    x = np.array([[1.5, -2.0, 0.0, 0.0]])
    y = oracle.rmsnorm_fwd(x, None, 0.0, "f64")["y"][0]
    np.testing.assert_allclose(y[:2], x[0, :2] / np.sqrt((1.5 ** 2 + 2.0 ** 2) / 4), rtol=1e-15)


def test_eps_inside_sqrt(oracle):
    """rrms = 1/sqrt(ms + eps), not 1/(sqrt(ms) + eps): distinguishable at small ms."""
    x = np.full((1, 4), 1e-3)
    eps = 1e-4
    e = oracle.eps_as_f32(eps)
    rrms = oracle.rmsnorm_fwd(x, None, eps, "f64")["rrms"][0]
    assert rrms == pytest.approx(1 / np.sqrt(1e-6 + e), rel=1e-14)
    assert abs(rrms - 1 / (1e-3 + e)) / rrms > 0.1


def test_no_weight_equals_unit_weight(oracle):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((5, 33)).astype(np.float32)
    a = oracle.rmsnorm_fwd(x, None, 1e-5, "f32")["y"]
    b = oracle.rmsnorm_fwd(x, np.ones(33, np.float32), 1e-5, "f32")["y"]
    assert np.array_equal(a, b)


def test_residual_fusion_equals_add_then_norm(oracle):
    """norm(x + r) with the add fused equals the add done first (binary64 storage)."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((7, 50))
    r = rng.standard_normal((7, 50))
    w = 1 + 0.1 * rng.standard_normal(50)
    fused = oracle.rmsnorm_fwd(x, w, 1e-5, "f64", residual=r)
    plain = oracle.rmsnorm_fwd(x + r, w, 1e-5, "f64")
    assert np.array_equal(fused["y"], plain["y"])
    assert np.array_equal(fused["s"], x + r)


def test_residual_fusion_bf16_exact_sums(oracle):
    """bf16 storage, sums that are exact in bf16: fused == add-then-norm bitwise."""
    rng = np.random.default_rng(15)
    # small integers: x + r stays an integer below 256, exact in bf16
    xv = rng.integers(-60, 60, (4, 24)).astype(np.float64)
    rv = rng.integers(-60, 60, (4, 24)).astype(np.float64)
    x, r = oracle.encode(xv, "bf16"), oracle.encode(rv, "bf16")
    s = oracle.encode(xv + rv, "bf16")
    w = oracle.encode(1 + 0.1 * rng.standard_normal(24), "bf16")
    fused = oracle.rmsnorm_fwd(x, w, 1e-6, "bf16", residual=r)
    plain = oracle.rmsnorm_fwd(s, w, 1e-6, "bf16")
    assert np.array_equal(fused["y"], plain["y"])


def test_strided_rows_and_threads(oracle):
    """A padded row stride and any thread count give the same numbers."""
    rng = np.random.default_rng(16)
    buf = rng.standard_normal((9, 40))
    x = buf[:, :33]
    w = rng.standard_normal(33)
    a = oracle.rmsnorm_fwd(x, w, 1e-5, "f64", nthreads=1)
    b = oracle.rmsnorm_fwd(np.ascontiguousarray(x), w, 1e-5, "f64", nthreads=4)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["rrms"], b["rrms"])
    dy = rng.standard_normal((9, 33))
    c = oracle.rmsnorm_bwd(dy, x, w, 1e-5, "f64", nthreads=1)
    d = oracle.rmsnorm_bwd(dy, np.ascontiguousarray(x), w, 1e-5, "f64", nthreads=3)
    for k in ("dx", "dweight", "dweight_abs", "rrms"):
        assert np.array_equal(c[k], d[k])


# --------------------------------------------------------------- backward --

def _loss(oracle, x, w, dy, eps):
    """L = sum(dy * y) with the oracle's binary64 forward."""
    return float(np.sum(dy * oracle.rmsnorm_fwd(_f64(x), None if w is None else _f64(w), eps, "f64")["y"]))


@pytest.mark.parametrize("M,H,weighted", [(3, 7, True), (2, 1, True), (4, 33, True),
                                          (3, 7, False), (4, 33, False)])
def test_backward_central_differences(oracle, M, H, weighted):
    rng = np.random.default_rng(100 + M * H)
    x = rng.standard_normal((M, H))
    w = 1 + 0.3 * rng.standard_normal(H) if weighted else None
    dy = rng.standard_normal((M, H))
    eps = 1e-3
    out = oracle.rmsnorm_bwd(dy, x, w, eps, "f64")
    h = 1e-6
    fd_dx = np.zeros_like(x)
    for i in range(M):
        for k in range(H):
            xp, xm = x.copy(), x.copy()
            xp[i, k] += h
            xm[i, k] -= h
            fd_dx[i, k] = (_loss(oracle, xp, w, dy, eps) - _loss(oracle, xm, w, dy, eps)) / (2 * h)
    np.testing.assert_allclose(out["dx"], fd_dx, rtol=1e-6, atol=1e-8)
    if weighted:
        fd_dw = np.zeros(H)
        for k in range(H):
            wp, wm = w.copy(), w.copy()
            wp[k] += h
            wm[k] -= h
            fd_dw[k] = (_loss(oracle, x, wp, dy, eps) - _loss(oracle, x, wm, dy, eps)) / (2 * h)
        np.testing.assert_allclose(out["dweight"], fd_dw, rtol=1e-6, atol=1e-8)


def test_dx_orthogonality_identity(oracle):
    """sum_h x_h dx_h = rrms * eps/(ms+eps) * sum_h dy_h w_h x_h; = 0 when eps = 0."""
    rng = np.random.default_rng(21)
    M, H = 5, 64
    x = rng.standard_normal((M, H))
    w = 1 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((M, H))
    for eps in (0.0, 0.5):
        e = oracle.eps_as_f32(eps)
        out = oracle.rmsnorm_bwd(dy, x, w, eps, "f64")
        ms = np.sum(x * x, axis=1) / H
        rrms = 1 / np.sqrt(ms + e)
        lhs = np.sum(x * out["dx"], axis=1)
        rhs = rrms * (e / (ms + e)) * np.sum(dy * w * x, axis=1)
        scale = np.sum(np.abs(x * out["dx"]), axis=1)
        assert np.all(np.abs(lhs - rhs) <= 1e-13 * scale)


def test_dweight_unit_upstream(oracle):
    """dy = 1 everywhere: dweight_h = sum_i xhat_ih."""
    rng = np.random.default_rng(22)
    x = rng.standard_normal((11, 20))
    out = oracle.rmsnorm_bwd(np.ones_like(x), x, np.ones(20), 1e-5, "f64")
    e = oracle.eps_as_f32(1e-5)
    xhat = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + e)
    np.testing.assert_allclose(out["dweight"], xhat.sum(axis=0), rtol=1e-13)
    np.testing.assert_allclose(out["dweight_abs"], np.abs(xhat).sum(axis=0), rtol=1e-13)


def test_dx_second_form(oracle):
    """The page's alternative form (1/rms)(dy*w - x/(H rms^2) sum(dy*w*x)) agrees."""
    rng = np.random.default_rng(23)
    M, H = 4, 31
    x = rng.standard_normal((M, H))
    w = 1 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((M, H))
    e = oracle.eps_as_f32(1e-5)
    out = oracle.rmsnorm_bwd(dy, x, w, 1e-5, "f64")
    rms = np.sqrt(np.mean(x * x, axis=1, keepdims=True) + e)
    alt = (1 / rms) * (dy * w - x / (H * rms ** 2) * np.sum(dy * w * x, axis=1, keepdims=True))
    np.testing.assert_allclose(out["dx"], alt, rtol=1e-12, atol=1e-14)


def test_backward_rrms_matches_forward(oracle):
    rng = np.random.default_rng(24)
    x = rng.standard_normal((6, 17)).astype(np.float32)
    f = oracle.rmsnorm_fwd(x, None, 1e-5, "f32")
    b = oracle.rmsnorm_bwd(np.ones_like(x), x, None, 1e-5, "f32", want_dx=False, want_dweight=False)
    assert np.array_equal(f["rrms"], b["rrms"])


def test_dx_scale_bounds_dx_and_single_column_form(oracle):
    """dx_scale = |rrms g| + |xhat rrms / H| sum|g xhat| >= |dx|; for H = 1 it is rrms |g| (1 + xhat^2)
    while dx = rrms g (1 - xhat^2) = rrms g eps / (x^2 + eps)."""
    rng = np.random.default_rng(25)
    x = rng.standard_normal((7, 1))
    dy = rng.standard_normal((7, 1))
    w = np.array([0.8])
    eps = 1e-3
    e = oracle.eps_as_f32(eps)
    out = oracle.rmsnorm_bwd(dy, x, w, eps, "f64")
    rrms = 1 / np.sqrt(x[:, 0] ** 2 + e)
    xh = x[:, 0] * rrms
    g = dy[:, 0] * 0.8
    np.testing.assert_allclose(out["dx_scale"][:, 0], rrms * np.abs(g) * (1 + xh ** 2), rtol=1e-14)
    np.testing.assert_allclose(out["dx"][:, 0], rrms * g * e / (x[:, 0] ** 2 + e), rtol=1e-9)
    big = oracle.rmsnorm_bwd(rng.standard_normal((5, 40)), rng.standard_normal((5, 40)), None, eps, "f64")
    assert np.all(big["dx_scale"] >= np.abs(big["dx"]))


def _loss_fused(oracle, x, r, w, dy, dres, eps):
    """L = sum(dy * y) + sum(dres * s) for the fused forward s = x + r, y = norm(s) * w."""
    out = oracle.rmsnorm_fwd(_f64(x), _f64(w), eps, "f64", residual=_f64(r))
    return float(np.sum(dy * out["y"]) + np.sum(dres * out["s"]))


@pytest.mark.parametrize("M,H", [(3, 7), (2, 1), (4, 33)])
def test_fused_backward_central_differences(oracle, M, H):
    """The fused forward's backward: d/dx and d/dresidual of sum(dy*y) + sum(dres*residual_out)
    both equal the norm's dx plus dres."""
    rng = np.random.default_rng(200 + M * H)
    x, r = rng.standard_normal((M, H)), rng.standard_normal((M, H))
    w = 1 + 0.3 * rng.standard_normal(H)
    dy, dres = rng.standard_normal((M, H)), rng.standard_normal((M, H))
    eps = 1e-3
    out = oracle.rmsnorm_bwd(dy, x + r, w, eps, "f64", dres=dres)
    h = 1e-6
    for which in ("x", "r"):
        fd = np.zeros((M, H))
        for i in range(M):
            for k in range(H):
                a, b = [x.copy(), r.copy()], [x.copy(), r.copy()]
                j = 0 if which == "x" else 1
                a[j][i, k] += h
                b[j][i, k] -= h
                fd[i, k] = (_loss_fused(oracle, a[0], a[1], w, dy, dres, eps)
                            - _loss_fused(oracle, b[0], b[1], w, dy, dres, eps)) / (2 * h)
        np.testing.assert_allclose(out["dx"], fd, rtol=1e-6, atol=1e-8)
    plain = oracle.rmsnorm_bwd(dy, x + r, w, eps, "f64")
    np.testing.assert_allclose(out["dweight"], plain["dweight"], rtol=0, atol=0)   # dres does not reach w
    assert np.all(out["dx_scale"] >= np.abs(out["dx"]))


# ------------------------------------------------------------------ AdaLN --

def test_adaln_reduces_to_rmsnorm(oracle):
    """scale = shift = 0: AdaLN is the plain forward, bit for bit."""
    rng = np.random.default_rng(40)
    x = rng.standard_normal((6, 48))
    w = 1 + 0.1 * rng.standard_normal(48)
    z = np.zeros((6, 48))
    a = oracle.rmsnorm_adaln_fwd(x, w, z, z, 1e-5, "f64")
    b = oracle.rmsnorm_fwd(x, w, 1e-5, "f64")
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["rrms"], b["rrms"])


def test_adaln_scale_and_shift_are_affine(oracle):
    """out = (1 + scale) * norm(x) * w + shift, per column and per conditioning row."""
    rng = np.random.default_rng(41)
    M, H = 5, 40
    x = rng.standard_normal((M, H))
    w = 1 + 0.1 * rng.standard_normal(H)
    sc = rng.standard_normal((M, H))
    sh = rng.standard_normal((M, H))
    plain = oracle.rmsnorm_fwd(x, w, 1e-5, "f64")["y"]
    got = oracle.rmsnorm_adaln_fwd(x, w, sc, sh, 1e-5, "f64")["y"]
    np.testing.assert_allclose(got, plain * (1 + sc) + sh, rtol=1e-13, atol=1e-13)


def test_adaln_broadcast_conditioning_rows(oracle):
    """rows_per_cond = S: the [B, 1, H] form equals the [B, S, H] form with the rows repeated."""
    rng = np.random.default_rng(42)
    B, S, H = 3, 4, 24
    x = rng.standard_normal((B * S, H))
    sc, sh = rng.standard_normal((B, H)), rng.standard_normal((B, H))
    a = oracle.rmsnorm_adaln_fwd(x, None, sc, sh, 1e-6, "f64", rows_per_cond=S)["y"]
    b = oracle.rmsnorm_adaln_fwd(x, None, np.repeat(sc, S, axis=0), np.repeat(sh, S, axis=0), 1e-6, "f64")["y"]
    assert np.array_equal(a, b)


def test_adaln_closed_form_single_column(oracle):
    """H = 1: out = x w (1 + s) / sqrt(x^2 + eps) + shift."""
    x = np.array([[2.0], [-0.5]])
    sc, sh = np.array([[0.25], [-1.5]]), np.array([[1.0], [3.0]])
    e = oracle.eps_as_f32(1e-3)
    got = oracle.rmsnorm_adaln_fwd(x, np.array([0.8]), sc, sh, 1e-3, "f64")
    want = x[:, 0] * 0.8 * (1 + sc[:, 0]) / np.sqrt(x[:, 0] ** 2 + e) + sh[:, 0]
    np.testing.assert_allclose(got["y"][:, 0], want, rtol=1e-15)
    assert np.all(got["y_scale"] >= np.abs(got["y"]))


# ------------------------------------------------------- residual + LayerNorm --
# The pages name the fused residual + LayerNorm ("SpeedROCm" page, item 4) but
# print no formula; the oracle takes the textbook LayerNorm (biased variance,
# eps inside the square root, per-column weight and bias).  These pins tie it
# to PyTorch's own LayerNorm (an independent implementation), to closed forms
# and to the RMSNorm oracle.

def test_layernorm_matches_torch_layer_norm(oracle):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(50)
    M, H = 7, 96
    x = rng.standard_normal((M, H)) * 3 + 1.5
    w = 1 + 0.1 * rng.standard_normal(H)
    b = 0.2 * rng.standard_normal(H)
    e = oracle.eps_as_f32(1e-5)
    for wv, bv in ((w, b), (None, None), (w, None), (None, b)):
        got = oracle.layernorm_fwd(x, wv, bv, 1e-5, "f64")
        want = torch.nn.functional.layer_norm(
            torch.from_numpy(x), (H,), None if wv is None else torch.from_numpy(wv),
            None if bv is None else torch.from_numpy(bv), eps=e).numpy()
        np.testing.assert_allclose(got["y"], want, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got["mean"], x.mean(axis=1), rtol=1e-13)


def test_layernorm_output_moments(oracle):
    """w = 1, b = 0: every row of y has mean 0 and mean square var / (var + eps)."""
    rng = np.random.default_rng(51)
    x = rng.standard_normal((5, 64)) * np.array([[0.01], [1], [10], [100], [0.3]]) + 7
    eps = 1e-3
    out = oracle.layernorm_fwd(x, None, None, eps, "f64")
    var = ((x - x.mean(axis=1, keepdims=True)) ** 2).mean(axis=1)
    e = oracle.eps_as_f32(eps)
    np.testing.assert_allclose(out["y"].mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose((out["y"] ** 2).mean(axis=1), var / (var + e), rtol=1e-12)
    np.testing.assert_allclose(out["rstd"], 1 / np.sqrt(var + e), rtol=1e-12)


def test_layernorm_shift_invariance(oracle):
    """LayerNorm(x + c) = LayerNorm(x) for a constant c (integer data: the adds are exact)."""
    rng = np.random.default_rng(52)
    x = rng.integers(-50, 50, (4, 33)).astype(np.float64)
    w = 1 + 0.1 * rng.standard_normal(33)
    b = rng.standard_normal(33)
    a = oracle.layernorm_fwd(x, w, b, 1e-5, "f64")["y"]
    c = oracle.layernorm_fwd(x + 1000.0, w, b, 1e-5, "f64")["y"]
    np.testing.assert_allclose(a, c, rtol=1e-13, atol=1e-13)


def test_layernorm_constant_rows_give_the_bias(oracle):
    """H = 1, or a constant row: s - mean = 0, so y = b exactly and rstd = 1/sqrt(eps)."""
    b = np.array([0.75, -2.0, 0.5])
    x = np.array([[4.0, 4.0, 4.0], [-1.5, -1.5, -1.5]])
    out = oracle.layernorm_fwd(x, np.array([3.0, 2.0, 1.0]), b, 1e-4, "f64")
    assert np.array_equal(out["y"], np.tile(b, (2, 1)))
    np.testing.assert_allclose(out["rstd"], 1 / np.sqrt(oracle.eps_as_f32(1e-4)), rtol=1e-15)
    assert np.array_equal(out["mean"], np.array([4.0, -1.5]))
    one = oracle.layernorm_fwd(np.array([[2.5], [-7.0]]), np.array([5.0]), np.array([0.125]), 1e-5, "f64")
    assert np.array_equal(one["y"][:, 0], np.array([0.125, 0.125]))


def test_layernorm_two_columns_closed_form(oracle):
    """s = [a, c]: mean = (a + c)/2, var = d^2 with d = (a - c)/2, y = (+-d / sqrt(d^2 + eps)) w + b."""
    a, c, eps = 3.0, -1.0, 0.5
    w, b = np.array([2.0, 0.5]), np.array([0.1, -0.3])
    out = oracle.layernorm_fwd(np.array([[a, c]]), w, b, eps, "f64")
    d = (a - c) / 2
    e = oracle.eps_as_f32(eps)
    want = np.array([d, -d]) / np.sqrt(d * d + e) * w + b
    np.testing.assert_allclose(out["y"][0], want, rtol=1e-15)
    assert out["mean"][0] == 1.0


def test_layernorm_residual_fusion_equals_add_then_norm(oracle):
    rng = np.random.default_rng(53)
    x, r = rng.standard_normal((6, 40)), rng.standard_normal((6, 40))
    w, b = 1 + 0.1 * rng.standard_normal(40), rng.standard_normal(40)
    fused = oracle.layernorm_fwd(x, w, b, 1e-5, "f64", residual=r)
    plain = oracle.layernorm_fwd(x + r, w, b, 1e-5, "f64")
    assert np.array_equal(fused["y"], plain["y"])
    assert np.array_equal(fused["s"], x + r)


def test_layernorm_of_zero_mean_rows_is_rmsnorm(oracle):
    """With a row mean of exactly 0 the variance is the mean square: LayerNorm without
    bias equals the RMSNorm oracle on the same row."""
    rng = np.random.default_rng(54)
    v = rng.standard_normal((5, 16))
    x = np.concatenate([v, -v], axis=1)        # exact zero mean
    w = 1 + 0.1 * rng.standard_normal(32)
    ln = oracle.layernorm_fwd(x, w, None, 1e-5, "f64")
    rms = oracle.rmsnorm_fwd(x, w, 1e-5, "f64")
    np.testing.assert_allclose(ln["y"], rms["y"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(ln["rstd"], rms["rrms"], rtol=1e-14)
    assert np.all(ln["y_scale"] >= np.abs(ln["y"]))
