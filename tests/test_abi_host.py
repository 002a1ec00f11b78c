"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/rmsnorm.h declares, and rejects invalid arguments
before touching the device (the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

import residual_add_rmsnorm_fwd_gb300 as rn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, ALIAS = 0, 1, 2


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from residual_add_rmsnorm_fwd_gb300 import build
    build.build()
    return rn.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"rmsnorm_fwd", "rmsnorm_fwd_residual", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
            "rmsnorm_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for s in range(6):
        assert rn.rmsnorm_status_string(s)
    assert rn.rmsnorm_status_string(99) == "unknown status"


X, R, W, Y, S, Q = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000


def fwd(lib, **kw):
    a = dict(x=X, w=W, y=Y, rrms=Q, stride=64, M=4, H=64, eps=1e-5, dtype=2, has_w=1)
    a.update(kw)
    return lib.rmsnorm_fwd(a["x"], a["w"], a["y"], a["rrms"], a["stride"], a["M"], a["H"], a["eps"],
                           a["dtype"], a["has_w"], None)


def fwd_res(lib, **kw):
    a = dict(x=X, r=R, w=W, y=Y, s=S, rrms=Q, stride=64, M=4, H=64, eps=1e-5, dtype=2, has_w=1)
    a.update(kw)
    return lib.rmsnorm_fwd_residual(a["x"], a["r"], a["w"], a["y"], a["s"], a["rrms"], a["stride"], a["M"],
                                    a["H"], a["eps"], a["dtype"], a["has_w"], None)


@pytest.mark.parametrize("kw", [
    dict(x=None), dict(y=None), dict(w=None), dict(H=0), dict(H=-3), dict(M=-1), dict(stride=63),
    dict(eps=-1e-6), dict(eps=float("nan")), dict(eps=float("inf")), dict(dtype=3), dict(dtype=-1),
    dict(x=X + 1), dict(y=Y + 1), dict(w=W + 1), dict(rrms=Q + 2), dict(H=(1 << 24) + 1, stride=(1 << 24) + 1),
    dict(M=1 << 62, stride=1 << 20, H=64),
])
def test_fwd_invalid(lib, kw):
    assert fwd(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(r=None), dict(s=None), dict(r=R + 1)])
def test_fwd_residual_invalid(lib, kw):
    assert fwd_res(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [
    dict(y=X + 2), dict(y=X + 2 * 64 * 3), dict(rrms=X + 8), dict(y=W), dict(rrms=Y + 100),
])
def test_fwd_alias(lib, kw):
    assert fwd(lib, **kw) == ALIAS


def test_exact_in_place_is_accepted(lib):
    # same pointer: validated, then (M = 0) nothing launched
    assert fwd(lib, y=X, M=0) == OK
    assert fwd_res(lib, y=X, s=R, M=0) == OK
    assert fwd_res(lib, s=R + 2, M=4) == ALIAS        # partial overlap stays rejected
    assert fwd_res(lib, y=R, M=4) == ALIAS            # y over the residual is not in place


@pytest.mark.parametrize("kw", [dict(s=X), dict(s=Y), dict(y=R + 64), dict(rrms=S)])
def test_fwd_residual_alias(lib, kw):
    assert fwd_res(lib, **kw) == ALIAS


def test_no_weight_ignores_weight_pointer(lib):
    # w is neither validated nor range-checked when has_weight == 0 (M = 0: no launch)
    assert fwd(lib, w=None, has_w=0, M=0) == OK
    assert fwd(lib, w=Y, has_w=0, M=0) == OK


def test_zero_rows_is_a_no_op(lib):
    assert fwd(lib, M=0) == OK
    assert fwd_res(lib, M=0) == OK
    assert fwd(lib, M=0, eps=0.0) == OK


def test_padded_rows_do_not_alias(lib):
    # y interleaved in x's padding is still rejected (ranges are compared, conservatively)
    assert fwd(lib, stride=128, y=X + 128) == ALIAS


def test_bwd_invalid(lib):
    D, XX, WW, RR, DX, DW = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000

    def bwd(**kw):
        a = dict(dy=D, x=XX, w=WW, rrms=RR, dx=DX, dw=DW, ws=0x700000, wsb=1 << 20, stride=64, M=4,
                 H=64, dtype=1, has_w=1)
        a.update(kw)
        return lib.rmsnorm_bwd(a["dy"], a["x"], a["w"], a["rrms"], a["dx"], a["dw"], a["ws"], a["wsb"],
                               a["stride"], a["M"], a["H"], a["dtype"], a["has_w"], None)

    for kw in (dict(dy=None), dict(x=None), dict(rrms=None), dict(dx=None), dict(w=None), dict(H=0),
               dict(stride=10), dict(dtype=9), dict(dx=DX + 1), dict(rrms=RR + 1), dict(dw=DW + 2), dict(M=-5)):
        assert bwd(**kw) == INVALID, kw


def test_workspace_bytes_invalid(lib):
    out = ctypes.c_size_t(123)
    assert lib.rmsnorm_bwd_workspace_bytes(4, 0, 2, ctypes.byref(out)) == INVALID
    assert lib.rmsnorm_bwd_workspace_bytes(4, 64, 2, None) == INVALID
    assert lib.rmsnorm_bwd_workspace_bytes(0, 64, 2, ctypes.byref(out)) == OK and out.value == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rn, "_lib", None)
    monkeypatch.setattr(rn, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        rn.lib()


def test_bwd_residual_invalid(lib):
    D, R, XX, WW, RR, DX, DW = 0x100000, 0x180000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000

    def bwd(**kw):
        a = dict(dy=D, dr=R, x=XX, w=WW, rrms=RR, dx=DX, dw=DW, ws=0x700000, wsb=1 << 20, stride=64, M=4,
                 H=64, dtype=2, has_w=1)
        a.update(kw)
        return lib.rmsnorm_bwd_residual(a["dy"], a["dr"], a["x"], a["w"], a["rrms"], a["dx"], a["dw"], a["ws"],
                                        a["wsb"], a["stride"], a["M"], a["H"], a["dtype"], a["has_w"], None)

    assert bwd(dr=None) == INVALID
    assert bwd(dr=R + 1) == INVALID
    assert bwd(M=0, dr=None, dw=None) == OK


SC, SH = 0x700000, 0x800000


def adaln(lib, **kw):
    a = dict(x=X, w=W, sc=SC, sh=SH, y=Y, rrms=Q, stride=64, cs=64, rpc=1, M=4, H=64, eps=1e-6, dtype=2,
             has_w=1)
    a.update(kw)
    return lib.rmsnorm_adaln_fwd(a["x"], a["w"], a["sc"], a["sh"], a["y"], a["rrms"], a["stride"], a["cs"],
                                 a["rpc"], a["M"], a["H"], a["eps"], a["dtype"], a["has_w"], None)


@pytest.mark.parametrize("kw", [
    dict(sc=None), dict(sh=None), dict(x=None), dict(y=None), dict(w=None), dict(rpc=0), dict(rpc=-2),
    dict(cs=63), dict(sc=SC + 1), dict(sh=SH + 1), dict(eps=-1.0), dict(dtype=5), dict(stride=32),
    dict(cs=1 << 60, M=5, rpc=1),
])
def test_adaln_invalid(lib, kw):
    assert adaln(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [
    dict(y=SC), dict(y=SH + 2 * 64 * 2), dict(rrms=SC + 16), dict(y=X + 2), dict(y=W),
    # with 2 rows per conditioning row, scale holds rows 0..1 only: row 1 of it still overlaps y
    dict(rpc=2, y=SC + 64 * 2),
])
def test_adaln_alias(lib, kw):
    assert adaln(lib, **kw) == ALIAS


def test_adaln_conditioning_extent(lib):
    # M = 4 rows, 2 per conditioning row: scale spans 2 rows (256 bytes in bf16), so y right after it
    # passes validation (the call then needs a device: no GPU here, so it stops there)
    passed = lambda st: st not in (INVALID, ALIAS)
    assert passed(adaln(lib, rpc=2, y=SC + 2 * 64 * 2))
    assert passed(adaln(lib, rpc=4, sh=SC + 64 * 2))   # one conditioning row each; inputs may overlap
    assert passed(adaln(lib, y=X))                     # in place
    assert adaln(lib, rpc=2, y=SC + 2 * 64 * 2 - 2) == ALIAS
    assert adaln(lib, sc=None, sh=None, x=None, y=None, M=0) == OK
    assert adaln(lib, w=None, has_w=0, M=0) == OK


B, MN = 0x900000, 0xa00000


def ln(lib, fused=False, **kw):
    a = dict(x=X, r=R, w=W, b=B, y=Y, s=S, mean=MN, rstd=Q, stride=64, M=4, H=64, eps=1e-5, dtype=2, has_w=1,
             has_b=1)
    a.update(kw)
    if fused:
        return lib.layernorm_fwd_residual(a["x"], a["r"], a["w"], a["b"], a["y"], a["s"], a["mean"], a["rstd"],
                                          a["stride"], a["M"], a["H"], a["eps"], a["dtype"], a["has_w"],
                                          a["has_b"], None)
    return lib.layernorm_fwd(a["x"], a["w"], a["b"], a["y"], a["mean"], a["rstd"], a["stride"], a["M"], a["H"],
                             a["eps"], a["dtype"], a["has_w"], a["has_b"], None)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("kw", [
    dict(x=None), dict(y=None), dict(w=None), dict(b=None), dict(b=B + 1), dict(mean=MN + 2), dict(rstd=Q + 1),
    dict(eps=-1.0), dict(eps=float("nan")), dict(stride=63), dict(dtype=7), dict(H=0),
])
def test_layernorm_invalid(lib, fused, kw):
    assert ln(lib, fused, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(r=None), dict(s=None), dict(r=R + 1)])
def test_layernorm_residual_invalid(lib, kw):
    assert ln(lib, True, **kw) == INVALID


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("kw", [
    dict(y=B), dict(mean=Y + 8), dict(rstd=MN), dict(mean=X + 4), dict(y=W + 2), dict(rstd=B + 64),
])
def test_layernorm_alias(lib, fused, kw):
    assert ln(lib, fused, **kw) == ALIAS


def test_layernorm_optional_arguments(lib):
    passed = lambda st: st not in (INVALID, ALIAS)   # validation passed; no GPU here to run it
    assert passed(ln(lib, w=None, has_w=0, b=None, has_b=0))
    assert passed(ln(lib, mean=None, rstd=None))
    assert passed(ln(lib, y=X))                                    # in place
    assert passed(ln(lib, True, y=X, s=R))                         # both in place
    assert ln(lib, True, s=X) == ALIAS                             # residual_out over x is not in place
    assert ln(lib, M=0, x=None, y=None) == OK
