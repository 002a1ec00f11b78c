"""Mutation check of the oracle's pins (no GPU).

Each case plants one plausible mistake in a copy of oracle/oracle.c, builds
the copy and runs the pins (tests/test_oracle_pins.py, tests/test_codec.py)
against it in a separate process: at least one pin must fail.  The unmutated
copy must pass, so a failure means a pin caught the planted mistake, not that
the harness broke.  Mistakes that would read outside the oracle's buffers are
not planted (the copy runs on the host, but an out-of-bounds read proves
nothing).
"""
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (what the mistake is, text in oracle.c, its replacement[, which occurrence, 1-based]);
# the first occurrence is replaced unless stated
MUTATIONS = [
    # RMSNorm forward
    ("saved rrms inverted", "c->rrms[i] = rrms;", "c->rrms[i] = 1.0 / rrms;"),
    ("eps outside the square root", "const double rrms = 1.0 / sqrt(ms + c->eps);",
     "const double rrms = 1.0 / (sqrt(ms) + c->eps);"),
    ("eps dropped", "const double rrms = 1.0 / sqrt(ms + c->eps);", "const double rrms = 1.0 / sqrt(ms);"),
    ("mean over H + 1", "const double ms = ss / (double)H;", "const double ms = ss / (double)(H + 1);"),
    ("weight indexed by row", "c->y[i * H + h] = (s[h] * rrms) * w;",
     "c->y[i * H + h] = (s[h] * rrms) * (c->w ? load_elem(c->dtype, c->w, i % H) : 1.0);"),
    ("residual subtracted", "s[h] += load_elem(c->dtype, c->r, row + h);",
     "s[h] -= load_elem(c->dtype, c->r, row + h);"),
    # backward
    ("dx sign", "c->dx[i * H + h] = rrms * g - xhat", "c->dx[i * H + h] = rrms * g + xhat"),
    ("dx projection without rrms", "xhat * (rrms / (double)H) * dot;", "xhat * (1.0 / (double)H) * dot;"),
    ("dweight term squared", "acc[h - h0] += t;", "acc[h - h0] += t * t;"),
    ("dweight columns reversed", "acc[h - h0] += t;", "acc[h1 - 1 - h] += t;"),
    ("dresidual_out subtracted", "c->dx[i * H + h] += d;", "c->dx[i * H + h] -= d;"),
    # storage codec
    ("f16 exponent bias", "v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    ("truncation instead of rounding", "double q = rint(ldexp(a, (p - 1) - e));",
     "double q = floor(ldexp(a, (p - 1) - e));"),
    # LayerNorm
    ("variance not centred", "sq += (s[h] - mean) * (s[h] - mean);", "sq += s[h] * s[h];"),
    ("unbiased variance", "const double rstd = 1.0 / sqrt(sq / (double)H + c->eps);",
     "const double rstd = 1.0 / sqrt(sq / (double)(H - 1) + c->eps);"),
    ("LayerNorm eps outside the square root", "const double rstd = 1.0 / sqrt(sq / (double)H + c->eps);",
     "const double rstd = 1.0 / (sqrt(sq / (double)H) + c->eps);"),
    ("no mean subtraction in y", "c->y[i * H + h] = ((s[h] - mean) * rstd) * w + b;",
     "c->y[i * H + h] = (s[h] * rstd) * w + b;"),
    ("bias dropped", "c->y[i * H + h] = ((s[h] - mean) * rstd) * w + b;",
     "c->y[i * H + h] = ((s[h] - mean) * rstd) * w;"),
    ("bias inside the weight", "c->y[i * H + h] = ((s[h] - mean) * rstd) * w + b;",
     "c->y[i * H + h] = ((s[h] - mean) * rstd) * (w + b);"),
    ("bias indexed by row", "const double b = c->b ? load_elem(c->dtype, c->b, h) : 0.0;",
     "const double b = c->b ? load_elem(c->dtype, c->b, i % H) : 0.0;"),
    ("LayerNorm mean over H + 1", "const double mean = sum / (double)H;",
     "const double mean = sum / (double)(H + 1);"),
    ("LayerNorm residual subtracted", "s[h] += load_elem(c->dtype, c->r, row + h);",
     "s[h] -= load_elem(c->dtype, c->r, row + h);", 2),
    # AdaLN
    ("AdaLN without the 1 +", "* w) * (1.0 + sc);", "* w) * (sc);"),
    ("AdaLN shift subtracted", "c->y[i * H + h] = t + sh;", "c->y[i * H + h] = t - sh;"),
    ("AdaLN always conditioning row 0", "const int64_t crow = (i / c->rows_per_cond) * c->cond_stride;",
     "const int64_t crow = (0 * i) * c->cond_stride;"),
]


def _copy_tree(dst):
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "helpers.py", "test_oracle_pins.py", "test_codec.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    for f in ("workloads.py", "pytest.ini"):
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))


def _run_pins(tree):
    env = dict(os.environ, PYTHONPATH=tree)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_codec.py"],
                       cwd=tree, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout + r.stderr


def test_unmutated_copy_passes_the_pins(tmp_path):
    tree = str(tmp_path / "tree")
    _copy_tree(tree)
    rc, out = _run_pins(tree)
    assert rc == 0, out[-2000:]


def _replace_nth(text, old, new, n):
    at = -1
    for _ in range(n):
        at = text.find(old, at + 1)
        assert at >= 0, f"occurrence {n} of the mutation site not found in oracle.c"
    return text[:at] + new + text[at + len(old):]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, mutation):
    what, old, new = mutation[:3]
    nth = mutation[3] if len(mutation) > 3 else 1
    tree = str(tmp_path / "tree")
    _copy_tree(tree)
    src = os.path.join(tree, "oracle", "oracle.c")
    with open(src) as f:
        text = f.read()
    with open(src, "w") as f:
        f.write(_replace_nth(text, old, new, nth))
    rc, out = _run_pins(tree)
    assert rc != 0 and re.search(r"\d+ failed", out), f"no pin caught '{what}':\n{out[-2000:]}"
