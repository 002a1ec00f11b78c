"""The oracle and the CUDA path share nothing (no GPU): the library package
neither imports nor includes anything of the oracle, the oracle neither
imports nor includes anything of the package, and bench.py loads the oracle
only inside its CPU-baseline and reference legs."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "residual_add_rmsnorm_fwd_gb300")


def _module_imports(path, top_level_only=False):
    tree = ast.parse(open(path).read())
    nodes = tree.body if top_level_only else ast.walk(tree)
    names = set()
    for n in nodes:
        if isinstance(n, ast.Import):
            names |= {a.name.split(".")[0] for a in n.names}
        elif isinstance(n, ast.ImportFrom) and n.module:
            names.add(n.module.split(".")[0])
    return names


def test_package_does_not_use_the_oracle():
    for py in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        assert "oracle" not in _module_imports(py), py
    for src in glob.glob(os.path.join(PKG, "csrc", "*")):
        text = open(src).read()
        for inc in re.findall(r'#include\s+"([^"]+)"', text):
            assert "oracle" not in inc, (src, inc)


def test_oracle_does_not_use_the_package():
    for py in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert "residual_add_rmsnorm_fwd_gb300" not in _module_imports(py), py
    text = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', text):
        assert "rmsnorm" not in inc and "csrc" not in inc, inc


def test_bench_imports_the_oracle_only_in_its_host_legs():
    path = os.path.join(ROOT, "bench.py")
    assert "oracle" not in _module_imports(path, top_level_only=True)
    tree = ast.parse(open(path).read())
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for n in ast.walk(fn):
                if isinstance(n, ast.Import) and any(a.name == "oracle" for a in n.names):
                    users.add(fn.name)
    assert users and users <= {"oracle_step", "run_reference", "cpu_baseline", "run_cpu_baseline"}, users


def test_workloads_holds_no_method_arithmetic():
    """The shared input module draws and rounds numbers only: no rsqrt, no
    mean of squares, no normalisation."""
    text = open(os.path.join(ROOT, "workloads.py")).read()
    for pattern in (r"rsqrt", r"\bsqrt\(", r"\*\*\s*2", r"mean\("):
        assert not re.search(pattern, text), pattern
