"""The ncu summaries under profiles/ (no GPU): each names the command that
made it (the committed benchmark), records the kernel-source hash it was
captured at, and, for kernel summaries, the DRAM bytes per launch that
bench.py reports as roofline.traffic when the hash still matches."""
import glob
import os
import re

import bench

PROFILES = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")))


def _fields(path):
    rec = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"- (\w+): `([^`]*)`", line)
            if m:
                rec[m.group(1)] = m.group(2)
    return rec


def test_every_summary_names_its_command_and_hash():
    assert PROFILES
    for p in PROFILES:
        text = open(p).read()
        assert "ncu " in text and "--clock-control none" in text, p
        assert "python bench.py" in text, p          # the capture ran the committed benchmark
        assert re.fullmatch(r"[0-9a-f]{16}", _fields(p).get("kernel_source_hash", "")), p


def test_kernel_summaries_record_dram_bytes():
    for p in PROFILES:
        if os.path.basename(p).startswith("launch_list"):
            continue
        assert int(_fields(p)["dram_bytes_per_launch"]) > 0, p


def test_all_summaries_come_from_one_build():
    assert len({_fields(p)["kernel_source_hash"] for p in PROFILES}) == 1


def test_benchmark_reads_the_step_summary():
    """The default step's dominant kernel has a summary under the label bench.py looks up."""
    assert os.path.exists(os.path.join(bench.ROOT, "profiles", "fwd_residual_bf16_16384x4096.md"))


def _bench_line(workload):
    path = os.path.join(bench.ROOT, "profiles", f"bench_{workload}.json")
    assert os.path.exists(path), f"no recorded benchmark line for workload {workload}"
    import json
    with open(path) as f:
        lines = [ln for ln in f.read().splitlines() if ln.strip()]
    assert len(lines) == 1, path
    return json.loads(lines[0])


def test_every_workload_has_a_recorded_line_from_the_current_kernels():
    """One JSON line per benchmark workload, written by `bench.py --record`
    from the kernel sources as they are now."""
    h = bench.kernel_source_hash()
    for w in bench.WORKLOADS:
        rec = _bench_line(w)
        assert rec["kernel_source_hash"] == h, f"{w}: recorded from other kernel sources"
        assert rec["command"].startswith("python bench.py") and f"--workload {w}" in rec["command"], w
        for key in ("metric", "value", "unit", "clocks", "kernels", "roofline", "cpu_baseline", "e2e", "spread"):
            assert key in rec, f"{w}: no {key}"
        assert rec["metric"] == bench.METRIC
        assert rec["clocks"]["samples"] > 0 and not set(rec["clocks"]["reasons"]) & {
            "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}, w
        assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1, w
        assert 0 < rec["roofline"]["frac"] < 1.2, w


def test_recorded_lines_are_self_consistent():
    """value = algorithmic bytes per step / ms per step, and the roofline
    fraction = achieved / peak, as bench.py computes them."""
    for w in bench.WORKLOADS:
        rec = _bench_line(w)
        b = rec["config"]["algorithmic_bytes_per_step"]
        assert abs(b / (rec["ms_per_step"] / 1e3) / 1e9 - rec["value"]) <= 0.01 * rec["value"], w
        r = rec["roofline"]
        assert abs(r["achieved"] / r["peak"] - r["frac"]) < 1e-3, w
