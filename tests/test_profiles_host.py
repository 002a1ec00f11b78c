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
