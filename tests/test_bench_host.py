"""Host-side logic of bench.py (no GPU): byte accounting, the clock-sample
parser, whole-job aggregation, and the multi-rank max-over-ranks path run as
two gloo ranks on the CPU."""
import os
import socket

import pytest

import bench


def test_algorithmic_bytes_match_the_workload_table():
    # fused forward, bf16, 16384 x 4096, no rrms: 4 tensors + weight
    assert bench.step_bytes(16384, 4096, 2, fused=True, weight=True, save_rrms=False, backward=False)[0] \
        == 536_879_104
    # forward saving rrms, and backward, bf16 16384 x 8192
    f, b = bench.step_bytes(16384, 8192, 2, fused=False, weight=True, save_rrms=True, backward=True)
    assert f == 536_952_832 and b == 805_421_056
    # fp16 fused forward + backward, 32768 x 6144 (padding excluded)
    f, b = bench.step_bytes(32768, 6144, 2, fused=True, weight=True, save_rrms=True, backward=True)
    assert f == 1_610_756_096 and b == 1_208_127_488
    # long rows: bf16 fused forward + backward, 4096 x 32768 (4 and 3 row streams of 256 MiB,
    # plus weight, rrms and, backward, the fp32 dweight)
    f, b = bench.step_bytes(4096, 32768, 2, fused=True, weight=True, save_rrms=True, backward=True)
    assert f == 4 * 2**28 + 65536 + 16384 and b == 3 * 2**28 + 65536 + 16384 + 131072


def test_long_rows_workload_is_registered_with_its_configuration():
    """The long-row workload is selectable and its configuration has the shape it measures."""
    import workloads as wl
    assert "long_rows" in bench.WORKLOADS
    assert wl.CONFIGS[6]["M"] == 4096 and wl.CONFIGS[6]["H"] == 32768
    assert wl.CONFIGS[4]["name"] == "fwd_bwd_bf16_16384x8192"


def test_odd_rows_workload_is_registered_with_its_configuration():
    """The misaligned-row workload is selectable; its contiguous rows of an odd
    length start at every element offset within 16 bytes in turn."""
    import workloads as wl
    assert "odd_rows" in bench.WORKLOADS
    c = wl.CONFIGS[7]
    assert c["H"] % 2 == 1 and c["stride"] == c["H"] and c["dtype"] == "bf16"
    offsets = {(r * c["stride"] * 2) % 16 for r in range(8)}
    assert offsets == set(range(0, 16, 2))


def test_aggregate_uses_slowest_rank():
    a = bench.aggregate([2.0, 4.0], units_per_rank=100, bytes_per_unit_rank=1e9)
    assert a["ms"] == 4.0
    assert a["units_per_s"] == pytest.approx(2 * 100 / 4e-3)
    assert a["gbs"] == pytest.approx(2 * 1e9 / 4e-3 / 1e9)


def test_clock_parser_and_summary():
    lines = [
        "2026/12/02 10:00:00.100, 0, 1965, 2070, 700.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.300, 0, 1980, 2070, 900.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    rows = bench.parse_clock_lines(lines)
    assert len(rows) == 2 and rows[1]["sw_power_cap"] and not rows[0]["sw_power_cap"]
    t0 = rows[0]["t"]
    s = bench.summarize_clocks(rows, t0, t0 + 1)
    assert s["sm_mhz"] == pytest.approx(1972.5) and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def test_profile_traffic_requires_matching_kernel_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "k.md").write_text(f"- kernel_source_hash: `{h}`\n- dram_bytes_per_launch: 123\n")
    assert bench.profile_traffic("k") == 123
    (tmp_path / "profiles" / "k.md").write_text("- kernel_source_hash: `other`\n- dram_bytes_per_launch: 123\n")
    assert bench.profile_traffic("k") is None
    assert bench.profile_traffic("missing") is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    per_rank_ms = [1.5, 3.0][rank]
    all_ms = bench.max_over_ranks(per_rank_ms, world)
    agg = bench.aggregate(all_ms, units_per_rank=16384, bytes_per_unit_rank=9.4e8)
    bench.barrier(world)
    dist.destroy_process_group()
    q.put((rank, all_ms, agg))


def test_two_rank_aggregation_gloo():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, all_ms, agg in out:
        assert sorted(all_ms) == [1.5, 3.0]
        assert agg["ms"] == 3.0                                # slowest rank
        assert agg["units_per_s"] == pytest.approx(2 * 16384 / 3e-3)


def test_reference_arm_prints_one_contract_line(capsys, monkeypatch):
    """--impl reference times the oracle on the host (no GPU) and prints the
    contract's JSON line; ranks other than 0 print nothing."""
    import json
    monkeypatch.setenv("RANK", "0")
    bench.main(["--impl", "reference", "--workload", "fwd_f32_small", "--steps", "3", "--warmup", "3"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["steps"] == 3 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "fwd_f32_64x1024"
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--workload", "fwd_f32_small", "--steps", "3", "--warmup", "3"])
    assert capsys.readouterr().out.strip() == ""


def test_measured_peak_from_the_peaks_file_else_the_fallback(tmp_path, monkeypatch):
    import json
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6794.8}))
    assert bench.measured_peak() == (6794.8, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text("{}")
    assert bench.measured_peak()[1] == "fallback"
