#!/usr/bin/env python3
"""Benchmark of the GB300 RMSNorm engine.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload step|fused_fwd|fused_fwd_bwd_residual|dit_mix|fwd_f32_small|
                                fwd_bwd_8192|fused_f16_padded|adaln|adaln_per_token|
                                ln_residual|ln_residual_f32|ln_plain|long_rows|odd_rows]

Default workload ("step"): one pass of the whole hot path on the
(B=8, T=2048, H=4096) bf16 activations, M = 16384 rows -- the fused
residual-add + RMSNorm forward (x, residual -> y, residual_out, rrms) followed
by the backward on its output (dy, residual_out, rrms -> dx, dweight).  Inputs
are seeded synthetic N(0, 1) activations and a 1 + 0.1 N(0, 1) weight.
The metric is achieved HBM bandwidth over the algorithmic bytes (every M x H
tensor read or written once, plus weight, rrms and dweight), with rows/s
beside it.

Prints ONE JSON line (rank 0).  Timing: W untimed warm-up steps, then K
steps between a barrier + synchronize on both sides, CUDA events on the
launching stream, max over ranks.  The K steps are replays of a CUDA graph
that holds R steps (R the largest divisor of K up to 10), so the host issues
no launch per kernel and nothing sits between the kernels.  Per-kernel
figures (and the roofline of the dominant kernel) come from a second pass
that brackets every call with CUDA events.  ``--eager`` launches every call
from the host instead.  The per-step working set (~0.94 GB) is
larger than L2, so no flush is needed between steps.

``--impl reference`` times the fp64 CPU oracle (the only other implementation
of this method here) on a bounded row sample of the same workload, on the
host cores, and prints the same line shape with "impl": "reference".
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and rows/s for residual+RMSNorm fwd/bwd"
NOMINAL_HBM_GBS = 8000.0
SPREAD_REPS = 50
L2_BYTES = 129 * 2 ** 20
ISOLATED_LAUNCHES = 8
ISOLATED_REPS = 20
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["residual_add_rmsnorm_fwd_gb300/csrc/*.cu", "residual_add_rmsnorm_fwd_gb300/csrc/*.cuh",
                  "residual_add_rmsnorm_fwd_gb300/csrc/*.h"]


# --------------------------------------------------------------------------
# small host utilities (no GPU needed; unit-tested on CPU)
# --------------------------------------------------------------------------

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for pat in KERNEL_SOURCES:
        for p in sorted(glob.glob(os.path.join(ROOT, pat))):
            h.update(os.path.basename(p).encode())
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    """(GB/s, source) from the generated peaks file, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_label: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, or
    None when no summary exists or the kernels changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel_label}.md")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                rec[k.strip()] = v.strip().strip("`")
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return int(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def aggregate(per_rank_ms, units_per_rank, bytes_per_unit_rank):
    """Whole-job numbers from per-rank timings: every rank processed the same
    units; the job time is the slowest rank's."""
    t = max(per_rank_ms)
    n = len(per_rank_ms)
    return {"ms": t, "units_per_s": n * units_per_rank / (t / 1e3),
            "gbs": n * bytes_per_unit_rank / (t / 1e3) / 1e9}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 10):
        self.gpu, self.period, self.proc, self.out = gpu_index, period_ms, None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_lines(out.splitlines())


def parse_clock_lines(lines):
    rows = []
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) != len(ClockSampler.FIELDS):
            continue
        try:
            ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            rows.append({"t": ts + frac, "sm": float(parts[2]), "sm_max": float(parts[3]),
                         "power": float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else None,
                         "hw_slowdown": parts[6] == "Active", "hw_thermal_slowdown": parts[7] == "Active",
                         "sw_thermal_slowdown": parts[8] == "Active", "sw_power_cap": parts[9] == "Active"})
        except (ValueError, IndexError):
            continue
    return rows


def summarize_clocks(rows, t0, t1, margin=0.02):
    """Clocks and throttle reasons of the samples taken in [t0, t1] (all
    samples when none fell inside)."""
    inside = [r for r in rows if t0 - margin <= r["t"] <= t1 + margin]
    use = inside if inside else rows
    if not use:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    reasons = sorted({k for r in use for k in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                                "sw_power_cap") if r[k]})
    return {"sm_mhz": statistics.median(r["sm"] for r in use), "sm_min_mhz": min(r["sm"] for r in use),
            "sm_max_mhz": max(r["sm_max"] for r in use), "reasons": reasons, "samples": len(use),
            "in_window": bool(inside)}


def spread_stats(ms_per_step):
    """Median and interquartile range of per-replay times (ms per step)."""
    v = sorted(ms_per_step)
    q = statistics.quantiles(v, n=4, method="inclusive") if len(v) >= 2 else [v[0]] * 3
    return {"reps": len(v), "ms_per_step_median": round(q[1], 5), "ms_per_step_p25": round(q[0], 5),
            "ms_per_step_p75": round(q[2], 5), "iqr_pct_of_median": round(100 * (q[2] - q[0]) / q[1], 3),
            "ms_per_step_min": round(v[0], 5), "ms_per_step_max": round(v[-1], 5)}


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

def step_bytes(M, H, es, fused=True, weight=True, save_rrms=True, backward=True, dres=False):
    """Algorithmic bytes: each M x H tensor once, plus weight, rrms, dweight
    (the fused backward also reads the residual stream's gradient)."""
    mh = M * H * es
    fwd = (4 if fused else 2) * mh + (H * es if weight else 0) + (M * 4 if save_rrms else 0)
    bwd = ((4 if dres else 3) * mh + M * 4 + (H * es + H * 4 if weight else 0)) if backward else 0
    return fwd, bwd


class StepWorkload:
    """Fused forward + backward on one batch (the default benchmark step)."""
    name = "fused_fwd_bwd_bf16_B8xT2048xH4096"

    flush_l2 = False

    def __init__(self, cfg_id=2, backward=True, fused=None, dres=False):
        import torch
        import residual_add_rmsnorm_fwd_gb300 as rn
        import workloads as wl
        self.torch, self.rn, self.wl = torch, rn, wl
        c = wl.CONFIGS[cfg_id]
        self.c, self.cfg_id = c, cfg_id
        self.fused = c["residual"] if fused is None else fused
        self.backward = backward
        self.M, self.H, self.S, self.dt = c["M"], c["H"], c["stride"], c["dtype"]
        self.es = wl.ELEM_BYTES[self.dt]
        self.dres = dres and self.fused and backward
        self.fwd_bytes, self.bwd_bytes = step_bytes(self.M, self.H, self.es, self.fused, True, backward, backward,
                                                    self.dres)
        self.bytes_per_step = self.fwd_bytes + self.bwd_bytes
        self.rows_per_step = self.M
        self.host = wl.generate(cfg_id, with_dy=backward)
        if self.dres:   # the residual stream's incoming gradient, drawn after dy
            rng = wl.rng_for(self.c["seed"] + 100)
            self.host["dres"] = wl.matrix(rng, self.M, self.H, self.dt, self.S)
        if cfg_id == 2:
            kind = "fused_fwd_bwd_residual" if self.dres else ("fused_fwd_bwd" if backward else "fused_fwd")
            self.name = kind + "_bf16_B8xT2048xH4096"
        else:
            self.name = c["name"]
        self.kernels_per_step = 1 + (2 if backward else 0)

    def _make_set(self):
        """One set of device buffers (inputs uploaded, outputs allocated)."""
        from types import SimpleNamespace
        torch, wl, dt = self.torch, self.wl, self.dt
        tdt = wl.torch_dtype(dt)
        dev = torch.device("cuda")
        M, H, S = self.M, self.H, self.S

        def up(a):
            return wl.to_torch(a, dt).to(dev)[:, :H]

        def out():
            return torch.empty(M, S, dtype=tdt, device=dev)[:, :H]

        b = SimpleNamespace()
        b.x = up(self.host["x"])
        b.r = up(self.host["residual"]) if self.fused else None
        b.y = out()
        b.s = out() if self.fused else None
        b.rrms = torch.empty(M, device=dev) if self.backward else None
        if self.backward:
            b.dy = up(self.host["dy"])
            b.dres = up(self.host["dres"]) if self.dres else None
            b.dx = out()
            b.dw = torch.empty(H, device=dev)
            b.ws = torch.empty(max(1, self.rn.rmsnorm_bwd_workspace_bytes(M, H, tdt)), dtype=torch.uint8,
                               device=dev)
        return b

    def setup(self):
        self.w = self.wl.to_torch(self.host["w"], self.dt).to(self.torch.device("cuda"))
        self.sets = [self._make_set()]
        return self

    def calls(self, k=0):
        """[(label, fn, algorithmic bytes)] on buffer set k, enqueued on the current stream, in order."""
        rn, eps, b = self.rn, self.c["eps"], self.sets[k]
        out = []
        if self.fused:
            out.append(("fwd_residual", lambda: rn.rmsnorm_fwd_residual(b.x, b.r, self.w, b.y, b.s, b.rrms, eps=eps),
                        self.fwd_bytes))
        else:
            out.append(("fwd", lambda: rn.rmsnorm_fwd(b.x, self.w, b.y, b.rrms, eps=eps), self.fwd_bytes))
        if self.dres:
            out.append(("bwd_residual", lambda: rn.rmsnorm_bwd_residual(b.dy, b.dres, b.s, self.w, b.rrms, b.dx, b.dw,
                                                                        b.ws), self.bwd_bytes))
        elif self.backward:
            xin = b.s if self.fused else b.x
            out.append(("bwd", lambda: rn.rmsnorm_bwd(b.dy, xin, self.w, b.rrms, b.dx, b.dw, b.ws), self.bwd_bytes))
        return out

    def config(self):
        cfg = {"workload": self.name, "M": self.M, "H": self.H, "row_stride": self.S, "dtype": self.dt,
               "fused_residual": self.fused, "backward": self.backward, "eps": self.c["eps"],
               "l2": ("flushed before every step (256 MiB write); time = sum of the per-call CUDA-event "
                      "intervals" if self.flush_l2 else "no flush: per-step working set larger than L2"),
               "algorithmic_bytes_per_step": self.bytes_per_step}
        if self.cfg_id == 2:
            cfg.update(B=8, T=2048)
        return cfg

    # end to end through the binding: pinned host inputs and outputs, two
    # device buffer sets so that copies of one step overlap another's kernels
    def e2e_setup(self):
        torch, b = self.torch, self.sets[0]
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
        host = lambda a: self.wl.to_torch(a, self.dt)[:, :self.H].contiguous().pin_memory()  # noqa: E731
        self.h_in = [host(self.host["x"])] + ([host(self.host["residual"])] if self.fused else []) + \
            ([host(self.host["dy"])] if self.backward else []) + ([host(self.host["dres"])] if self.dres else [])
        outs = [b.y] + ([b.s] if self.fused else []) + ([b.dx, b.dw] if self.backward else [])
        self.h_out = [pin(t) for t in outs]
        while len(self.sets) < 2:
            self.sets.append(self._make_set())
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out)

    def e2e_transfers(self, k):
        """([(device, host)] inputs, [(host, device)] results) of buffer set k."""
        b = self.sets[k]
        dev_in = [b.x] + ([b.r] if self.fused else []) + ([b.dy] if self.backward else []) + \
            ([b.dres] if self.dres else [])
        dev_out = [b.y] + ([b.s] if self.fused else []) + ([b.dx, b.dw] if self.backward else [])
        return list(zip(dev_in, self.h_in)), list(zip(self.h_out, dev_out))

    # CPU oracle on a row sample of the same inputs
    def oracle_step(self, rows):
        import oracle
        H, dt, eps = self.H, self.dt, self.c["eps"]
        x = self.host["x"][:rows, :H]
        r = self.host["residual"][:rows, :H] if self.fused else None
        f = oracle.rmsnorm_fwd(x, self.host["w"], eps, dt, residual=r)
        if self.backward:
            s = oracle.encode(f["s"], dt)
            oracle.rmsnorm_bwd(self.host["dy"][:rows, :H], s, self.host["w"], eps, dt,
                               dres=self.host["dres"][:rows, :H] if self.dres else None)
        return rows * self.bytes_per_step / self.M


class DitMixWorkload:
    """The DiT/video norm mix: 168 forward calls on 12288 x 2048 bf16 tokens
    (56 with a weight, 112 without, interleaved) plus one per-head norm on
    393216 x 64, per step.  Four x/y buffer sets rotate so that consecutive
    calls never find their operands in L2."""
    name = "dit_mix_bf16_168x12288x2048_plus_heads_393216x64"
    flush_l2 = False

    def __init__(self):
        import torch
        import residual_add_rmsnorm_fwd_gb300 as rn
        import workloads as wl
        self.torch, self.rn, self.wl = torch, rn, wl
        self.c = wl.CONFIGS[3]
        c = self.c
        self.M, self.H, self.S, self.dt = c["M"], c["H"], c["stride"], c["dtype"]
        self.es = wl.ELEM_BYTES[self.dt]
        self.n_calls = c["calls_weighted"] + c["calls_unweighted"]
        self.host = wl.generate(3)
        mh = self.M * self.H * self.es
        hb = c["head_M"] * c["head_H"] * self.es
        self.call_bytes_w, self.call_bytes_nw = 2 * mh + self.H * self.es, 2 * mh
        self.head_bytes = 2 * hb + c["head_H"] * self.es
        self.bytes_per_step = (c["calls_weighted"] * self.call_bytes_w + c["calls_unweighted"] * self.call_bytes_nw
                               + self.head_bytes)
        self.rows_per_step = self.n_calls * self.M + c["head_M"]
        self.kernels_per_step = self.n_calls + 1

    def _make_set(self):
        from types import SimpleNamespace
        torch, wl, dt = self.torch, self.wl, self.dt
        dev = torch.device("cuda")
        b = SimpleNamespace()
        b.xs = [wl.to_torch(a, dt).to(dev) for a in self.host["xs"]]
        b.ys = [torch.empty_like(x) for x in b.xs]
        b.hx = wl.to_torch(self.host["head_x"], dt).to(dev)
        b.hy = torch.empty_like(b.hx)
        return b

    def setup(self):
        dev = self.torch.device("cuda")
        self.w = self.wl.to_torch(self.host["w"], self.dt).to(dev)
        self.hw = self.wl.to_torch(self.host["head_w"], self.dt).to(dev)
        self.sets = [self._make_set()]
        return self

    def calls(self, k=0):
        rn, eps, b = self.rn, self.c["eps"], self.sets[k]
        nb = len(b.xs)
        out = []
        for i in range(self.n_calls):
            x, y = b.xs[i % nb], b.ys[i % nb]
            if i % 3 == 0:   # one call in three has a weight: 56 of 168
                out.append(("fwd_2048_weighted", lambda x=x, y=y: rn.rmsnorm_fwd(x, self.w, y, None, eps=eps),
                            self.call_bytes_w))
            else:
                out.append(("fwd_2048_unweighted", lambda x=x, y=y: rn.rmsnorm_fwd(x, None, y, None, eps=eps),
                            self.call_bytes_nw))
        out.append(("fwd_heads_64", lambda: rn.rmsnorm_fwd(b.hx, self.hw, b.hy, None, eps=eps), self.head_bytes))
        return out

    def config(self):
        c = self.c
        return {"workload": self.name, "M": self.M, "H": self.H, "dtype": self.dt, "calls_per_step": self.n_calls,
                "weighted_calls": c["calls_weighted"], "unweighted_calls": c["calls_unweighted"],
                "head_M": c["head_M"], "head_H": c["head_H"], "eps": c["eps"],
                "l2": f"{len(self.sets[0].xs)} rotating x/y buffer sets of {2 * self.M * self.H * self.es} bytes",
                "algorithmic_bytes_per_step": self.bytes_per_step}

    def e2e_setup(self):
        torch, b = self.torch, self.sets[0]
        self.h_in = [x.cpu().pin_memory() for x in b.xs] + [b.hx.cpu().pin_memory()]
        self.h_out = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in b.ys + [b.hy]]
        while len(self.sets) < 2:
            self.sets.append(self._make_set())
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out)

    def e2e_transfers(self, k):
        b = self.sets[k]
        return list(zip(b.xs + [b.hx], self.h_in)), list(zip(self.h_out, b.ys + [b.hy]))

    def oracle_step(self, rows):
        import oracle
        x = self.host["xs"][0][:rows]
        oracle.rmsnorm_fwd(x, self.host["w"], self.c["eps"], self.dt)
        return rows * self.call_bytes_w / self.M


class AdalnWorkload:
    """AdaLN forward of a DiT block: y = norm(x) * w * (1 + scale) + shift on
    2 sequences x 6144 tokens x 2048 bf16 (the video-DiT token shape of the
    168-call mix), one conditioning row per sequence broadcast over its
    tokens (``per_token``: one conditioning row per token, scale and shift
    as large as x).  Eight calls per step over four rotating buffer sets, so
    that no call finds its operands in L2."""
    flush_l2 = False
    n_calls, n_sets = 8, 4

    def __init__(self, per_token=False):
        import torch
        import residual_add_rmsnorm_fwd_gb300 as rn
        import workloads as wl
        self.torch, self.rn, self.wl = torch, rn, wl
        self.B, self.T, self.H, self.dt, self.eps = 2, 6144, 2048, "bf16", 1e-6
        self.M, self.S = self.B * self.T, self.H
        self.es = wl.ELEM_BYTES[self.dt]
        self.per_token = per_token
        self.rpc = 1 if per_token else self.T
        self.n_cond = self.M // self.rpc
        self.name = f"adaln_bf16_2x6144x2048_per_{'token' if per_token else 'sequence'}"
        rng = wl.rng_for(41 if per_token else 40)
        self.host = {"xs": [wl.matrix(rng, self.M, self.H, self.dt) for _ in range(self.n_sets)],
                     "w": wl.weight(rng, self.H, self.dt)}
        n_cond_sets = self.n_sets if per_token else 1
        self.host["scales"] = [wl.conditioning(rng, self.n_cond, self.H, self.dt) for _ in range(n_cond_sets)]
        self.host["shifts"] = [wl.conditioning(rng, self.n_cond, self.H, self.dt) for _ in range(n_cond_sets)]
        self.call_bytes = (2 * self.M * self.H + 2 * self.n_cond * self.H + self.H) * self.es
        self.bytes_per_step = self.n_calls * self.call_bytes
        self.rows_per_step = self.n_calls * self.M
        self.kernels_per_step = self.n_calls

    def _make_set(self):
        from types import SimpleNamespace
        torch, wl, dt = self.torch, self.wl, self.dt
        dev = torch.device("cuda")
        b = SimpleNamespace()
        up = lambda a: wl.to_torch(a, dt).to(dev)  # noqa: E731
        b.xs = [up(a) for a in self.host["xs"]]
        b.ys = [torch.empty_like(x) for x in b.xs]
        b.scs = [up(a) for a in self.host["scales"]]
        b.shs = [up(a) for a in self.host["shifts"]]
        return b

    def setup(self):
        self.w = self.wl.to_torch(self.host["w"], self.dt).to(self.torch.device("cuda"))
        self.sets = [self._make_set()]
        return self

    def calls(self, k=0):
        rn, b, n = self.rn, self.sets[k], self.n_sets
        label = "adaln_per_token" if self.per_token else "adaln"
        return [(label, lambda x=b.xs[i % n], y=b.ys[i % n], sc=b.scs[i % len(b.scs)], sh=b.shs[i % len(b.shs)]:
                 rn.rmsnorm_adaln_fwd(x, self.w, sc, sh, y, rows_per_cond=self.rpc, eps=self.eps), self.call_bytes)
                for i in range(self.n_calls)]

    def config(self):
        return {"workload": self.name, "M": self.M, "H": self.H, "B": self.B, "T": self.T, "dtype": self.dt,
                "rows_per_cond": self.rpc, "calls_per_step": self.n_calls, "eps": self.eps,
                "l2": f"{self.n_sets} rotating buffer sets of {self.call_bytes} bytes",
                "algorithmic_bytes_per_step": self.bytes_per_step}

    def e2e_setup(self):
        torch, b = self.torch, self.sets[0]
        self.h_in = [t.cpu().pin_memory() for t in b.xs + b.scs + b.shs]
        self.h_out = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in b.ys]
        while len(self.sets) < 2:
            self.sets.append(self._make_set())
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out)

    def e2e_transfers(self, k):
        b = self.sets[k]
        return list(zip(b.xs + b.scs + b.shs, self.h_in)), list(zip(self.h_out, b.ys))

    def oracle_step(self, rows):
        import oracle
        n = -(-rows // self.rpc)
        oracle.rmsnorm_adaln_fwd(self.host["xs"][0][:rows], self.host["w"], self.host["scales"][0][:n],
                                 self.host["shifts"][0][:n], self.eps, self.dt, rows_per_cond=self.rpc)
        return rows * self.call_bytes / self.M


class LayerNormWorkload:
    """Residual + LayerNorm forward: residual_out = x + r, y = LayerNorm(x + r)
    * w + b, on the token shape of the default step (B 8 x T 2048 x H 4096,
    bf16) or on fp32 rows of 1024 (the fp32 eval-mode setting of the page's
    fused residual + LayerNorm); ``fused=False``: the plain LayerNorm y =
    LayerNorm(x) * w + b on the same shape.  Inputs are larger than L2; mean
    and rstd are saved."""
    flush_l2 = False

    def __init__(self, dtype="bf16", M=16384, H=4096, fused=True):
        import torch
        import residual_add_rmsnorm_fwd_gb300 as rn
        import workloads as wl
        self.torch, self.rn, self.wl = torch, rn, wl
        self.dt, self.M, self.H, self.S, self.eps = dtype, M, H, H, 1e-5
        self.es = wl.ELEM_BYTES[dtype]
        self.fused = fused
        self.name = f"ln_{'residual' if fused else 'plain'}_{dtype}_{M}x{H}"
        rng = wl.rng_for(60)
        self.host = {"x": wl.matrix(rng, M, H, dtype), "residual": wl.matrix(rng, M, H, dtype),
                     "w": wl.weight(rng, H, dtype), "b": wl.conditioning(rng, 1, H, dtype, sigma=0.1)[0]}
        self.bytes_per_step = (4 if fused else 2) * M * H * self.es + 2 * H * self.es + 2 * M * 4
        self.rows_per_step = M
        self.kernels_per_step = 1

    def _make_set(self):
        from types import SimpleNamespace
        torch, wl, dt = self.torch, self.wl, self.dt
        dev = torch.device("cuda")
        b = SimpleNamespace()
        b.x = wl.to_torch(self.host["x"], dt).to(dev)
        b.r = wl.to_torch(self.host["residual"], dt).to(dev)
        b.y, b.s = torch.empty_like(b.x), torch.empty_like(b.x)
        b.mean = torch.empty(self.M, device=dev)
        b.rstd = torch.empty(self.M, device=dev)
        return b

    def setup(self):
        dev = self.torch.device("cuda")
        self.w = self.wl.to_torch(self.host["w"], self.dt).to(dev)
        self.bias = self.wl.to_torch(self.host["b"], self.dt).to(dev)
        self.sets = [self._make_set()]
        return self

    def calls(self, k=0):
        rn, b = self.rn, self.sets[k]
        if not self.fused:
            return [("ln", lambda: rn.layernorm_fwd(b.x, self.w, self.bias, b.y, b.mean, b.rstd, eps=self.eps),
                     self.bytes_per_step)]
        return [("ln_residual", lambda: rn.layernorm_fwd_residual(b.x, b.r, self.w, self.bias, b.y, b.s, b.mean,
                                                                  b.rstd, eps=self.eps), self.bytes_per_step)]

    def config(self):
        return {"workload": self.name, "M": self.M, "H": self.H, "dtype": self.dt, "fused_residual": self.fused,
                "bias": True, "eps": self.eps, "l2": "no flush: per-step working set larger than L2",
                "algorithmic_bytes_per_step": self.bytes_per_step}

    def e2e_setup(self):
        torch, b = self.torch, self.sets[0]
        ins = [b.x, b.r] if self.fused else [b.x]
        outs = [b.y, b.s] if self.fused else [b.y]
        self.h_in = [t.cpu().pin_memory() for t in ins]
        self.h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        while len(self.sets) < 2:
            self.sets.append(self._make_set())
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out)

    def e2e_transfers(self, k):
        b = self.sets[k]
        ins = [b.x, b.r] if self.fused else [b.x]
        outs = [b.y, b.s] if self.fused else [b.y]
        return list(zip(ins, self.h_in)), list(zip(self.h_out, outs))

    def oracle_step(self, rows):
        import oracle
        oracle.layernorm_fwd(self.host["x"][:rows], self.host["w"], self.host["b"], self.eps, self.dt,
                             residual=self.host["residual"][:rows] if self.fused else None)
        return rows * self.bytes_per_step / self.M


class SmallFwdWorkload(StepWorkload):
    """The fp32 forward on 64 x 1024 rows: 528 KB, resident in L2 unless
    flushed, so L2 is flushed before every step and only the kernel's own
    interval is timed.  Latency-bound: its number is microseconds per call."""
    name = "fwd_f32_64x1024"
    flush_l2 = True

    def __init__(self):
        super().__init__(1, backward=False)


WORKLOADS = {
    "fwd_f32_small": SmallFwdWorkload,
    "dit_mix": DitMixWorkload,
    "adaln": AdalnWorkload,
    "adaln_per_token": lambda: AdalnWorkload(per_token=True),
    "ln_residual": LayerNormWorkload,
    "ln_residual_f32": lambda: LayerNormWorkload("f32", 65536, 1024),
    "ln_plain": lambda: LayerNormWorkload(fused=False),
    "step": lambda: StepWorkload(2, backward=True),
    "fused_fwd": lambda: StepWorkload(2, backward=False),
    "fused_fwd_bwd_residual": lambda: StepWorkload(2, backward=True, dres=True),
    "fwd_bwd_8192": lambda: StepWorkload(4, backward=True),
    "fused_f16_padded": lambda: StepWorkload(5, backward=True),
    "long_rows": lambda: StepWorkload(6, backward=True),
    "odd_rows": lambda: StepWorkload(7, backward=True),
}


# --------------------------------------------------------------------------
# timing
# --------------------------------------------------------------------------

def dist_setup(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return [v]
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


def replay_divisor(K, cap=10):
    """Steps per captured graph: the largest divisor of K not above `cap`."""
    return max(r for r in range(1, min(K, cap) + 1) if K % r == 0)


def capture_steps(torch, calls, R, timed_calls):
    """Capture R steps of `calls` into a CUDA graph.  With `timed_calls`,
    every call is bracketed by timing events recorded as graph nodes (None
    when this torch cannot record events inside a capture)."""
    ev = None
    if timed_calls:
        try:
            ev = [[(torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True)) for _ in calls] for _ in range(R)]
        except TypeError:
            return None
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for r in range(R):
                for j, (_, fn, _) in enumerate(calls):
                    if ev is not None:
                        ev[r][j][0].record()
                    fn()
                    if ev is not None:
                        ev[r][j][1].record()
    torch.cuda.current_stream().wait_stream(side)
    g.replay()                      # one untimed replay
    torch.cuda.synchronize()
    return g, ev, R


def time_calls(torch, calls, stream, n_steps, graph_ok, flush=None):
    """Per-call durations (ms), each call bracketed by CUDA events on the
    launching stream: a graph with event nodes replayed step by step, or
    eager launches (with an L2 flush before every step when `flush`)."""
    samples = [[] for _ in calls]
    cap = capture_steps(torch, calls, 1, True) if (graph_ok and flush is None) else None
    if cap is not None:
        g, ev, _ = cap
        for _ in range(n_steps):
            g.replay()
            torch.cuda.synchronize()
            for j in range(len(calls)):
                samples[j].append(ev[0][j][0].elapsed_time(ev[0][j][1]))
        return samples
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
          for _ in range(n_steps)]
    for k in range(n_steps):
        if flush is not None:
            flush.fill_(k & 0xFF)
        for j, (_, fn, _) in enumerate(calls):
            ev[k][j][0].record(stream)
            fn()
            ev[k][j][1].record(stream)
    torch.cuda.synchronize()
    for k in range(n_steps):
        for j in range(len(calls)):
            samples[j].append(ev[k][j][0].elapsed_time(ev[k][j][1]))
    return samples


def time_isolated(torch, calls, stream, reps=ISOLATED_REPS):
    """Per call label: the average duration of one launch when the label's
    calls run back to back (a CUDA graph of at least ISOLATED_LAUNCHES of
    them, in step order, replayed `reps` times with one pair of events on
    the launching stream around each replay): no timing node sits between
    the launches.  Labels whose calls touch less than twice the L2 capacity
    in all would find their operands in L2 when repeated, and are skipped."""
    out = {}
    for label in dict.fromkeys(c[0] for c in calls):
        group = [c for c in calls if c[0] == label]
        if sum(c[2] for c in group) < 2 * L2_BYTES:
            continue
        seq = [group[i % len(group)] for i in range(max(ISOLATED_LAUNCHES, len(group)))]
        cap = capture_steps(torch, seq, 1, False)
        if cap is None:
            continue
        g = cap[0]
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        out[label] = [a.elapsed_time(b) / len(seq) for a, b in ev]
    return out


def run_e2e(torch, wk, K, world):
    """ms per step end to end: every step copies its inputs from pinned host
    memory, runs the calls through the binding and copies its results back.
    Two device buffer sets and three streams (upload, compute, download) let
    step k's copies overlap step k-1's kernels and each other; events keep a
    set's inputs until its kernels consumed them and its outputs until they
    were copied out."""
    wk.e2e_setup()
    comp, up, down = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    nset = 2
    up_done = [torch.cuda.Event() for _ in range(nset)]
    comp_done = [torch.cuda.Event() for _ in range(nset)]
    down_done = [torch.cuda.Event() for _ in range(nset)]
    calls = [wk.calls(b) for b in range(nset)]
    transfers = [wk.e2e_transfers(b) for b in range(nset)]

    def step(k):
        b = k % nset
        h2d, d2h = transfers[b]
        if k >= nset:
            up.wait_event(comp_done[b])        # set b's inputs were consumed
        with torch.cuda.stream(up):
            for dev, host in h2d:
                dev.copy_(host, non_blocking=True)
            up_done[b].record(up)
        comp.wait_event(up_done[b])
        if k >= nset:
            comp.wait_event(down_done[b])      # set b's results were copied out
        for _, fn, _ in calls[b]:
            fn()
        comp_done[b].record(comp)
        down.wait_event(comp_done[b])
        with torch.cuda.stream(down):
            for host, dev in d2h:
                host.copy_(dev, non_blocking=True)
            down_done[b].record(down)

    k = 0
    for _ in range(2):
        step(k)
        k += 1
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    up.wait_event(e0)
    for _ in range(K):
        step(k)
        k += 1
    comp.wait_event(down_done[(k - 1) % nset])
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / K


def run_native(args):
    import torch
    rank, world, local = dist_setup(args.gpus)
    wk = WORKLOADS[args.workload]().setup()
    calls = wk.calls()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for _, fn, _ in calls:
            fn()
    torch.cuda.synchronize()

    K = args.steps
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if wk.flush_l2 else None
    graph = None
    if args.graph and flush is None:
        graph = capture_steps(torch, calls, replay_divisor(K), False)
    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    flush_ms = 0.0
    if graph is not None:
        # the timed region: a CUDA graph of R steps replayed K / R times, no
        # host work and no timing nodes between the kernels
        g, _, R = graph
        start.record(stream)
        for _ in range(K // R):
            g.replay()
        stop.record(stream)
        torch.cuda.synchronize()
    else:
        fe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        start.record(stream)
        for k in range(K):
            if flush is not None:
                fe[k][0].record(stream)
                flush.fill_(k & 0xFF)
                fe[k][1].record(stream)
            for _, fn, _ in calls:
                fn()
        stop.record(stream)
        torch.cuda.synchronize()
        if flush is not None:   # the L2 flushes are not part of the step
            flush_ms = sum(a.elapsed_time(b) for a, b in fe)
    t1 = time.time()
    # spread: the same work replayed SPREAD_REPS more times right after the
    # timed region, each replay between its own pair of events (clocks are
    # sampled over both)
    spread_ms = []
    if graph is not None:
        g, _, R = graph
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(SPREAD_REPS)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        spread_ms = [a.elapsed_time(b) / R for a, b in ev]
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(SPREAD_REPS)]
        for k, (a, b) in enumerate(ev):
            if flush is not None:
                flush.fill_(k & 0xFF)
            a.record(stream)
            for _, fn, _ in calls:
                fn()
            b.record(stream)
        torch.cuda.synchronize()
        spread_ms = [a.elapsed_time(b) for a, b in ev]
    t2 = time.time()
    barrier(world)
    ms_total = start.elapsed_time(stop) - flush_ms
    # per-kernel durations: a second pass with CUDA events around every call
    n_kernel_steps = max(1, min(K, 200))
    per_call_ms = time_calls(torch, calls, stream, n_kernel_steps, args.graph, flush)
    isolated_ms = time_isolated(torch, calls, stream) if (args.graph and flush is None) else {}

    # end to end with pinned host buffers (fewer steps: host copies dominate)
    Ke = max(3, min(K, 20))
    e2e_ms = run_e2e(torch, wk, Ke, world)

    clock_rows = sampler.stop() if sampler else None
    clocks = None
    if clock_rows is not None:
        clocks = summarize_clocks(clock_rows, t0, t2)
        clocks["window"] = (f"timed region ({(t1 - t0) * 1e3:.1f} ms) and the {SPREAD_REPS}-replay spread pass "
                            f"after it ({(t2 - t1) * 1e3:.1f} ms), nvidia-smi every {sampler.period} ms")
        clocks["samples_in_timed_region"] = sum(1 for r in clock_rows if t0 <= r["t"] <= t1)
    all_ms = max_over_ranks(ms_total / K, world)
    all_e2e = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return None

    agg = aggregate(all_ms, wk.rows_per_step, wk.bytes_per_step)
    agg_e2e = aggregate(all_e2e, wk.rows_per_step, wk.bytes_per_step)
    peak, peak_src = measured_peak()
    kern = {}
    for label in dict.fromkeys(c[0] for c in calls):
        idx = [j for j, c in enumerate(calls) if c[0] == label]
        samples = [t for j in idx for t in per_call_ms[j]]
        nbytes = calls[idx[0]][2]
        avg = sum(samples) / len(samples)
        kern[label] = {"launches_per_step": len(idx), "avg_us": avg * 1e3,
                       "median_us": statistics.median(samples) * 1e3,
                       "gbs": nbytes / (avg / 1e3) / 1e9, "algorithmic_bytes": nbytes,
                       "frac_of_measured_peak": nbytes / (avg / 1e3) / 1e9 / peak,
                       "share_of_step": avg * len(idx) / (ms_total / K)}
        if label in isolated_ms:
            iso = statistics.median(isolated_ms[label])
            kern[label].update(isolated_us=iso * 1e3, isolated_gbs=nbytes / (iso / 1e3) / 1e9,
                               isolated_frac_of_measured_peak=nbytes / (iso / 1e3) / 1e9 / peak)
    dom = max(kern, key=lambda k: kern[k]["share_of_step"])
    traffic = profile_traffic(f"{dom}_{wk.dt}_{wk.M}x{wk.H}")
    # the dominant kernel's duration: back-to-back launches without timing
    # nodes between them when measured, else the in-step event interval (an
    # upper bound: the events add a launch bubble)
    d = kern[dom]
    dom_gbs, dom_how = ((d["isolated_gbs"], f"median over {ISOLATED_REPS} replays of back-to-back launches")
                        if "isolated_gbs" in d else (d["gbs"], "in-step CUDA-event interval (upper bound)"))
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(dom_gbs, 1), "peak": peak,
                "unit": "GB/s", "frac": round(dom_gbs / peak, 4), "peak_source": peak_src,
                "traffic": traffic, "algorithmic_bytes_per_launch": d["algorithmic_bytes"], "duration": dom_how,
                "in_step_event_frac": round(d["frac_of_measured_peak"], 4)}
    line = {
        "metric": METRIC, "value": round(agg["gbs"], 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(agg["ms"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wk.dt, "data": "synthetic (seeded N(0,1) activations, 1+0.1N(0,1) weight)",
        "config": wk.config(), "rows_per_s": round(agg["units_per_s"], 1),
        "pct_of_measured_peak": round(100 * agg["gbs"] / peak, 2),
        "pct_of_nominal_8tbs": round(100 * agg["gbs"] / NOMINAL_HBM_GBS, 2),
        "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                    for k, v in kern.items()},
        "roofline": roofline,
        "e2e": {"value": round(agg_e2e["gbs"], 2), "unit": "GB/s", "h2d_bytes_per_step": wk.h2d,
                "d2h_bytes_per_step": wk.d2h, "ms_per_step": round(agg_e2e["ms"], 4), "steps": Ke,
                "mode": "pinned host buffers; 2 device buffer sets; upload, compute, download streams overlap"},
        "gpu_launches": K * wk.kernels_per_step,
        "launch_mode": (f"CUDA graph of {graph[2]} steps replayed {K // graph[2]} times" if graph is not None
                        else "eager launches"),
        "kernel_timing": (f"{n_kernel_steps} further steps with CUDA events around every call on the launching "
                          "stream (events add a short launch bubble, so per-kernel times are upper bounds); "
                          f"isolated_*: each call label's calls back to back, a graph of at least "
                          f"{ISOLATED_LAUNCHES} launches between one pair of events, median of {ISOLATED_REPS} "
                          "replays (labels whose calls fit twice in L2 are not isolated)"),
        "clocks": clocks,
        "spread": dict(spread_stats(spread_ms), steps_per_rep=(graph[2] if graph is not None else 1),
                       what="per-replay CUDA-event time of the same steps, replayed right after the timed region"),
        "kernel_source_hash": kernel_source_hash(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wk, budget_s=args.cpu_seconds)
    return line


def cpu_baseline(wk, budget_s=10.0, rows=None):
    """The fp64 oracle as it stands, all host cores, on the first `rows` rows
    of the same seeded inputs, repeated for about `budget_s` seconds."""
    import oracle
    rows = rows or min(wk.M, 1024)
    wk.oracle_step(min(rows, 16))  # build + warm
    n_bytes, t0, reps = 0.0, time.perf_counter(), 0
    while True:
        n_bytes += wk.oracle_step(rows)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.default_threads(),
            "kind": "oracle", "rows_per_s": round(reps * rows / dt, 1),
            "sample": f"first {rows} rows of the same seeded workload, fwd+bwd, repeated {reps}x in {dt:.1f}s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    wk = WORKLOADS[args.workload]()
    import oracle
    oracle.build()
    # size the row sample so the whole run stays within about a minute
    probe_rows = 64
    t = time.perf_counter()
    wk.oracle_step(probe_rows)
    per_row = (time.perf_counter() - t) / probe_rows
    total_steps = args.steps + args.warmup
    rows = int(max(8, min(wk.M, 60.0 / max(total_steps, 1) / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        wk.oracle_step(rows)
    t0 = time.perf_counter()
    nbytes = 0.0
    for _ in range(args.steps):
        nbytes += wk.oracle_step(rows)
    dt = time.perf_counter() - t0
    gbs = nbytes / dt / 1e9
    cores = oracle.default_threads()
    sample = f"first {rows} of {wk.M} rows per step, fwd+bwd fp64 oracle"
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wk.dt,
            "data": "synthetic", "config": dict(wk.config(), sample_rows=rows),
            "rows_per_s": round(rows * args.steps / dt, 1),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--record", metavar="PATH",
                    help="also write the JSON line, with the command that made it, to PATH")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        line = run_reference(args)
    else:
        import residual_add_rmsnorm_fwd_gb300 as rn
        rn.lib()  # fail loudly before any work if the library is missing
        line = run_native(args)
    if line is not None:
        print(json.dumps(line), flush=True)
        if args.record:
            argv_used = list(sys.argv[1:] if argv is None else argv)
            if "--record" in argv_used:
                i = argv_used.index("--record")
                del argv_used[i:i + 2]
            argv_used = [a for a in argv_used if not a.startswith("--record=")]
            rec = dict(line, command=" ".join(["python bench.py"] + argv_used))
            with open(args.record, "w") as f:
                f.write(json.dumps(rec) + "\n")


if __name__ == "__main__":
    main()
