"""Benchmark: attention forward + backward at N=8192, D=512, bf16 on GB300.

One step = one pass of the whole hot path on one batch of synthetic input:
ffpa_fwd (O, lse) then ffpa_bwd (dQ, dK, dV) for self-attention with B=1,
Hq=Hkv=8, Nq=Nkv=8192, D=512, bf16, non-causal, scale 1/sqrt(D).  The metric
is attention TFLOPS counted the way the FFPA Attention Benchmark page counts
it ("More Benchmark": forward 2 GEMMs = 4 Nq Nkv D per head, backward the
standard 5 GEMMs = 10 Nq Nkv D per head; the extra GEMM passes an
implementation runs are not counted).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ffpa|reference]

With N > 1 (launched by torch.distributed.run) each rank runs its own batch
(weak scaling: independent problems, no collective on the data path); rank 0
prints one JSON line.  ``--impl reference`` times the CPU fp64 oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

B, H, N, D = 1, 8, 8192, 512
FWD_FLOP = 4 * B * H * N * N * D
BWD_FLOP = 10 * B * H * N * N * D
METRIC = "attention TFLOPS fwd/bwd at N=8192 D=512 bf16, % of GB300 dense peak"
WORKLOAD = "self-attention forward+backward, B=1, Hq=Hkv=8, Nq=Nkv=8192, D=512, bf16, non-causal"
CPU_ROWS = 1024      # cpu_baseline sample: query rows of head 0 against all keys
REF_ROWS = 512       # reference-arm sample per step


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample_step(rows: int):
    """The fp64 oracle on a bounded sample of the workload: head 0, the first
    `rows` query rows against all 8192 keys, forward + backward.  Returns
    (seconds, algorithmic flops of the sample)."""
    import torch

    import oracle.attn_ref as ref

    g = torch.Generator("cpu").manual_seed(0)
    q = torch.randn(1, 1, rows, D, generator=g).to(torch.bfloat16).double().numpy()
    k = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).double().numpy()
    v = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).double().numpy()
    do = torch.randn(1, 1, rows, D, generator=g).to(torch.bfloat16).double().numpy()
    t = time.perf_counter()
    ref.attn_fwd(q, k, v, scale=D ** -0.5)
    ref.attn_bwd(q, k, v, do, scale=D ** -0.5)
    return time.perf_counter() - t, 14 * rows * N * D


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample_step(REF_ROWS)
    secs, flops = 0.0, 0
    for _ in range(args.steps):
        s, f = oracle_sample_step(REF_ROWS)
        secs += s
        flops += f
    value = flops / secs / 1e12
    sample = f"head 0, query rows 0..{REF_ROWS - 1} vs all {N} keys, fwd+bwd in fp64 (numpy), per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD + " (oracle on a bounded sample)",
                                        "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
