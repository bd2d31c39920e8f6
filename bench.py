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

def attention_flops(nq: int, nkv: int, d: int, bh: int, causal: bool = False, backward: bool = False) -> float:
    """FLOP counted for one attention pass, the FFPA Attention Benchmark page's rule
    ("More Benchmark"): forward 2 GEMMs = 4 Nq Nkv D per (batch, query head),
    backward the standard 5 GEMMs = 10 Nq Nkv D; both halved when causal."""
    f = (10 if backward else 4) * nq * nkv * d * bh
    return f / 2 if causal else f


B, H, N, D = 1, 8, 8192, 512
FWD_FLOP = attention_flops(N, N, D, B * H)
BWD_FLOP = attention_flops(N, N, D, B * H, backward=True)
METRIC = "attention TFLOPS fwd/bwd at N=8192 D=512 bf16, % of GB300 dense peak"
WORKLOAD = "self-attention forward+backward, B=1, Hq=Hkv=8, Nq=Nkv=8192, D=512, bf16, non-causal"
CPU_ROWS = 1024      # cpu_baseline probe: query rows of one head against all keys
REF_ROWS = 2048      # reference-arm sample per step


# NVIDIA's nominal dense BF16/FP16 tensor figure for one GB300 (Blackwell
# Ultra) GPU: the HGX B300 platform is quoted at 36 PFLOPS FP16/BF16 with 2:4
# sparsity for eight GPUs, i.e. 4.5 PFLOPS sparse and 2.25 PFLOPS dense per GPU.
PUBLISHED_BF16_DENSE_TFLOPS = 2250.0


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
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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


def oracle_sample_step(rows: int, head: int = 0):
    """The fp64 oracle on a bounded sample of the workload: one head, the first
    `rows` query rows against all 8192 keys, forward + backward.  Returns
    (seconds, algorithmic flops of the sample)."""
    import torch

    import oracle.attn_ref as ref

    g = torch.Generator("cpu").manual_seed(head)
    q = torch.randn(1, 1, rows, D, generator=g).to(torch.bfloat16).double().numpy()
    k = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).double().numpy()
    v = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).double().numpy()
    do = torch.randn(1, 1, rows, D, generator=g).to(torch.bfloat16).double().numpy()
    t = time.perf_counter()
    ref.attn_fwd(q, k, v, scale=D ** -0.5)
    ref.attn_bwd(q, k, v, do, scale=D ** -0.5)
    return time.perf_counter() - t, 14 * rows * N * D


def oracle_time_bounded(budget_s: float = 10.0):
    """Oracle over whole heads of the workload (8192 query rows each) until about
    `budget_s` seconds of CPU work or all 8 heads are done."""
    secs, flop, heads = 0.0, 0, 0
    rows = CPU_ROWS
    while heads < H and secs < budget_s:
        s, f = oracle_sample_step(rows, head=heads)
        secs += s
        flop += f
        heads += 1
        if secs < 1.0 and heads == 1 and rows < N:
            rows = N  # tiny first probe: switch to whole heads
            secs, flop, heads = 0.0, 0, 0
    return secs, flop, heads, rows


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


def run_ffpa(args, rank, world):
    import torch
    import torch.distributed as dist

    from head_dim_attention_gb300 import ffpa_bwd, ffpa_check_status, ffpa_fwd, load
    from head_dim_attention_gb300._lib import ffpa_set_timing_events
    from head_dim_attention_gb300.shard import max_over_ranks
    from head_dim_attention_gb300.synth import make_inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    load()
    peaks = load_peaks()
    scale = 1.0 / math.sqrt(D)
    inp = make_inputs(B, H, H, N, N, D, torch.bfloat16, grad=True, seed=1234 + rank)
    q, k, v, do = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.do))
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    names = ["fwd_main", "bwd_preprocess", "bwd_dkv", "bwd_dq"]

    def step(evs=None):
        if evs:
            ffpa_set_timing_events(evs[0:2])
        ffpa_fwd(q, k, v, None, 0, scale, out, lse)
        if evs:
            ffpa_set_timing_events(evs[2:6])
        ffpa_bwd(q, k, v, None, 0, scale, out, lse, do, dq, dk, dv)
        if evs:
            ffpa_set_timing_events(None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ffpa_check_status() != 0:
        raise RuntimeError("a kernel reported a timeout during warm-up")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for row in evs:
        for e in row:
            e.record()  # torch creates the CUDA event on first record
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0.record()
        for i in range(K):
            step(evs[i])
        t1.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if ffpa_check_status() != 0:
        raise RuntimeError("a kernel reported a timeout in the timed region")
    ms = t0.elapsed_time(t1)
    spans = [(0, 1), (2, 3), (3, 4), (4, 5)]
    kern_ms = {n: statistics.mean(evs[i][a].elapsed_time(evs[i][b]) for i in range(K))
               for n, (a, b) in zip(names, spans)}
    ms = max_over_ranks(ms, dev)  # the slowest rank sets the job's time
    step_flop = FWD_FLOP + BWD_FLOP
    value = world * step_flop * K / (ms / 1e3) / 1e12

    # dominant kernel: the largest share of the step; its own GEMMs as algorithmic work
    # fused dK/dV: S^T, dP^T, dK and dV products (4 x 2 N^2 D per head); dQ: S, dP, dQ
    gemm_flop = {"fwd_main": FWD_FLOP, "bwd_preprocess": 0, "bwd_dkv": 8 * B * H * N * N * D,
                 "bwd_dq": 6 * B * H * N * N * D}
    dom = max(kern_ms, key=kern_ms.get)
    achieved = gemm_flop[dom] / (kern_ms[dom] / 1e3) / 1e12
    # The timed region lasts a fraction of a second at the maximum SM clock:
    # burst conditions, so the burst matmul peak is the denominator; the
    # sustained (power-capped, seconds-long) figure and NVIDIA's nominal dense
    # figure are reported beside it.
    peak = peaks["bf16_tflops"]
    fwd_tf = FWD_FLOP / (kern_ms["fwd_main"] / 1e3) / 1e12
    bwd_tf = BWD_FLOP / (sum(kern_ms[n] for n in names[1:]) / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": TRAFFIC.get(dom),
                "traffic_from": TRAFFIC_FROM if dom in TRAFFIC else None,
                "peak_kind": f"bf16 dense, {peaks['source']} burst (timed region well under a second)",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "frac_of_published": achieved / PUBLISHED_BF16_DENSE_TFLOPS,
                "peaks": {"burst": peaks["bf16_tflops"], "sustained": peaks["bf16_tflops_sustained"],
                          "published_dense": PUBLISHED_BF16_DENSE_TFLOPS},
                "kernel_ms": kern_ms,
                "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
                "fwd_frac": fwd_tf / peak, "bwd_frac": bwd_tf / peak,
                "algorithmic_flop": {n: gemm_flop[n] for n in names}}

    e2e = measure_e2e(inp, scale, world, dev)
    decode = measure_decode(dev, peaks)
    variants = measure_variants(dev, peaks) if rank == 0 else None
    cpu = None
    if rank == 0 and world == 1:
        secs, flop, heads, rows = oracle_time_bounded()
        cpu = {"value": flop / secs / 1e12, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{heads} head(s) x {rows} query rows vs all {N} keys, fwd+bwd in fp64 (numpy); "
                         f"{secs:.1f} s"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "D": D, "causal": False,
                       "parallelism": f"dp{world}: one independent problem per rank, no collective",
                       "l2": "no flush: each step reads Q/K/V/O/dO and writes O/dQ/dK/dV, 512 MiB > 129 MB L2",
                       "frac_of_peak": {"burst": value / world / peaks["bf16_tflops"],
                                        "sustained": value / world / peaks["bf16_tflops_sustained"]}},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": len(names) * K,
            "clocks": clocks.summary(), "decode": decode, "variants": variants,
        }
        print(json.dumps(line), flush=True)


# DRAM bytes (read + write) per launch, dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of the same workload; a kernel
# changed since its capture is left out (its traffic is then reported as null).
TRAFFIC: dict = {"fwd_main": 249217920, "bwd_dkv": 373564672, "bwd_dq": 323346560}
TRAFFIC_FROM = "ncu capture of the same workload (dram__bytes_read.sum + dram__bytes_write.sum per launch)"


def measure_variants(dev, peaks, iters=10, warmup=3):
    """The other configurations of the method at their full sizes, each timed
    alone: median device time of one library call (CUDA events around it) and
    the counted TFLOPS (the same rule as the headline).  Inputs are N(0,1)
    drawn on the device (the values do not change the work)."""
    import torch

    from head_dim_attention_gb300 import ffpa_bwd, ffpa_bwd_dropout, ffpa_fwd, ffpa_fwd_dropout

    g = torch.Generator(device=dev)
    g.manual_seed(11)

    def rnd(*shape, dtype):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(dtype)

    def median_ms(fn):
        for _ in range(warmup):
            fn()
        times = []
        for _ in range(iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            # keep the GPU busy while the host enqueues the call, so that the
            # events bracket the call's device work and not host-side gaps
            torch.cuda._sleep(1000000)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    out_lines = {}

    def case(name, b, hq, hkv, nq, nkv, d, dtype, causal=False, bias=False, backward=False, dropout=0.0):
        q = rnd(b, hq, nq, d, dtype=dtype)
        k, v = rnd(b, hkv, nkv, d, dtype=dtype), rnd(b, hkv, nkv, d, dtype=dtype)
        bb = rnd(1, 1, 1, nkv, dtype=torch.float32) if bias else None
        out, lse = torch.empty_like(q), torch.empty(b, hq, nq, dtype=torch.float32, device=dev)
        sc = d ** -0.5
        if dropout:
            fwd = lambda: ffpa_fwd_dropout(q, k, v, bb, int(causal), sc, dropout, 7, 0, out, lse)  # noqa: E731
        else:
            fwd = lambda: ffpa_fwd(q, k, v, bb, int(causal), sc, out, lse)  # noqa: E731
        ms = median_ms(fwd)
        rec = {"fwd_ms": ms, "fwd_tflops": attention_flops(nq, nkv, d, b * hq, causal) / (ms / 1e3) / 1e12}
        if backward:
            do = rnd(b, hq, nq, d, dtype=dtype)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            fwd()
            if dropout:
                bms = median_ms(lambda: ffpa_bwd_dropout(q, k, v, bb, int(causal), sc, dropout, 7, 0, out, lse, do,
                                                         dq, dk, dv))
            else:
                bms = median_ms(lambda: ffpa_bwd(q, k, v, bb, int(causal), sc, out, lse, do, dq, dk, dv))
            rec["bwd_ms"] = bms
            rec["bwd_tflops"] = attention_flops(nq, nkv, d, b * hq, causal, backward=True) / (bms / 1e3) / 1e12
        for key in [kk for kk in rec if kk.endswith("tflops")]:
            rec[key.replace("tflops", "frac")] = rec[key] / peaks["bf16_tflops"]
        out_lines[name] = rec
        del q, k, v, out, lse

    bf, fp = torch.bfloat16, torch.float16
    case("causal_N8192_D512_bf16", 1, 8, 8, 8192, 8192, 512, bf, causal=True, backward=True)
    case("gqa_Hkv2_N8192_D512_bf16", 1, 8, 2, 8192, 8192, 512, bf, backward=True)
    case("nonaligned_N8191_D512_bf16", 1, 8, 8, 8191, 8191, 512, bf)
    case("cross_Nq1024_Nkv8192_bias_D512_bf16", 1, 8, 8, 1024, 8192, 512, bf, bias=True)
    case("short_Nq64_Nkv8192_D512_bf16", 1, 8, 8, 64, 8192, 512, bf)
    case("dropout_p0.1_N8192_D512_bf16", 1, 8, 8, 8192, 8192, 512, bf, backward=True, dropout=0.1)
    for d in (320, 384, 448, 512, 576, 640, 768, 1024):
        case(f"dsweep_N4096_D{d}_fp16", 1, 8, 8, 4096, 4096, d, fp, backward=True)
    return {"peak": peaks["bf16_tflops"], "timing": "median of 10 calls after 3 warm-up calls, each timed alone "
            "with CUDA events around the call while a spin kernel keeps the GPU busy during the host's enqueue "
            "(device time, host marshalling excluded); TFLOPS counted by the headline's rule (4 / 10 Nq Nkv D "
            "per head, halved when causal)", "cases": out_lines}


def measure_e2e(inp, scale, world, dev, steps=8):
    """The same fwd+bwd step through the public API, fed from pinned host
    memory: every step copies its Q, K, V, dO host->device and its dQ, dK, dV
    device->host inside the timed region.  As in a training or serving
    pipeline, the copies of neighbouring steps overlap this step's kernels:
    two device buffer sets alternate, host->device copies run on one stream and
    device->host copies on another, and a step's compute waits for its inputs
    while a set is reloaded only after its previous results were read back."""
    import torch
    import torch.distributed as dist

    from head_dim_attention_gb300 import ffpa_bwd, ffpa_fwd
    from head_dim_attention_gb300.shard import max_over_ranks

    hosts = [t.pin_memory() for t in (inp.q, inp.k, inp.v, inp.do)]
    sets = []
    for _ in range(2):
        q, k, v, do = (torch.empty(t.shape, dtype=t.dtype, device=dev) for t in hosts)
        sets.append({"in": (q, k, v, do), "out": torch.empty_like(q),
                     "lse": torch.empty(q.shape[:3], dtype=torch.float32, device=dev),
                     "grads": (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))})
    outs = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in sets[0]["grads"]] for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        h2d_done, comp_done, d2h_done = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]

        def load_inputs(i):
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(d2h_done[i - 2])  # set i % 2 read back
                for d, h in zip(sets[i % 2]["in"], hosts):
                    d.copy_(h, non_blocking=True)
                h2d_done[i].record(h2d)

        load_inputs(0)
        for i in range(n):
            st = sets[i % 2]
            q, k, v, do = st["in"]
            comp.wait_event(h2d_done[i])
            ffpa_fwd(q, k, v, None, 0, scale, st["out"], st["lse"])
            ffpa_bwd(q, k, v, None, 0, scale, st["out"], st["lse"], do, *st["grads"])
            comp_done[i].record(comp)
            if i + 1 < n:
                load_inputs(i + 1)
            with torch.cuda.stream(d2h):
                d2h.wait_event(comp_done[i])
                for h, d in zip(outs[i % 2], st["grads"]):
                    h.copy_(d, non_blocking=True)
                d2h_done[i].record(d2h)
        comp.wait_event(d2h_done[n - 1])

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(comp)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    run(steps)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, dev)
    return {"value": world * (FWD_FLOP + BWD_FLOP) / (ms / 1e3) / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hosts),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs[0]),
            "ms_per_step": ms, "steps": steps,
            "overlap": "double-buffered: each step's copies overlap the neighbouring steps' kernels"}


def _call_times(sets, out, lse, ffpa_fwd, iters=10):
    """Wall time of whole decode API calls (host marshalling, scratch
    allocation and launches included), GPU idle before each."""
    import torch

    times = []
    for i in range(iters):
        q, k, v = sets[i % 3]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ffpa_fwd(q, k, v, None, 0, 512 ** -0.5, out, lse)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return times


def measure_decode(dev, peaks, iters=21):
    """Decode-shaped forward (Nq=1, Nkv=8192, H=8, D=512, bf16): HBM-bound.
    Every call reads K and V that are not resident in L2: three separate input
    sets of 134 MB are used in turn (inputs larger than L2), so no flush write
    leaves dirty lines for the call to write back.  For comparison the same
    calls are also timed after a 256 MiB flush write (dirty L2).  The GB/s
    figures use the device time of the call's launches (events around the
    call, with the GPU kept busy while the host enqueues it); a second pass
    with the library's timing hook splits off the split kernel's share.
    `call_us` is the whole API call, host marshalling and scratch allocation
    included, on an idle GPU."""
    import torch

    from head_dim_attention_gb300 import ffpa_fwd
    from head_dim_attention_gb300._lib import ffpa_set_timing_events
    from head_dim_attention_gb300.synth import make_inputs

    inp = make_inputs(1, 8, 8, 1, 8192, 512, torch.bfloat16, seed=7)
    sets = [tuple(t.to(dev).clone() for t in (inp.q, inp.k, inp.v)) for _ in range(3)]
    out = torch.empty_like(sets[0][0])
    lse = torch.empty(1, 8, 1, dtype=torch.float32, device=dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    hook = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in hook:
        e.record()  # the hook needs events that exist on the device

    def timed(dirty, breakdown):
        """Median device time of the call's launches.  The GPU is kept busy
        (a spin kernel) while the host enqueues the call, so the events
        bracket GPU work, not host-side gaps.  Without `breakdown` the events
        sit outside the call, so the two launches stay adjacent on the stream
        (the second is a programmatic dependent of the first); with it, the
        library's timing hook adds an event between them to split the time."""
        kern, split = [], []
        for i in range(iters + 3):
            q, k, v = sets[i % 3]
            if dirty:
                flush.fill_(float(i))
            torch.cuda._sleep(1000000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            if breakdown:
                ffpa_set_timing_events(hook)
            ffpa_fwd(q, k, v, None, 0, 512 ** -0.5, out, lse)
            if breakdown:
                ffpa_set_timing_events(None)
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                kern.append(e0.elapsed_time(e1))
                if breakdown:
                    split.append(hook[0].elapsed_time(hook[1]))
        return statistics.median(kern), (statistics.median(split) if breakdown else None)

    ms, _ = timed(False, False)
    ms_hooked, split_ms = timed(False, True)
    ms_dirty, _ = timed(True, False)
    call_ms = statistics.median(_call_times(sets, out, lse, ffpa_fwd))
    q, k, v = sets[0]
    nbytes = sum(t.numel() * t.element_size() for t in (q, k, v, out))
    gbs = nbytes / (ms / 1e3) / 1e9

    # GQA decode, Hq = 8 on Hkv = 2: one CTA per (slice, kv head) scores the
    # group's four query heads, so the K/V bytes required are those of two kv
    # heads (33.5 MB); five input sets in turn keep each call's K/V out of L2
    ginp = make_inputs(1, 8, 2, 1, 8192, 512, torch.bfloat16, seed=8)
    gsets = [tuple(t.to(dev).clone() for t in (ginp.q, ginp.k, ginp.v)) for _ in range(5)]
    gms = []
    for i in range(iters + 5):
        gq, gk, gv = gsets[i % 5]
        torch.cuda._sleep(1000000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ffpa_fwd(gq, gk, gv, None, 0, 512 ** -0.5, out, lse)
        e1.record()
        torch.cuda.synchronize()
        if i >= 5:
            gms.append(e0.elapsed_time(e1))
    gms = statistics.median(gms)
    gq, gk, gv = gsets[0]
    gbytes = sum(t.numel() * t.element_size() for t in (gq, gk, gv, out))
    ggbs = gbytes / (gms / 1e3) / 1e9
    gqa = {"workload": "decode Nq=1, Nkv=8192, Hq=8, Hkv=2, D=512, bf16", "us": gms * 1e3, "bytes": gbytes,
           "gbps": ggbs, "frac_of_hbm": ggbs / peaks["hbm_gbs"],
           "bytes_one_read_per_query_head": sum(t.numel() * t.element_size() for t in (gq, out)) + 4 * (
               gk.numel() + gv.numel()) * gk.element_size(),
           "l2": "cold: five 33.5 MB K/V sets used in turn"}
    return {"workload": "decode Nq=1, Nkv=8192, H=8, D=512, bf16", "us": ms * 1e3, "bytes": nbytes, "gqa": gqa,
            "gbps": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"], "split_us": split_ms * 1e3,
            "combine_us_with_event_between": (ms_hooked - split_ms) * 1e3, "call_us": call_ms * 1e3,
            "l2": "cold: three 134 MB input sets used in turn (no flush writes)",
            "us_after_dirty_flush": ms_dirty * 1e3, "gbps_after_dirty_flush": nbytes / (ms_dirty / 1e3) / 1e9,
            "timing": "device time of the call's split + combine launches (events around the call, GPU busy "
                      "while it is enqueued); split_us from the library's timing hook in a second pass"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ffpa", "reference"], default="ffpa")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist

    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        run_ffpa(args, rank, world)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
