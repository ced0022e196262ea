#!/usr/bin/env python
"""Benchmark of the FP4 communication codec's hot path on GB300.

One step = one emulated R-rank compressed AllReduce of a tensor-parallel activation
(workload: two [4096, 4096] bfloat16 partial sums drawn like the 4096 x 4096 TP activation
of a 7B-class model, seeds 0 and 1): compress each rank's partial, fused
decompress-sum-requantize of the R payloads, then decompress-accumulate the reduced payload
into a bfloat16 residual stream. Every kernel of the path runs once per step (R compresses,
one reduce, one decompress-accumulate).

Metric: GB/s of BF16 input (R * 2n bytes per step / step time), with each kernel's
achieved algorithmic bandwidth against the measured HBM copy peak. The step time comes from
CUDA events at step boundaries only (the kernels launch with programmatic stream
serialisation, and an event between two kernels would stop that overlap); the per-kernel
durations come from a second pass of the same steps with an event between kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica on its own GPU (weak scaling; the
codec has no data-path collective), the timed region is bracketed by barriers and the
slowest rank's time is reported. --impl reference times the CPU oracle (the plain scalar
restatement used by the tests) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

R_RANKS = 2
TOKENS, HIDDEN = 4096, 4096
GROUP, FWHT = 16, 1
WORKLOAD = "tp_activation_4096x4096_allreduce_r2"
METRIC = "compress / decompress-accumulate GB/s of BF16 input"
UNIT = "GB/s"
L2_FLUSH_BYTES = 512 << 20

# algorithmic bytes per element (G = 16): what each kernel must move at minimum
ALG_BYTES = {
    "compress": 2 + 0.5 + 1 / 16 + 4 / 256,
    "reduce": (R_RANKS + 1) * (0.5 + 1 / 16 + 4 / 256),
    "decompress_accumulate": 0.5 + 1 / 16 + 4 / 256 + 4,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: torch copy)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


def kernel_source_sha() -> str:
    """Hash of the code the kernels are built from (csrc/*.cu, csrc/*.cuh, include/fp4q.h),
    with comments and blank lines removed, so that editing a comment does not orphan the
    ncu summaries taken on the same code."""
    csrc = os.path.join(ROOT, "fp4_communication_compression_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh")))
    h = hashlib.sha256()
    for f in files + [os.path.join(ROOT, "include", "fp4q.h")]:
        text = open(f).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or None when the
    summary is missing or was taken on a different kernel source."""
    sha = kernel_source_sha()
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))) if os.path.isdir(os.path.join(ROOT, "profiles")) else []:
        if not name.endswith(".md"):
            continue
        text = open(os.path.join(ROOT, "profiles", name)).read()
        m = re.search(r"bench-traffic kernel=(\w+) source_sha256=(\w+) dram_bytes_per_launch=(\d+)", text)
        if m and m.group(1) == kernel and m.group(2) == sha:
            return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed loop runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.5)
        return self

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}

    def __exit__(self, *exc):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (the slowest rank's time)."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time (GB/s)."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


def make_inputs():
    from fp4_communication_compression_gb300 import inputs
    xs = [inputs.tp_activation(seed=r, tokens=TOKENS, hidden=HIDDEN) for r in range(R_RANKS)]
    resid = inputs.tp_activation(seed=100, tokens=TOKENS, hidden=HIDDEN)
    return xs, resid


# ------------------------------------------------------------------ CPU oracle timing

def oracle_step(xs, resid):
    import oracle
    n = xs[0].size
    pays = [oracle.compress(x.ravel(), GROUP, FWHT) for x in xs]
    red = oracle.reduce_requantize(pays, n, GROUP)
    return oracle.decompress_accumulate(red, n, resid.ravel().copy(), beta=1, group=GROUP, fwht=FWHT)


def time_oracle(xs, resid, min_seconds=10.0, max_reps=50):
    import oracle
    oracle.set_threads(os.cpu_count() or 1)
    cores = oracle.max_threads()
    n = xs[0].size
    oracle_step(xs, resid)                         # build + warm
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_step(xs, resid)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    gbs = R_RANKS * 2 * n * reps / el / 1e9
    return {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} full steps of {WORKLOAD} ({R_RANKS} x {TOKENS}x{HIDDEN} bf16), "
                      f"{el:.1f} s wall, OpenMP over 256-element blocks"}


def reference_arm(args, rank, world):
    """CPU oracle as the reference implementation: same workload, metric and unit."""
    if rank != 0:
        return 0
    xs, resid = make_inputs()
    import oracle
    oracle.set_threads(os.cpu_count() or 1)
    cores = oracle.max_threads()
    n = xs[0].size
    for _ in range(max(args.warmup, 0)):
        oracle_step(xs, resid)
    # each timed step is the full workload; keep the run to a few minutes
    steps = max(1, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(xs, resid)
    el = time.perf_counter() - t0
    v = R_RANKS * 2 * n * steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "ranks": R_RANKS, "shape": [TOKENS, HIDDEN], "group": GROUP,
                       "block": 256, "fwht": FWHT},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{steps} full step{'s' if steps > 1 else ''} of {WORKLOAD}" + (
                                 f" (the requested {args.steps} capped at 20)" if args.steps > steps else "")},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import numpy as np
    import torch

    import fp4_communication_compression_gb300 as fq
    from fp4_communication_compression_gb300 import inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    fq.build()

    xs_np, resid_np = make_inputs()
    n = xs_np[0].size
    xs = [inputs.bits_to_torch(x.ravel(), dev) for x in xs_np]
    resid = inputs.bits_to_torch(resid_np.ravel(), dev)
    dst = resid.clone()
    pb = fq.payload_bytes(n, GROUP, FWHT)
    pays = [torch.empty(pb, dtype=torch.uint8, device=dev) for _ in range(R_RANKS)]
    red = torch.empty(pb, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the reads evict the dirty
        # lines, so their write-back is not charged to the next timed kernel
        flush.zero_()
        clean.sum()
    stream = torch.cuda.current_stream(dev)
    names = ["compress"] * R_RANKS + ["reduce", "decompress_accumulate"]

    def step(ev=None):
        # ev: None, [start, end] (step boundaries only) or one event before each kernel plus
        # one at the end (per-kernel durations; the extra records keep each kernel from
        # overlapping its launch with the previous kernel's tail)
        each = ev is not None and len(ev) > 2
        if ev is not None:
            ev[0].record(stream)
        for r in range(R_RANKS):
            fq.compress(xs[r], payload=pays[r], group=GROUP, fwht=FWHT, stream=stream)
            if each:
                ev[1 + r].record(stream)
        fq.reduce_requantize(pays, n, out=red, group=GROUP, fwht=FWHT, stream=stream)
        if each:
            ev[1 + R_RANKS].record(stream)
        fq.decompress_accumulate(red, n, dst, beta=1, group=GROUP, fwht=FWHT, stream=stream)
        if ev is not None:
            ev[-1].record(stream)

    # correctness / error report on fresh buffers (not timed)
    step()
    torch.cuda.synchronize(dev)
    ref = sum(inputs.bf16_bits_to_f32(x.ravel()).astype(np.float64) for x in xs_np) + \
        inputs.bf16_bits_to_f32(resid_np.ravel()).astype(np.float64)
    first_bits = inputs.torch_to_bits(dst)          # one step's result from the residual
    got = inputs.bf16_bits_to_f32(first_bits).astype(np.float64)
    delta = ref - inputs.bf16_bits_to_f32(resid_np.ravel()).astype(np.float64)
    rel_l2 = float(np.linalg.norm(got - ref) / np.linalg.norm(delta))

    for _ in range(args.warmup):
        flush_l2()
        step()
    def new_events(count):
        return [[torch.cuda.Event(enable_timing=True) for _ in range(count)] for _ in range(args.steps)]
    events = new_events(2)
    with ClockSampler(dev.index) as clk:
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for k in range(args.steps):
            flush_l2()                        # evict the step's working set from L2 (not timed)
            step(events[k])
        torch.cuda.synchronize(dev)
        t1 = time.time()
        if pg:
            pg.barrier()
        clocks = clk.stop(t0, t1)
        # kernel pass: the same K steps again with an event between kernels, for the
        # per-kernel durations behind "kernels" and "roofline" (not part of "value")
        kevents = new_events(1 + len(names))
        torch.cuda.synchronize(dev)
        for k in range(args.steps):
            flush_l2()
            step(kevents[k])
        torch.cuda.synchronize(dev)
    per_kernel = {name: [] for name in set(names)}
    step_ms = [ev[0].elapsed_time(ev[-1]) for ev in events]
    for ev in kevents:
        for i, name in enumerate(names):
            per_kernel[name].append(ev[i].elapsed_time(ev[i + 1]))
    dev_ms = float(sum(step_ms))
    if pg:
        dev_ms = max_over_ranks(dev_ms, pg, dev)
    ms_per_step = dev_ms / args.steps
    bytes_in = R_RANKS * 2 * n
    value = job_gbs(bytes_in, args.steps, world, dev_ms)

    peak, peak_src = measured_peak()
    kern = {}
    for name, ts in per_kernel.items():
        mean_ms = statistics.fmean(ts)
        ach = ALG_BYTES[name] * n / (mean_ms * 1e-3) / 1e9
        kern[name] = {"ms": round(mean_ms, 5), "launches_per_step": names.count(name),
                      "alg_gbs": round(ach, 1), "frac_of_peak": round(ach / peak, 4),
                      "bf16_in_gbs": round((R_RANKS if name == "reduce" else 1) * 2 * n / (mean_ms * 1e-3) / 1e9, 1)}
    dom = max(kern, key=lambda k: kern[k]["ms"] * kern[k]["launches_per_step"])
    traffic = ncu_traffic({"compress": "compress_kernel", "reduce": "reduce_kernel",
                           "decompress_accumulate": "decompress_kernel"}[dom])

    # end to end through the public API: pinned host inputs in, result back to the host.
    # Every step copies its own inputs in and reads its own result back inside the timed
    # region; the copies of step k + 1 run on a copy stream while step k computes (two sets
    # of input / result buffers), and the read-back runs on a third stream.
    hx = [inputs.bits_to_torch(x.ravel()).pin_memory() for x in xs_np]
    hres = inputs.bits_to_torch(resid_np.ravel()).pin_memory()
    hout = torch.empty_like(hres).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    sets = [([torch.empty_like(x) for x in xs], torch.empty_like(dst)) for _ in range(2)]
    s_in, s_back = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e(steps):
        ev = lambda: torch.cuda.Event()                   # noqa: E731
        ins, dones, backs = [], [], []
        for k in range(steps):
            sx, sd = sets[k % 2]
            with torch.cuda.stream(s_in):
                if k >= 2:                                # the set is free once step k-2 is read back
                    s_in.wait_event(backs[k - 2])
                for r in range(R_RANKS):
                    sx[r].copy_(hx[r], non_blocking=True)
                sd.copy_(hres, non_blocking=True)
                ins.append(ev())
                ins[-1].record(s_in)
            stream.wait_event(ins[k])
            for r in range(R_RANKS):
                fq.compress(sx[r], payload=pays[r], group=GROUP, fwht=FWHT, stream=stream)
            fq.reduce_requantize(pays, n, out=red, group=GROUP, fwht=FWHT, stream=stream)
            fq.decompress_accumulate(red, n, sd, beta=1, group=GROUP, fwht=FWHT, stream=stream)
            dones.append(ev())
            dones[-1].record(stream)
            with torch.cuda.stream(s_back):
                s_back.wait_event(dones[k])
                hout.copy_(sd, non_blocking=True)
                backs.append(ev())
                backs[-1].record(s_back)
        return backs[-1]

    e2e(2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    last = e2e(e2e_steps)
    s_back.wait_event(last)
    e1.record(s_back)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    assert np.array_equal(inputs.torch_to_bits(hout), first_bits), "end-to-end result differs from the device step"
    h2d = (R_RANKS + 1) * 2 * n
    d2h = 2 * n

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "ranks": R_RANKS, "shape": [TOKENS, HIDDEN], "group": GROUP,
                   "block": 256, "fwht": FWHT, "parallelism": f"replicas x{world}",
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write + {L2_FLUSH_BYTES >> 20} MiB read, outside the step events)"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": kern[dom]["alg_gbs"], "peak": peak,
                     "unit": "GB/s", "frac": kern[dom]["frac_of_peak"], "traffic": traffic,
                     "peak_source": peak_src,
                     "alg_bytes_per_elem": round(ALG_BYTES[dom], 6), "elems_per_launch": n},
        "kernels": kern,
        "kernels_timing": "second pass of the K steps with a CUDA event between kernels; the events "
                          "stop each kernel's launch from overlapping the previous kernel's tail, so "
                          "these durations add up to more than ms_per_step",
        "rel_l2_error": round(rel_l2, 6),
        "gpu_launches": len(names) * args.steps,
        "clocks": clocks,
        "e2e": {"value": round(world * bytes_in / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "wall_ms_timed_region": round((t1 - t0) * 1e3, 2),
        "kernel_source_sha256": kernel_source_sha(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(xs_np, resid_np)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
