"""Benchmark of the latent-MoE output tail on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|stress|tiny|decode_T1|...]

A step is one call of the whole tail (routed reduce + RMSNorm, up-projection,
shared-partial epilogue) on one batch of synthetic inputs. The default workload
is the largest benchmark configuration, the stress workload (P=16, T=16384,
L=2048, H=7168, 1% of rows x100 and 1% x1e-3). Inputs rotate over enough seeded
sets that their total exceeds twice the L2 size, so every step streams W and the
partials from HBM. Steps are replayed from CUDA graphs and timed with CUDA
events on the launching stream, between a barrier and a device synchronize on
both sides; a timed region holds exactly K steps and is repeated (about one
second of timed work in all, so the clock samples come from inside the regions),
and the median region is reported. With N > 1 each rank runs its own replica
(token batches are independent, no collective) and the max time over ranks is
used.

The line also carries, under "workloads", µs/call, tokens/s, the roofline of
the dominant kernel and the single-call latency of every other benchmark
configuration (decode P8 T16, the decode sweep T = 1, 2, 4, 8, 32, 64, 128, prefill P8 T8192 and
the pre-reduced P=1 prefill).

`single_call_us_median` is the median device time of one call with nothing else
on the GPU before or after it (an eager call enqueued behind a spin kernel): the
latency a single call sees, without the overlap between consecutive calls.

The `e2e` figure times the same steps through the host-buffer entry point
(latent_tail_forward_host): each step's partials start in page-locked host
memory and its result ends there, inside the timed region. Next to it,
`staged_copies_us_per_step` times explicit pinned-host <-> device copies around
the device entry point.

Prints one JSON line. `--impl reference` times the CPU oracle instead (the
only other code path this file may run), on a bounded sample of the same
workload. `--capture w1,w2@T,...` prints no JSON: it runs one forward call per
listed workload and nothing else, the launch list that one ncu pass captures
for the per-workload DRAM traffic figures.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024  # replaced by the device's value at run time


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="stress")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other benchmark configurations (the 'workloads' record)")
    ap.add_argument("--repeats", type=int, default=0,
                    help="timed regions of K steps (0: enough for about one second)")
    ap.add_argument("--T", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps")
    ap.add_argument("--shards", type=int, default=0,
                    help="also time each step as N column-range calls covering [0, H)")
    ap.add_argument("--capture", default="",
                    help="comma-separated workloads (name or name@T): run one forward call "
                         "of each, in order, and nothing else (a launch list for ncu)")
    return ap.parse_args()


def capture_calls(spec):
    """One forward call per listed workload, inputs resident in HBM, synchronized
    after each: under ncu each kernel of the list is captured once, in order."""
    import dataclasses

    import torch

    from latent_moe_output_gb300 import binding, inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load_library()
    for item in spec.split(","):
        name, _, t = item.partition("@")
        w = workload(name)
        if t:
            w = dataclasses.replace(w, name=f"{w.name}_T{int(t)}", T=int(t))
        x = inputs.make_workload(w, device=dev)
        out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(binding.latent_tail_workspace_size(w.P, w.T, w.L, w.H), 256),
                         dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev)
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws, stream)
        binding.latent_tail_check(stream)
        print(f"captured call: workload {w.name}, P {w.P}, T {w.T}, L {w.L}, H {w.H}", flush=True)
        del x, out, ws


def workload(name):
    from latent_moe_output_gb300 import inputs

    if name not in inputs.WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(inputs.WORKLOADS)}")
    return inputs.WORKLOADS[name]


def call_bytes(P, T, L, width):
    """Algorithmic bytes of one call: routed + shared columns + W rows + out + g."""
    return P * T * L * 2 + P * T * width * 2 + width * L * 2 + T * width * 2 + L * 4


def project_bytes(P, T, L, width):
    """Algorithmic bytes of the up-projection kernel alone: latent y + shared
    columns + W rows + out."""
    return T * L * 2 + P * T * width * 2 + width * L * 2 + T * width * 2


def flops(T, L, width):
    return 2 * T * width * L


# Largest token count the decode kernel serves at the bench's widths (L = 2048).
DECODE_TOKENS = 224


def profiled_traffic(kernel, workload_name, T):
    """DRAM bytes per launch of `kernel` (dram__bytes_read.sum + dram__bytes_write.sum)
    from the ncu summary committed under profiles/, or None when no capture matches
    this workload and token count, or the kernel's source changed since the capture
    (its sha256 is recorded next to the figure)."""
    import glob
    import hashlib
    import re

    src = os.path.join(ROOT, "latent_moe_output_gb300", "csrc", kernel.replace("_kernel", "") + ".cu")
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    pat = re.compile(r"^traffic_per_launch_bytes: (\d+) \(workload (\w+), T (\d+), "
                     r"(\S+) sha256 ([0-9a-f]{16})\)", re.M)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", kernel + "_*.md"))):
        with open(path) as f:
            for m in pat.finditer(f.read()):
                if (m.group(2) == workload_name and int(m.group(3)) == T
                        and m.group(4) == os.path.basename(src) and m.group(5) == digest):
                    return int(m.group(1))
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region.

    The sampler is started, and its first sample awaited, before the region
    opens, so nvidia-smi's start-up does not eat into it. A region shorter than a
    few sampling periods also takes the samples of the next 0.2 s (said so in
    the summary)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.t_open = self.t_close = 0.0

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append((time.perf_counter(), line))

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            deadline = time.perf_counter() + 5.0
            while not self.lines and time.perf_counter() < deadline:
                time.sleep(0.005)
        self.t_open = time.perf_counter()
        return self

    def __exit__(self, *exc):
        self.t_close = time.perf_counter()
        if self.proc is None:
            return
        deadline = self.t_close + 0.2
        while (time.perf_counter() < deadline
               and sum(1 for t, _ in self.lines if t >= self.t_open) < 3):
            time.sleep(0.005)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.reader.join(timeout=5)

    def summary(self):
        inside = [l for t, l in self.lines if self.t_open <= t <= self.t_close + 0.03]
        window = "timed region"
        if len(inside) < 3:
            inside = [l for t, l in self.lines if t >= self.t_open][:3]
            window = "timed region and up to 0.2 s after it (region shorter than 3 samples)"
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in inside:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v, world, device="cuda"):
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step, steps, world, seconds):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / seconds


def host_cpu_model():
    """The host CPU's model name (Linux /proc/cpuinfo, else the platform string)."""
    import platform

    part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip() in ("model name", "Model name") and val.strip():
                    return val.strip()
                if key.strip() == "CPU part" and val.strip():
                    part = val.strip()
    except OSError:
        pass
    if part:  # Arm: no model name, only the part number (0xd4f is Neoverse V2)
        return f"{platform.machine()} CPU part {part}"
    return platform.processor() or platform.machine()


def cpu_baseline(w, budget_s=12.0, max_tokens=None):
    """The oracle as it stands, single-threaded, on a bounded sample of tokens
    of the same workload (drawn on the CPU with the workload's seed)."""
    import numpy as np

    import oracle
    from latent_moe_output_gb300 import inputs

    lib = oracle.load()
    tokens = w.T if max_tokens is None else min(w.T, max_tokens)
    x = inputs.make(w.P, tokens, w.L, w.H, w.seed, device="cpu", outliers=w.outlier_rows)
    done, t0 = 0, time.perf_counter()
    # one token first to size the sample
    oracle.forward(x.routed[:, :1], x.shared[:, :1], x.g, x.W, x.eps, lib=lib)
    per_tok = time.perf_counter() - t0
    n = int(max(1, min(tokens, budget_s / max(per_tok, 1e-9))))
    # repeat the n-token call until about budget_s of CPU work has been timed
    reps, dt = 0, 0.0
    while reps == 0 or dt < 0.8 * budget_s:
        t0 = time.perf_counter()
        oracle.forward(x.routed[:, :n], x.shared[:, :n], x.g, x.W, x.eps, lib=lib)
        dt += time.perf_counter() - t0
        reps += 1
    done = n * reps
    return {"value": done / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} call(s) of {n} of the {w.T} tokens of the {w.name} workload "
                      f"(P={w.P}, L={w.L}, H={w.H}), FP32 single-threaded, {dt:.2f} s",
            "host_cores": os.cpu_count(), "host_cpu": host_cpu_model()}


def reference_arm(args):
    """CPU oracle as the reference arm: K timed steps, each a bounded token sample."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from latent_moe_output_gb300 import inputs

    w = workload(args.workload)
    lib = oracle.load()
    steps = max(1, args.steps)
    total = steps + max(0, args.warmup)
    x1 = inputs.make(w.P, 1, w.L, w.H, w.seed, device="cpu", outliers=w.outlier_rows)
    t0 = time.perf_counter()
    oracle.forward(x1.routed, x1.shared, x1.g, x1.W, x1.eps, lib=lib)
    per_tok = time.perf_counter() - t0
    per_step_budget = 120.0 / total
    # at most 2048 tokens per step, so that the sample's inputs stay small on the host
    n = int(max(1, min(w.T, 2048, per_step_budget / max(per_tok, 1e-9))))
    # When even one token per step exceeds the budget (many steps), a step is one
    # token over the first `width` output columns and counts as width/H of a
    # token: the oracle's time per token is proportional to the columns it
    # computes (the norm of one token is ~1/H of its projection).
    width = w.H
    if per_tok > per_step_budget:
        width = max(8, min(w.H, int(w.H * per_step_budget / per_tok) // 8 * 8))
    x = inputs.make(w.P, n, w.L, w.H, w.seed, device="cpu", outliers=w.outlier_rows)
    for _ in range(max(0, args.warmup)):
        oracle.forward(x.routed, x.shared, x.g, x.W, x.eps, 0, width, lib=lib)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.forward(x.routed, x.shared, x.g, x.W, x.eps, 0, width, lib=lib)
    dt = time.perf_counter() - t0
    value = n * (width / w.H) * steps / dt
    line = {
        "impl": "reference", "metric": "latent-tail tokens/s", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "P": w.P, "T": w.T, "L": w.L, "H": w.H,
                   "sample_tokens_per_step": n, "sample_columns_per_step": width},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle", "cores": 1,
                         "sample": f"{n} of {w.T} tokens x {width} of {w.H} columns per "
                                   f"step (counted as {n * width / w.H:.4g} tokens)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# The other benchmark configurations, measured after the headline workload and
# reported under "workloads" in the same line.
SUB_WORKLOADS = ("decode", "decode_T1", "decode_T2", "decode_T4", "decode_T8", "decode_T32", "decode_T64",
                 "decode_T128", "prefill", "prefill_p1")


def roofline_of(w, us_proj, us_call, hbm, tc_burst, peak_kind):
    """Roofline of the dominant (projection) kernel and of the whole call. The
    binding roofline is HBM unless the kernel's flops take longer at the tensor
    peak than its bytes at the HBM peak (the P = 1 prefill)."""
    P, T, L, H = w.P, w.T, w.L, w.H
    pb, cb, fl = project_bytes(P, T, L, H), call_bytes(P, T, L, H), flops(T, L, H)
    # Which kernel a call runs at the bench's widths (L = 2048, H = 7168): T <= 2
    # the one-launch CUDA-core kernel (one SM's W slice fits in shared memory),
    # up to 224 tokens the split-K decode kernel, above it the prefill kernel.
    kname = "gemv_kernel" if T <= 2 else "decode_kernel" if T <= DECODE_TOKENS else "prefill_kernel"
    proj_gbs = pb / (us_proj * 1e-6) / 1e9
    if fl / (tc_burst * 1e12) > pb / (hbm * 1e9):
        proj_tf = fl / (us_proj * 1e-6) / 1e12
        roof = {"kernel": kname, "bound": "tensor", "achieved": round(proj_tf, 1),
                "peak": tc_burst, "unit": "TFLOP/s", "frac": round(proj_tf / tc_burst, 4),
                "traffic": profiled_traffic(kname, w.name, T), "algorithmic_bytes_per_launch": pb,
                "algorithmic_flops_per_launch": fl,
                "us_per_launch": round(us_proj, 3), "peak_source": peak_kind}
    else:
        roof = {"kernel": kname, "bound": "hbm", "achieved": round(proj_gbs, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(proj_gbs / hbm, 4),
                "traffic": profiled_traffic(kname, w.name, T),
                "algorithmic_bytes_per_launch": pb, "us_per_launch": round(us_proj, 3),
                "peak_source": peak_kind}
    call_gbs = cb / (us_call * 1e-6) / 1e9
    call_roof = {"achieved": round(call_gbs, 1), "peak": hbm, "unit": "GB/s",
                 "frac": round(call_gbs / hbm, 4), "algorithmic_bytes_per_call": cb,
                 "tensor_tflops": round(fl / (us_call * 1e-6) / 1e12, 2),
                 "tensor_frac_of_burst_peak": round(fl / (us_call * 1e-6) / 1e12 / tc_burst, 4)}
    return roof, call_roof


class Bench:
    """Timing of one workload: rotating input sets resident in HBM, steps replayed
    from CUDA graphs, CUDA events on the launching stream."""

    def __init__(self, w, args, dev, rank, world):
        import torch

        from latent_moe_output_gb300 import binding, inputs

        self.torch, self.binding, self.inputs = torch, binding, inputs
        self.w, self.args, self.dev, self.rank, self.world = w, args, dev, rank, world
        P, T, L, H = w.P, w.T, w.L, w.H
        props = torch.cuda.get_device_properties(dev)
        self.l2 = getattr(props, "L2_cache_size", L2_BYTES) or L2_BYTES
        binding.load_library()
        self.ws_bytes = binding.latent_tail_workspace_size(P, T, L, H)
        self.set_bytes = call_bytes(P, T, L, H) + self.ws_bytes
        # enough sets that their total exceeds twice L2: every step reads from HBM
        self.n_sets = max(2, -(-2 * self.l2 // self.set_bytes) + 1)
        self.sets = []
        for r in range(self.n_sets):
            x = inputs.make(P, T, L, H, w.seed + 7919 * r + 104729 * rank, device=dev,
                            outliers=w.outlier_rows)
            out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
            ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
            self.sets.append((x, out, ws))
        self.stream = torch.cuda.Stream(device=dev)

    def step(self, i):
        x, out, ws = self.sets[i % self.n_sets]
        self.binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws,
                                         self.stream)

    def project_only(self, i):
        T, L, H = self.w.T, self.w.L, self.w.H
        x, out, ws = self.sets[i % self.n_sets]
        y = ws[:T * L * 2].view(self.torch.bfloat16).view(T, L)
        self.binding.latent_tail_project_cols(y, x.shared, x.W, out, 0, H, self.stream)

    def warm(self, n):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for i in range(max(3, n)):
                self.step(i)
        self.binding.latent_tail_check(self.stream)
        # rough per-call time, to size the timed regions of the extra workloads
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for i in range(5):
                self.step(i)
            e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3 / 5

    def timed(self, fn, steps, repeats):
        """Seconds of each of `repeats` timed regions of exactly `steps` steps,
        each region bracketed by a barrier and a device synchronize."""
        torch = self.torch
        chunk = min(steps, 50 * self.n_sets)
        graphs, plan, left = {}, [], steps
        while left > 0:
            n = min(chunk, left)
            if n not in graphs:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(self.stream):
                    with torch.cuda.graph(g, stream=self.stream):
                        for i in range(n):
                            fn(i)
                graphs[n] = g
            plan.append(graphs[n])
            left -= n
        self.graph_calls = chunk
        out = []
        # CUDAGraph.replay() launches on the current stream: make it the stream the
        # events are recorded on.
        with torch.cuda.stream(self.stream):
            for g in graphs.values():  # untimed replay: settle clocks and caches
                g.replay()
            self.stream.synchronize()
            for _ in range(repeats):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                barrier(self.world)
                torch.cuda.synchronize(self.dev)
                e0.record(self.stream)
                for g in plan:
                    g.replay()
                e1.record(self.stream)
                torch.cuda.synchronize(self.dev)
                barrier(self.world)
                out.append(e0.elapsed_time(e1) / 1e3)
        return out

    def single_call_us(self, n):
        """Median device time of one call with nothing else on the GPU before or
        after it: a spin kernel keeps the GPU busy while the events and the call's
        launches are enqueued, so the interval holds only the call's own time."""
        torch = self.torch
        single = []
        with torch.cuda.stream(self.stream):
            for i in range(self.n_sets + n):
                torch.cuda._sleep(200000)  # ~100 us at 2 GHz
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
                self.step(i)
                b.record(self.stream)
                b.synchronize()
                if i >= self.n_sets:  # first round over the sets: warm-up
                    single.append(a.elapsed_time(b) * 1e3)
        self.binding.latent_tail_check(self.stream)
        return max_over_ranks(statistics.median(single) * 1e-6, self.world) * 1e6

    def release(self):
        self.sets = []
        self.torch.cuda.synchronize(self.dev)
        self.torch.cuda.empty_cache()


def region_plan(us_est, min_steps, target_s, max_repeats=200):
    """Steps per timed region and number of regions: at least `min_steps` steps
    and about 2 ms per region, repeated until about `target_s` seconds are timed."""
    steps = max(min_steps, int(2000.0 / max(us_est, 1e-3)) + 1)
    region_s = steps * us_est * 1e-6
    repeats = int(min(max_repeats, max(3, round(target_s / max(region_s, 1e-9)))))
    return steps, repeats


def measure_extra(w, args, dev, rank, world, peak):
    """µs/call, tokens/s, the roofline of the dominant kernel and the single-call
    latency of one more benchmark configuration."""
    b = Bench(w, args, dev, rank, world)
    us_est = b.warm(args.warmup)
    steps, repeats = region_plan(us_est, args.steps, 0.05)
    t_call = max_over_ranks(statistics.median(b.timed(b.step, steps, repeats)), world)
    t_proj = max_over_ranks(statistics.median(b.timed(b.project_only, steps, repeats)), world)
    b.binding.latent_tail_check(b.stream)
    us_call, us_proj = t_call / steps * 1e6, t_proj / steps * 1e6
    roof, call_roof = roofline_of(w, us_proj, us_call, *peak)
    rec = {"workload": w.name, "P": w.P, "T": w.T, "L": w.L, "H": w.H,
           "us_per_call": round(us_call, 3),
           "tokens_per_s": round(job_throughput(w.T, steps, world, t_call), 1),
           "single_call_us_median": round(b.single_call_us(100 if w.T <= DECODE_TOKENS else 5), 3),
           "roofline": roof, "call_roofline": call_roof,
           "timing": f"median of {repeats} regions of {steps} graph-replayed calls"}
    b.release()
    return rec


def ours(args):
    import torch

    from latent_moe_output_gb300 import binding, inputs

    rank, world, local = dist_setup(args.gpus)
    w = workload(args.workload)
    if args.T:
        import dataclasses

        w = dataclasses.replace(w, name=f"{w.name}_T{args.T}", T=args.T)
    P, T, L, H = w.P, w.T, w.L, w.H
    dev = torch.device("cuda", local)
    hbm, tc_burst, tc_sus, peak_kind = peaks()
    peak = (hbm, tc_burst, peak_kind)

    b = Bench(w, args, dev, rank, world)
    us_est = b.warm(args.warmup)
    K = args.steps
    # Exactly K steps per timed region; the region is repeated so that the timed
    # time adds up to about a second (clock samples come from inside it).
    repeats = args.repeats or int(min(2000, max(3, round(1.0 / max(K * us_est * 1e-6, 1e-9)))))
    for _, out, _ in b.sets:  # poison outputs: the timed steps must overwrite them
        out.fill_(float("nan"))
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        regions = b.timed(b.step, K, repeats)
    binding.latent_tail_check(b.stream)
    for _, out, _ in b.sets[:min(K, b.n_sets)]:
        if not torch.isfinite(out.float()).all():
            raise RuntimeError("timed steps did not write their outputs")
    t_step = max_over_ranks(statistics.median(regions), world)
    t_proj = max_over_ranks(statistics.median(b.timed(b.project_only, K, repeats)), world)
    binding.latent_tail_check(b.stream)
    graph_calls = b.graph_calls

    # Column-shard form: a step is N latent_tail_forward_cols calls whose ranges
    # (multiples of 8) tile [0, H); together they write the whole output.
    shard_line = None
    if args.shards > 0:
        bounds = [((H // 8) * k // args.shards) * 8 for k in range(args.shards)] + [H]

        def shard_step(i):
            x, out, ws = b.sets[i % b.n_sets]
            for k in range(args.shards):
                binding.latent_tail_forward_cols(x.routed, x.shared, x.g, x.W, out, x.eps,
                                                 bounds[k], bounds[k + 1], ws, b.stream)

        # The same shards with the latent computed once per step: one norm call,
        # then N projection calls over [0, H).
        def shard_step_norm_once(i):
            x, out, ws = b.sets[i % b.n_sets]
            y = ws[:T * L * 2].view(torch.bfloat16).view(T, L)
            binding.latent_tail_norm(x.routed, x.g, y, x.eps, b.stream)
            for k in range(args.shards):
                binding.latent_tail_project_cols(y, x.shared, x.W, out, bounds[k], bounds[k + 1],
                                                 b.stream)

        shard_steps = max(1, min(K, 20))
        t_shards = max_over_ranks(statistics.median(b.timed(shard_step, shard_steps, 3)), world)
        t_once = max_over_ranks(statistics.median(b.timed(shard_step_norm_once, shard_steps, 3)),
                                world)
        binding.latent_tail_check(b.stream)
        shard_line = {"calls_per_step": args.shards, "steps": shard_steps,
                      "us_per_step": round(t_shards / shard_steps * 1e6, 3),
                      "tokens_per_s": round(job_throughput(T, shard_steps, world, t_shards), 1),
                      "note": "each call reduces and normalizes all T tokens again",
                      "norm_once_us_per_step": round(t_once / shard_steps * 1e6, 3),
                      "norm_once_note": "latent_tail_norm once, then N latent_tail_project_cols"}

    us_single = b.single_call_us(100 if T <= DECODE_TOKENS else 5)

    # End to end through the host-buffer entry point: every step takes its
    # partials from page-locked host memory and leaves its result there. The
    # host sets rotate like the device-resident ones (one set when a set exceeds
    # 1 GB: the host link, not L2, bounds such a step).
    e2e_steps = args.e2e_steps or K
    n_host = b.n_sets if b.set_bytes < (1 << 30) else 1
    def pinned_copy(t):  # page-locked host copy without a pageable intermediate
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    hsets = [(pinned_copy(x.routed), pinned_copy(x.shared)) for x, _, _ in b.sets[:n_host]]
    h_out = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    h_ws = torch.empty(binding.latent_tail_host_workspace_size(P, T, L, H), dtype=torch.uint8,
                       device=dev)

    def e2e_step(i):
        x = b.sets[i % b.n_sets][0]
        hr, hs = hsets[i % n_host]
        binding.latent_tail_forward_host(hr, hs, x.g, x.W, h_out, x.eps, h_ws, b.stream)

    # The same step with explicit staging copies issued from Python around the
    # device entry point (pinned host -> device, call, device -> pinned host).
    d_in = {"routed": torch.empty_like(b.sets[0][0].routed),
            "shared": torch.empty_like(b.sets[0][0].shared),
            "out": torch.empty(T, H, dtype=torch.bfloat16, device=dev)}

    def staged_step(i):
        x, _, ws = b.sets[i % b.n_sets]
        hr, hs = hsets[i % n_host]
        d_in["routed"].copy_(hr, non_blocking=True)
        d_in["shared"].copy_(hs, non_blocking=True)
        binding.latent_tail_forward(d_in["routed"], d_in["shared"], x.g, x.W, d_in["out"],
                                    x.eps, ws, b.stream)
        h_out.copy_(d_in["out"], non_blocking=True)

    with torch.cuda.stream(b.stream):
        for i in range(3):
            e2e_step(i)
    b.stream.synchronize()
    e2e_reps = 3
    t_e2e = max_over_ranks(statistics.median(b.timed(e2e_step, e2e_steps, e2e_reps)), world)
    binding.latent_tail_check(b.stream)
    if not torch.isfinite(h_out.float()).all():
        raise RuntimeError("end-to-end steps did not produce a finite result")
    t_staged = max_over_ranks(statistics.median(b.timed(staged_step, e2e_steps, e2e_reps)), world)
    binding.latent_tail_check(b.stream)
    n_sets, set_bytes, l2 = b.n_sets, b.set_bytes, b.l2
    del hsets, h_out, h_ws, d_in
    b.release()

    extra = []
    if not args.no_workloads:
        for name in SUB_WORKLOADS:
            if name != w.name:
                extra.append(measure_extra(workload(name), args, dev, rank, world, peak))

    if rank != 0:
        return
    us_call = t_step / K * 1e6
    us_proj = t_proj / K * 1e6
    roof, call_roof = roofline_of(w, us_proj, us_call, *peak)
    line = {
        "metric": "latent-tail tokens/s", "value": round(job_throughput(T, K, world, t_step), 1),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(t_step / K * 1e3, 6), "us_per_call": round(us_call, 3),
        "single_call_us_median": round(us_single, 3),
        **({"column_shards": shard_line} if shard_line else {}),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "P": P, "T": T, "L": L, "H": H, "eps": inputs.EPS,
                   "parallelism": f"replicas{world}",
                   "l2": f"inputs rotate over {n_sets} sets, {n_sets * set_bytes / 2**20:.0f} MiB"
                         f" > 2x L2 ({l2 / 2**20:.0f} MiB)",
                   "timing": f"median of {repeats} timed regions of exactly {K} steps, each "
                             f"replayed from CUDA graphs of up to {graph_calls} calls and timed "
                             "with CUDA events on the launching stream"},
        "roofline": roof, "call_roofline": call_roof,
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(),
        "e2e": {"value": round(job_throughput(T, e2e_steps, world, t_e2e), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": P * T * L * 2 + P * T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "steps": e2e_steps,
                "us_per_step": round(t_e2e / e2e_steps * 1e6, 3),
                "api": "latent_tail_forward_host (page-locked host partials and result; "
                       + ("kernels read/write them across the host link"
                          if T <= DECODE_TOKENS else "staged with one copy per tensor") + ")",
                "staged_copies_us_per_step": round(t_staged / e2e_steps * 1e6, 3),
                "timing": f"median of {e2e_reps} regions, CUDA graphs, CUDA events, "
                          f"{n_host} pinned host set(s)"},
        "workloads": extra,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, max_tokens=1024)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.capture:
        capture_calls(args.capture)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
