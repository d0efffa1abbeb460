"""Benchmark of the latent-MoE output tail on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|stress|tiny|decode_T1|...]

A step is one call of the whole tail (routed reduce + RMSNorm, up-projection,
shared-partial epilogue) on one batch of synthetic inputs. The default workload
is the decode configuration (P=8, T=16, L=2048, H=7168). Inputs rotate over
enough seeded sets that their total exceeds twice the L2 size, so every step
streams W and the partials from HBM. Steps are replayed from CUDA graphs and
timed with CUDA events on the launching stream, between a barrier and a device
synchronize on both sides; with N > 1 each rank runs its own replica (token
batches are independent, no collective) and the max time over ranks is used.

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
workload.
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
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps (capped)")
    ap.add_argument("--shards", type=int, default=0,
                    help="also time each step as N column-range calls covering [0, H)")
    return ap.parse_args()


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
            "host_cores": os.cpu_count()}


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
    n = int(max(1, min(w.T, per_step_budget / max(per_tok, 1e-9))))
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
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", L2_BYTES) or L2_BYTES
    lib = binding.load_library()

    set_bytes = call_bytes(P, T, L, H) + binding.latent_tail_workspace_size(P, T, L, H)
    n_sets = max(2, -(-2 * l2 // set_bytes) + 1)
    sets = []
    for r in range(n_sets):
        x = inputs.make(P, T, L, H, w.seed + 7919 * r + 104729 * rank, device=dev,
                        outliers=w.outlier_rows)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(binding.latent_tail_workspace_size(P, T, L, H), dtype=torch.uint8,
                         device=dev)
        sets.append((x, out, ws))
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        x, out, ws = sets[i % n_sets]
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws, stream)

    def project_only(i):
        x, out, ws = sets[i % n_sets]
        y = ws[:T * L * 2].view(torch.bfloat16).view(T, L)
        binding.latent_tail_project_cols(y, x.shared, x.W, out, 0, H, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    binding.latent_tail_check(stream)

    chunk = min(args.steps, 50 * n_sets)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    fn(i)
        return g

    def timed(fn, steps):
        graphs = {}
        plan = []
        left = steps
        while left > 0:
            n = min(chunk, left)
            if n not in graphs:
                graphs[n] = capture(fn, n)
            plan.append(graphs[n])
            left -= n
        # CUDAGraph.replay() launches on the current stream: make it `stream`,
        # the stream the events are recorded on.
        with torch.cuda.stream(stream):
            for g in graphs.values():  # untimed replay: settle clocks and caches
                g.replay()
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            barrier(world)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for g in plan:
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            barrier(world)
        return e0.elapsed_time(e1) / 1e3  # seconds

    for _, out, _ in sets:  # poison outputs: the timed steps must overwrite them
        out.fill_(float("nan"))
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        t_step = timed(step, args.steps)
    binding.latent_tail_check(stream)
    written = min(args.steps, n_sets)
    for _, out, _ in sets[:written]:
        if not torch.isfinite(out.float()).all():
            raise RuntimeError("timed steps did not write their outputs")
    t_step = max_over_ranks(t_step, world)
    t_proj = max_over_ranks(timed(project_only, args.steps), world)
    binding.latent_tail_check(stream)

    # Column-shard form: a step is N latent_tail_forward_cols calls whose ranges
    # (multiples of 8) tile [0, H); together they write the whole output.
    shard_line = None
    if args.shards > 0:
        bounds = [((H // 8) * k // args.shards) * 8 for k in range(args.shards)] + [H]

        def shard_step(i):
            x, out, ws = sets[i % n_sets]
            for k in range(args.shards):
                binding.latent_tail_forward_cols(x.routed, x.shared, x.g, x.W, out, x.eps,
                                                 bounds[k], bounds[k + 1], ws, stream)

        # The same shards with the latent computed once per step: one norm call,
        # then N projection calls over [0, H).
        def shard_step_norm_once(i):
            x, out, ws = sets[i % n_sets]
            y = ws[:T * L * 2].view(torch.bfloat16).view(T, L)
            binding.latent_tail_norm(x.routed, x.g, y, x.eps, stream)
            for k in range(args.shards):
                binding.latent_tail_project_cols(y, x.shared, x.W, out, bounds[k], bounds[k + 1],
                                                 stream)

        shard_steps = max(1, min(args.steps, 20))
        t_shards = max_over_ranks(timed(shard_step, shard_steps), world)
        t_once = max_over_ranks(timed(shard_step_norm_once, shard_steps), world)
        binding.latent_tail_check(stream)
        shard_line = {"calls_per_step": args.shards, "steps": shard_steps,
                      "us_per_step": round(t_shards / shard_steps * 1e6, 3),
                      "tokens_per_s": round(job_throughput(T, shard_steps, world, t_shards), 1),
                      "note": "each call reduces and normalizes all T tokens again",
                      "norm_once_us_per_step": round(t_once / shard_steps * 1e6, 3),
                      "norm_once_note": "latent_tail_norm once, then N latent_tail_project_cols"}

    # One call at a time, with nothing before or after it on the GPU (no overlap
    # with a neighbouring call): a spin kernel keeps the GPU busy while the
    # events and the call's two kernel launches are enqueued, so the interval
    # holds only the call's own device time.
    single = []
    with torch.cuda.stream(stream):
        for i in range(max(100, 2 * n_sets) if T <= 128 else 3 * n_sets):
            torch.cuda._sleep(200000)  # ~100 us at 2 GHz
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step(i)
            b.record(stream)
            b.synchronize()
            if i >= n_sets:  # first round over the sets: warm-up
                single.append(a.elapsed_time(b) * 1e3)
    binding.latent_tail_check(stream)
    us_single = max_over_ranks(statistics.median(single) * 1e-6, world) * 1e6

    # End to end through the host-buffer entry point: every step takes its
    # partials from page-locked host memory and leaves its result there. Each
    # input set has its own pinned host copy; steps rotate over them as the
    # device-resident steps do, and are replayed from CUDA graphs the same way.
    e2e_steps = args.e2e_steps or min(args.steps, 500)
    hsets = [(x.routed.cpu().pin_memory(), x.shared.cpu().pin_memory()) for x, _, _ in sets]
    h_out = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    h_ws = torch.empty(binding.latent_tail_host_workspace_size(P, T, L, H), dtype=torch.uint8,
                       device=dev)

    def e2e_step(i):
        x = sets[i % n_sets][0]
        hr, hs = hsets[i % n_sets]
        binding.latent_tail_forward_host(hr, hs, x.g, x.W, h_out, x.eps, h_ws, stream)

    # The same step with explicit staging copies issued from Python around the
    # device entry point (pinned host -> device, call, device -> pinned host).
    d_in = {"routed": torch.empty_like(sets[0][0].routed),
            "shared": torch.empty_like(sets[0][0].shared),
            "out": torch.empty(T, H, dtype=torch.bfloat16, device=dev)}

    def staged_step(i):
        x, _, ws = sets[i % n_sets]
        hr, hs = hsets[i % n_sets]
        d_in["routed"].copy_(hr, non_blocking=True)
        d_in["shared"].copy_(hs, non_blocking=True)
        binding.latent_tail_forward(d_in["routed"], d_in["shared"], x.g, x.W, d_in["out"],
                                    x.eps, ws, stream)
        h_out.copy_(d_in["out"], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    stream.synchronize()
    t_e2e = max_over_ranks(timed(e2e_step, e2e_steps), world)
    binding.latent_tail_check(stream)
    if not torch.isfinite(h_out.float()).all():
        raise RuntimeError("end-to-end steps did not produce a finite result")
    t_staged = max_over_ranks(timed(staged_step, e2e_steps), world)
    binding.latent_tail_check(stream)

    if rank != 0:
        return
    hbm, tc_burst, tc_sus, peak_kind = peaks()
    tokens_per_s = job_throughput(T, args.steps, world, t_step)
    us_call = t_step / args.steps * 1e6
    us_proj = t_proj / args.steps * 1e6
    pb = project_bytes(P, T, L, H)
    cb = call_bytes(P, T, L, H)
    fl = flops(T, L, H)
    proj_gbs = pb / (us_proj * 1e-6) / 1e9
    call_gbs = cb / (us_call * 1e-6) / 1e9
    # The binding roofline of the projection kernel: HBM unless its flops take
    # longer at the tensor peak than its bytes at the HBM peak (P = 1 prefill).
    tensor_bound = fl / (tc_burst * 1e12) > pb / (hbm * 1e9)
    kname = "decode_kernel" if T <= 128 else "prefill_kernel"
    if tensor_bound:
        proj_tf = fl / (us_proj * 1e-6) / 1e12
        roof = {"kernel": kname, "bound": "tensor", "achieved": round(proj_tf, 1),
                "peak": tc_burst, "unit": "TFLOP/s", "frac": round(proj_tf / tc_burst, 4),
                "traffic": None, "algorithmic_flops_per_launch": fl,
                "us_per_launch": round(us_proj, 3), "peak_source": peak_kind}
    else:
        roof = {"kernel": kname, "bound": "hbm", "achieved": round(proj_gbs, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(proj_gbs / hbm, 4),
                "traffic": profiled_traffic(kname, w.name, T),
                "algorithmic_bytes_per_launch": pb, "us_per_launch": round(us_proj, 3),
                "peak_source": peak_kind}
    call_roof = {"achieved": round(call_gbs, 1), "peak": hbm, "unit": "GB/s",
                 "frac": round(call_gbs / hbm, 4), "algorithmic_bytes_per_call": cb,
                 "tensor_tflops": round(fl / (us_call * 1e-6) / 1e12, 2),
                 "tensor_frac_of_burst_peak": round(fl / (us_call * 1e-6) / 1e12 / tc_burst, 4)}
    line = {
        "metric": "latent-tail tokens/s", "value": round(tokens_per_s, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_step / args.steps * 1e3, 6), "us_per_call": round(us_call, 3),
        "single_call_us_median": round(us_single, 3),
        **({"column_shards": shard_line} if shard_line else {}),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "P": P, "T": T, "L": L, "H": H, "eps": inputs.EPS,
                   "parallelism": f"replicas{world}",
                   "l2": f"inputs rotate over {n_sets} sets, {n_sets * set_bytes / 2**20:.0f} MiB"
                         f" > 2x L2 ({l2 / 2**20:.0f} MiB)",
                   "timing": "CUDA graphs of up to %d calls, CUDA events on the launching stream"
                             % chunk},
        "roofline": roof, "call_roofline": call_roof,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
        "e2e": {"value": round(job_throughput(T, e2e_steps, world, t_e2e), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": P * T * L * 2 + P * T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "steps": e2e_steps,
                "us_per_step": round(t_e2e / e2e_steps * 1e6, 3),
                "api": "latent_tail_forward_host (page-locked host partials and result; "
                       + ("kernels read/write them across the host link"
                          if T <= 128 else "staged with one copy per tensor") + ")",
                "staged_copies_us_per_step": round(t_staged / e2e_steps * 1e6, 3),
                "timing": "CUDA graphs, CUDA events, inputs rotate over pinned host sets"},
    }
    if not args.no_cpu_baseline and world >= 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
