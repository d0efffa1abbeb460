"""bench.py's host-side arithmetic and bookkeeping (no GPU): the algorithmic byte
and flop counts the roofline divides by, the whole-job throughput, and the rule
that a profiled DRAM traffic figure is reported only while the kernel's source is
the one that was captured."""

import hashlib
import importlib
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
bench = importlib.import_module("bench")


@pytest.mark.parametrize("P,T,width,mb,gflop", [
    # bytes = P*T*L*2 (routed) + P*T*w*2 (shared) + w*L*2 (W) + T*w*2 (out) + L*4 (g)
    (8, 1, 7168, 29.53, 0.02936),
    (8, 16, 7168, 31.96, 0.470),
    (8, 128, 7168, 50.08, 3.758),
    (8, 8192, 7168, 1354.8, 240.5),
    (16, 16384, 7168, 5096.1, 481.0),
    (16, 16384, 448, 1325.1, 30.1),   # one of the 16 stress column shards
    (1, 8192, 7168, 297.8, 240.5),    # pre-reduced P = 1 workload
])
def test_algorithmic_bytes_and_flops(P, T, width, mb, gflop):
    L = 2048
    assert bench.call_bytes(P, T, L, width) / 1e6 == pytest.approx(mb, abs=0.06)
    assert bench.flops(T, L, width) / 1e9 == pytest.approx(gflop, rel=2e-3)


def test_projection_bytes_exclude_the_routed_partials():
    P, T, L, w = 8, 16, 2048, 7168
    # the projection reads the latent y (T*L*2) instead of the P routed partials
    assert bench.call_bytes(P, T, L, w) - bench.project_bytes(P, T, L, w) == \
        P * T * L * 2 - T * L * 2 + L * 4


def test_job_throughput_counts_every_rank_over_the_slowest_time():
    assert bench.job_throughput(16, 1000, 4, 0.01) == pytest.approx(16 * 1000 * 4 / 0.01)


def _write_profile(dirpath, kernel, digest, workload="decode", T=16, nbytes=31292160):
    (dirpath / f"{kernel}_X.md").write_text(
        f"# summary\n\ntraffic_per_launch_bytes: {nbytes} (workload {workload}, T {T}, "
        f"{kernel.replace('_kernel', '')}.cu sha256 {digest})\n")


def test_profiled_traffic_needs_matching_workload_and_source(tmp_path, monkeypatch):
    csrc = tmp_path / "latent_moe_output_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "decode.cu"
    src.write_text("// kernel source as captured\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    _write_profile(tmp_path / "profiles", "decode_kernel", digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("decode_kernel", "decode", 16) == 31292160
    assert bench.profiled_traffic("decode_kernel", "decode", 8) is None        # other T
    assert bench.profiled_traffic("decode_kernel", "prefill", 16) is None      # other workload
    src.write_text("// kernel source changed since the capture\n")
    assert bench.profiled_traffic("decode_kernel", "decode", 16) is None       # stale capture


def test_committed_traffic_lines_name_a_kernel_source():
    """Every traffic figure under profiles/ names a workload of the benchmark list
    and a kernel source file of the library (bench.py uses a figure only while
    that file still has the recorded hash)."""
    import re

    from latent_moe_output_gb300 import inputs

    pat = re.compile(r"^\w*traffic_per_launch_bytes: (\d+) \(workload (\w+), T (\d+), "
                     r"(\S+) sha256 ([0-9a-f]{16})\)", re.M)
    found = 0
    for path in (ROOT / "profiles").glob("*.md"):
        for m in pat.finditer(path.read_text()):
            found += 1
            assert (ROOT / "latent_moe_output_gb300" / "csrc" / m.group(4)).exists(), path
            base = m.group(2).split("_T")[0] if m.group(2) not in inputs.WORKLOADS else m.group(2)
            assert base in inputs.WORKLOADS, path
    assert found > 0


def test_workloads_are_the_benchmark_configurations():
    from latent_moe_output_gb300 import inputs

    w = inputs.WORKLOADS
    assert (w["tiny"].P, w["tiny"].T, w["tiny"].L, w["tiny"].H, w["tiny"].seed) == (2, 5, 64, 128, 0)
    assert (w["decode"].P, w["decode"].T, w["decode"].L, w["decode"].H) == (8, 16, 2048, 7168)
    assert sorted(x.T for x in inputs.DECODE_SWEEP) == [1, 2, 4, 8, 32, 64, 128]
    assert all(x.seed == 1000 + x.T and x.P == 8 for x in inputs.DECODE_SWEEP)
    assert (w["prefill"].P, w["prefill"].T) == (8, 8192)
    assert (w["stress"].P, w["stress"].T, w["stress"].outlier_rows) == (16, 16384, True)
    assert inputs.STRESS_SHARDS == 16 and w["stress"].H % inputs.STRESS_SHARDS == 0
    assert inputs.EPS == 1e-6


def test_reference_arm_prints_one_complete_line(capsys, monkeypatch):
    """`bench.py --impl reference` times the oracle and prints the contract's keys,
    on rank 0 only."""
    import json
    import types

    args = types.SimpleNamespace(workload="tiny", steps=2, warmup=1, gpus=1)
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.reference_arm(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    monkeypatch.setenv("RANK", "1")
    bench.reference_arm(args)
    assert capsys.readouterr().out.strip() == ""


def test_every_benchmark_workload_has_current_traffic():
    """Every configuration bench.py reports (the headline and its workloads record)
    has a DRAM-traffic figure under profiles/ taken on the current source of the
    kernel that dominates it: a kernel change without a new capture fails here."""
    from latent_moe_output_gb300 import inputs

    names = ["stress", "prefill", "prefill_p1", "decode"] + [w.name for w in inputs.DECODE_SWEEP]
    for name in names:
        w = inputs.WORKLOADS[name]
        kname = ("gemv_kernel" if w.T <= 2 else
                 "decode_kernel" if w.T <= bench.DECODE_TOKENS else "prefill_kernel")
        assert bench.profiled_traffic(kname, w.name, w.T) is not None, (name, kname)
