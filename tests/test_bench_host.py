"""Host-side checks of bench.py that need no GPU: the reference arm's JSON line (the CPU
oracle timed on a bounded sample), the warm-up rule, and the rule that recorded DRAM
traffic is reported only for the kernel sources it was measured on."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["unit"] == "TFLOP/s" and j["higher_is_better"] is True
    assert j["value"] > 0 and j["steps"] == 1 and j["warmup"] == 3
    assert "workload" in j["config"]
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr


def test_recorded_traffic_only_for_current_sources(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    workload, kernel = "dense_pair", "prefill"
    entry = rec[workload][kernel]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: entry["kernel_source_hash"])
    assert bench.recorded_traffic(workload, kernel) == entry["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic(workload, kernel) is None
    assert bench.recorded_traffic("no_such_workload", kernel) is None


def test_recorded_traffic_matches_the_committed_sources():
    """The committed ncu traffic was taken on the committed kernel sources."""
    sys.path.insert(0, ROOT)
    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    hashes = {e["kernel_source_hash"] for wl, ks in rec.items() if not wl.startswith("_")
              for e in ks.values()}
    if hashes != {bench.kernel_source_hash()}:
        pytest.skip("kernel sources changed since the last ncu capture (traffic reported as null)")
    assert bench.recorded_traffic("prefill", "prefill") is not None


def _gloo_rank(rank, world, port, values, out_q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(torch, dist, values[rank], "cpu")
        out_q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    """The N > 1 timing path: every rank ends with the slowest rank's time."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    values = [1.25, 3.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gloo_rank, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


def test_whole_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, None, 2.0, "cpu") == 2.0
    # two ranks, 1e12 FLOP each per step, slowest step 2 ms: 1000 TFLOP/s for the job
    assert bench.whole_job_tflops(2, 1e12, 2.0) == pytest.approx(1000.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_arm_samples_each_step_when_full_steps_do_not_fit(monkeypatch, capsys):
    """With many steps the reference arm bounds its work: each step becomes the first rows
    of every output (the sample is named in the line)."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 0.05)
    # smaller shapes of the same pair keep the CPU suite quick
    monkeypatch.setattr(bench.DensePair, "SHAPES", [("prefill", 512, 1024, 512), ("decode", 64, 1024, 1024)])
    monkeypatch.setattr(bench.DensePair, "_oracle_inputs", None)
    args = argparse.Namespace(workload="dense_pair", steps=50, warmup=3, gpus=1)
    assert bench.run_reference(args) == 0
    j = json.loads([ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")][0])
    assert j["steps"] == 50 and j["value"] > 0
    assert "first" in j["cpu_baseline"]["sample"]
