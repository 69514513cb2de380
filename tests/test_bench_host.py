"""Host-side logic of bench.py: the multi-rank aggregation (as gloo ranks on
the CPU) and the reference arm (the CPU oracle), on small workloads."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r "took" (r + 1) seconds for 10 units of work
    slowest = bench.aggregate_max(float(rank + 1), world)
    bench.barrier(world)
    out[rank] = (slowest, bench.whole_job_value(10.0, slowest, world))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    port = 29000 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, value = res[r]
        assert slowest == 2.0                 # the max over ranks
        assert value == pytest.approx(10.0 * world / 2.0)


def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the same config object as the GPU arm prints for this workload
    from nvfp4_block_scaled_linear_gb300.inputs import WORKLOADS
    w = WORKLOADS["tiny"]
    assert d["config"] == bench.workload_config("tiny", w.draw(), w.swiglu)


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_traffic_is_reported_only_for_the_profiled_sources(monkeypatch):
    """roofline.traffic comes from the committed ncu summary only while the
    kernel sources hash to what the capture recorded; any other hash (the
    sources changed since) turns it into null."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recorded = json.load(f)["smallm"]["decode_gate_up"]["source_hash"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: recorded)
    v = bench.profiled_traffic("smallm", "decode_gate_up")
    assert v is not None and 0.9 * 100_349_956 < v < 1.2 * 100_349_956
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic("smallm", "decode_gate_up") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: recorded)
    assert bench.profiled_traffic("no_such_kernel", "decode_gate_up") is None
