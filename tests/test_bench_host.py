"""Host-side logic of bench.py that needs no GPU: the max-over-ranks job time
of N replicas (two gloo ranks on CPU), the whole-job throughput formula, and
the reference arm (the CPU oracle on a bounded sample), which rank 0 alone
runs and prints."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(1.5 + rank)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    port = 29500 + (os.getpid() % 2000)
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_and_job_value():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    # N replicas each doing the whole step: the job's rate is N times one rank's
    assert bench.job_tflops(1, 3.3e12, 2.0) == pytest.approx(1650.0)
    assert bench.job_tflops(4, 3.3e12, 2.0) == pytest.approx(4 * 1650.0)


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_silently():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2"}, "--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_line():
    r = _bench({"RANK": "0", "WORLD_SIZE": "1"}, "--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_parse_cpulist():
    import bench
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("5") == {5}
    assert bench.parse_cpulist("") == set()


def test_issue_roofline(monkeypatch):
    import bench
    r = bench.issue_roofline([3000.0, 4000.0, 1500.0], 2000.0)
    assert r is not None and r["bound"] == "alu"
    n = r["instructions_per_element"]["dual_sr"]
    # 152 SMs x 4 schedulers x 32 lanes x 2.0e9 clocks / n elements per second, 3.125 B each
    want = 152 * 4 * 32 * 2.0e9 / n * 3.125 / 1e9
    assert r["peak"]["dY_dual_sr"] == pytest.approx(want)
    assert r["frac"]["dY_dual_sr"] == pytest.approx(1500.0 / want)
    # counts taken on other sources are not used; nor without a sampled clock
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda files: "0" * 16)
    assert bench.issue_roofline([3000.0, 4000.0, 1500.0], 2000.0) is None
    monkeypatch.undo()
    assert bench.issue_roofline([3000.0, 4000.0, 1500.0], None) is None
