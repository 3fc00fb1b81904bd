"""The CPU legs of bench.py, run here without a GPU.

`--impl reference` times the unmodified oracle as parallel replicas in
spawned processes, one step per barrier; a rank other than 0 does no work.
The all-cores cpu_baseline leg adds the one-core figure beside its own.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    return out.stdout


def test_reference_arm_line():
    out = _run("--impl", "reference", "--steps", "2", "--warmup", "3", "--fixed-sample",
               "--sample-tokens", "256", "--reference-cores", "2")
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3
    assert d["config"]["sample_tokens"] == 256 and d["config"]["replicas"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    out = _run("--impl", "reference", "--steps", "1", "--warmup", "3", env_extra={"RANK": "1"})
    assert out.strip() == ""


def test_cpu_baseline_all_cores_leg():
    sys.path.insert(0, ROOT)
    import bench

    got = bench.cpu_baseline(256, 0.5, 2)
    assert got["cores"] == 2 and got["kind"] == "oracle" and got["value"] > 0
    one = got["single_core"]
    assert one["cores"] == 1 and one["value"] > 0
    assert bench.cpu_baseline(256, 0.2, 1)["cores"] == 1


def test_replica_count_respects_host_memory():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.replica_count(256, 4) == 4
    assert bench.replica_count(256, 0) == 1
    # a sample far beyond host memory leaves one replica
    assert bench.replica_count(1 << 40, 64) == 1
