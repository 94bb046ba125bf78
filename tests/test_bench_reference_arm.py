"""bench.py --impl reference (the oracle on the host, the reference arm):
one JSON line with the contract's keys, runnable without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "ring4_int", "--steps", "2", "--warmup", "3"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s" and d["steps"] == 2
    assert d["config"]["workload"] == "ring4_int"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_on_an_n_d_torus_sample():
    """The reference arm's oracle sample keeps the workload's schedule: an
    n-D torus with layer-list buckets, cut to 20,000 elements per rank."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "torus4x4x4_resnet101", "--elems", "20000", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    assert d["config"]["schedules"] == ["torus 4x4x4"] and d["value"] > 0


def test_reference_arm_default_is_the_three_schedule_sweep():
    """With no --workload the reference arm times the same step as the GPU
    arm: ring, multi-ring k=2 and 4x4 torus on the 300M-parameter language
    model's P=16 problem (here cut to 20,000 elements per rank), and states
    the host cores it ran on."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--elems", "20000",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    assert d["config"]["workload"] == "lm300m_sweep"
    assert d["config"]["schedules"] == ["ring", "multi-ring k=2", "torus 4x4"]
    assert d["config"]["P"] == 16 and d["config"]["sample_elems_per_rank"] == 20000
    cb = d["cpu_baseline"]
    assert cb["cores"] == 1 and cb["nproc"] >= 1 and cb["cpu_model"]
