"""bench.py --impl reference on the CPU: the reference arm (the oracle, timed on the host
cores) prints one JSON line with the driver's keys, the arm's own e2e object and a
cpu_baseline describing the run; under several ranks only rank 0 prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", *args], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_line_has_the_driver_keys():
    (line,) = _run(None, "--workload", "indexer_fp32", "--M", "1")
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["higher_is_better"] is False
    assert line["unit"] == "µs/call" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_prints_on_rank_zero_only():
    assert _run({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}, "--workload", "indexer_fp32", "--M", "1") == []


def test_reference_config_is_the_gpu_arms_config():
    """Both arms describe the same workload with the same config object (bench.py builds
    both from workload_config), so the driver can pair their lines."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    (line,) = _run(None, "--workload", "wq_a_wkv", "--M", "8")
    assert line["config"] == bench.workload_config(W.WORKLOADS["wq_a_wkv"], 8, False, 1)
    assert "tf32" in bench.workload_config(W.WORKLOADS["indexer_fp32"], 64, True, 1)["workload"]
