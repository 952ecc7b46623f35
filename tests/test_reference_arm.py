"""The benchmark's reference arm (no GPU needed): `bench.py --impl reference` times the fp64
oracle on the host cores and prints one JSON line with the same metric, unit and config as the
CUDA arm, plus `impl`, a `cpu_baseline` describing the run and an `e2e` entry with no
host-device copies."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    sys.path.insert(0, ROOT)
    import bench
    assert j["metric"] == bench.METRIC and j["unit"] == bench.UNIT and j["higher_is_better"] is True
    assert j["config"]["workload"] == "b2_t4096" and j["n_gpus"] == 1 and j["steps"] == 1
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["cores"] >= 1 and j["cpu_baseline"]["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
