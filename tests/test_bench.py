"""bench.py's JSON line: the oracle arm on the host, and the CUDA arm on a small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_runs_the_oracle_on_the_host():
    line = _run(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
                 "--ref-seconds", "1"], timeout=300)
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("tiny-")


@pytest.mark.gpu
def test_cuda_arm_line(cuda_device):
    line = _run(["--config", "tiny", "--steps", "4", "--warmup", "3", "--no-cpu-baseline"], timeout=600)
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["steps"] == 4 and line["warmup"] == 3
    assert line["n_gpus"] == 1 and line["scaling"] == "weak" and line["vs_baseline"] is None
    roof = line["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["unit"] in ("GB/s", "TFLOP/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert "traffic" in roof
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])
    assert line["stages"]["pass"]["ms_per_step"] > 0
