"""bench.py's GPU arm, run briefly as a user runs it: one JSON line with the contract's keys,
a decode roofline against the measured peak, a prefill roofline on the mixed workload, the
end-to-end leg with its host copies, and the clocks seen."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", [1, 5])
def test_gpu_arm_prints_the_contract_line(workload):
    j = _run("--workload", str(workload), "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    assert j["metric"] == bench.METRIC and j["unit"] == bench.UNIT and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 5 and j["warmup"] == 3 and j["scaling"] == "weak"
    assert j["value"] > 0 and j["ms_per_step"] > 0 and j["dtype"] == "bf16" and j["data"] == "synthetic"
    assert j["gpu_launches"] >= 3 * 5
    r = j["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert 0 < r["frac"] < 1.2 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["traffic"] is None or r["traffic"] > 0
    e = j["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in j["clocks"] and "reasons" in j["clocks"]
    if workload == 5:  # chunked prefill spans: the tensor roofline of the prefill tiles
        rp = j["roofline_prefill"]
        assert rp["bound"] == "tensor" and rp["unit"] == "TFLOP/s" and rp["algorithmic_flops"] > 0
        assert 0 < rp["frac"] < 1.2 and 0 < rp["frac_of_its_sms"] < 1.2
        assert j["config"]["stream_early"] is True
    else:
        assert j["roofline_prefill"] is None
        assert j["config"]["stream_early"] is False  # a small batch: the flag does not pay
