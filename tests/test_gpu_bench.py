"""bench.py on the GPU prints one JSON line with every key of the bench
contract: the headline metric, the roofline block of the forward kernel, the
end-to-end figure through the host-buffer API, the launch count and the SM
clocks sampled during the timed region.  Runs the headline only (--quick) in
a subprocess."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_prints_the_contract_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--quick", "--steps", "3", "--warmup", "3",
                          "--no-cpu"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["unit"] == "TFLOP/s" and d["dtype"] == "bf16" and d["higher_is_better"] is True
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 3 * 4 * 32 * 4096 * 128 * 2
    assert e["d2h_bytes_per_step"] == 4 * 32 * 4096 * 128 * 2 + 4 * 32 * 4096 * 4
    assert d["gpu_launches"] >= d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert "l2" in d["config"] and "workload" in d["config"]
