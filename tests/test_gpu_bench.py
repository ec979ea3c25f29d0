"""The bench's own arm on the GPU: one short run on the tiny workload prints
one JSON line with the keys the bench contract names (value, roofline with
measured peak and kernel, e2e with the bytes copied, cpu_baseline, clocks,
gpu_launches)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_on_tiny():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "20",
                          "--warmup", "3", "--e2e-steps", "5", "--cpu-seconds", "1", "--configs", "tiny,many_small",
                          "--config-steps", "5"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
                "kernels", "route", "double_buffer", "dispatch_unpack"):
        assert key in d, key
    assert d["steps"] == 20 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["value"] > 0
    assert d["gpu_launches"] == 2 * d["steps"]
    assert d["config"]["workload"] == "tiny"
    rl = d["roofline"]
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s" and rl["peak"] > 0 and rl["achieved"] > 0
    assert abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-3
    assert rl["kernel"] in ("dispatch_kernel", "combine_kernel")
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    cf = d["configs"]  # every requested workload's round, measured the same way
    assert set(cf) == {"tiny", "many_small"}
    for name, c in cf.items():
        for key in ("round_us", "dispatch_us", "combine_us", "effective_gbs", "frac_of_measured_hbm", "shape"):
            assert key in c, (name, key)
        assert c["round_us"] > 0 and c["dispatch_us"] > 0 and c["combine_us"] > 0
