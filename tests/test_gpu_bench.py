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


@pytest.mark.gpu
def test_e2e_schedule_matches_oracle_every_step():
    # the bench's e2e schedule (double-buffered uploads and downloads on their
    # own streams around the kernels) with a different input every step:
    # each step's output is the oracle's identity-expert layer for that step's
    # input, so no copy overwrote a buffer that a kernel still read
    import types

    import numpy as np
    import torch

    import bench
    import oracle
    from combine_routing_count_prefix_gb300 import llmoe
    from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS["skewed"]
    inps = [make_inputs(w, seed=s) for s in (3, 4, 5)]
    hins = [bench.pack_e2e_input(inp) for inp in inps]
    steps = 6
    houts = [torch.empty((w.R, w.T, w.H), dtype=torch.int16).pin_memory() for _ in range(steps)]
    rb = llmoe.RankBuffers(w.T, w.H, w.R, w.E, fill=0xA5)
    args = types.SimpleNamespace(e2e_steps=steps)
    bench.run_e2e_pipelined(args, llmoe, w, hins, houts, rb, w.T, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for i in range(steps):
        inp = inps[i % len(inps)]
        u = oracle.unpack(inp["x"], inp["topk_idx"], w.E, num_max_tokens=w.T)
        ref, _ = oracle.combine(u["recv_x"], inp["topk_idx"], inp["topk_w"], w.H, w.E, num_max_tokens=w.T)
        got = houts[i].numpy().view(np.uint16)
        assert np.array_equal(got, ref), f"step {i}: {int((got != ref).sum())} elements differ"
