"""The bench's multi-rank path on CPU: world size 2 over gloo.

With several GPUs the bench runs one independent replica per rank (the data
path does not shard across GPUs); what crosses ranks is the barrier and the
max over ranks of the timed values, and only rank 0 prints.  Those host-side
pieces run here with the gloo backend.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    got = bench.max_over_ranks([rank + 1.0, 10.0 - rank, 3.5], world)
    dist.barrier()
    # the reference arm: only rank 0 runs and prints
    buf = io.StringIO()
    if rank != 0:
        with redirect_stdout(buf):
            bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]), rank)
    dist.destroy_process_group()
    q.put((rank, got, buf.getvalue()))


def test_max_over_ranks_and_rank0_only_reference():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict((r, (g, out)) for r, g, out in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        got, out = results[r]
        assert got == [2.0, 10.0, 3.5]
    assert results[1][1] == ""  # rank 1 printed nothing for the reference arm


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([1, 2.5], 1) == [1.0, 2.5]


def test_reference_arm_prints_one_json_line():
    # the reference arm (the CPU oracle) on the tiny workload, as the driver
    # launches it: one JSON line with the keys the bench contract names
    import json
    import subprocess

    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["steps"] == 2 and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
