#!/usr/bin/env python
"""Benchmark: microseconds per dispatch + combine round on one GB300.

A step is one round on one batch of synthetic input, through the C ABI:
    llmoe_dispatch(set 0); llmoe_combine(set 1)
with each call also zeroing the other buffer set's signal words (the two
llmoe_clean calls of a round, fused into the data kernels); the same round as
four separate calls (clean, dispatch, clean, combine) is reported beside it,
on the DeepSeek-V3-shaped decode workload (R=8 simulated ranks, T=128 tokens
per rank, H=7168 bf16, E=256 experts, top-8, uniform routing) unless
--workload says otherwise.  Inputs are resident in HBM; L2 is flushed before
every timed step, outside the step's events (a 512 MB write, then a 256 MB
read so the written lines are evicted before the step).  ``value`` comes from
events around whole rounds; a second pass with events around every kernel
gives the per-kernel times and the roofline.

Printed (rank 0, one JSON line): the mean step time as ``value``; the
effective HBM bandwidth of the algorithmic bytes; per-kernel times; the
roofline of the dominant kernel against the measured copy bandwidth; the
end-to-end time of one MoE layer with identity experts through the C ABI
with host buffers (x, topk_idx, topk_w copied from pinned host memory,
dispatch, unpack, combine over the unpacked rows, output read back, all
inside the timed region), and of the bench round with the dense expert
outputs also uploaded; the CPU oracle timed on a bounded sample on the host;
GPU clocks sampled during the timed region.

--impl reference times the CPU oracle alone on the host cores (the
reference arm; rank 0 only when launched with several ranks).
--gpus N > 1 (under torchrun): N independent replicas, one per GPU (the data
path does not shard across GPUs here); value is the slowest rank's step time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per dispatch+combine round and effective HBM GB/s (% of 8 TB/s) at 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20
FLUSH_READ_BYTES = 256 << 20


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="dsv3")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--dtype", choices=["bf16", "fp16", "fp32"], default="bf16", help="payload type T")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-e2e-dense-y", action="store_true", help="skip the e2e leg that uploads the dense y")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true", help="skip the other workloads' rounds")
    p.add_argument("--configs", default="tiny,dsv3,skewed,many_small,large",
                   help="workloads whose round the line's configs object reports")
    p.add_argument("--config-steps", type=int, default=50, help="rounds timed per other workload (at most --steps)")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# algorithmic bytes (per launch / per round)
# ---------------------------------------------------------------------------

def algorithmic_bytes(w, n_valid: int, tokens: int, es: int = 2) -> dict:
    """Bytes the path must move, no re-reads or staging counted.

    dispatch = x read + top-k ids read + N messages written + R*E count words
    combine  = ids + weights read + N expert rows read + output written + R*E flag words
    clean    = R*E signal words per set
    """
    R, H, E, K = w.R, w.H, w.E, w.K
    row = es * H
    disp = R * tokens * row + R * tokens * K * 8 + n_valid * (4 + row) + R * E * 8
    comb = R * tokens * K * 12 + n_valid * row + R * tokens * row + R * E * 8
    clean = R * E * 8
    return {"dispatch": disp, "combine": comb, "clean": clean, "round": disp + comb + 2 * clean}


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source with comments and blank space removed (neither string
    literal of the library holds a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest() -> str:
    """Digest of the library's code (kernels and header), comments and layout
    ignored: the traffic figures stay valid across comment-only edits."""
    h = hashlib.sha256()
    for rel in ("combine_routing_count_prefix_gb300/csrc/llmoe.cu", "include/llmoe.h"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when there is none or it was taken on different kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            return int(parts[2]) if parts[3] == digest else None
    return None


def max_over_ranks(values, world: int):
    """Elementwise maximum of a list of floats over all ranks (the slowest
    rank's time); identity for one rank.  Uses the process group's device:
    CUDA for nccl, CPU for gloo."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch

    try:
        p = torch.cuda.get_device_properties(device_index)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[device_index] if vis else str(device_index)


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_round(inp, w, tokens: int):
    """One oracle round on the first `tokens` tokens of every rank."""
    import oracle

    x = np.ascontiguousarray(inp["x"][:, :tokens])
    idx = np.ascontiguousarray(inp["topk_idx"][:, :tokens])
    wt = np.ascontiguousarray(inp["topk_w"][:, :tokens])
    oracle.clean(w.R, w.E)
    oracle.dispatch(x, idx, w.E, num_max_tokens=w.T)
    oracle.clean(w.R, w.E)
    oracle.combine((inp["y_pool"], inp["y_row_map"]), idx, wt, w.H, w.E, num_max_tokens=w.T)


def cores_used() -> int:
    return 1  # the oracle is single-threaded


def cpu_baseline(inp, w, budget_s: float) -> dict:
    """Full oracle rounds until the budget is spent (at least one)."""
    import oracle

    oracle.build()
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t0 = time.perf_counter()
        oracle_round(inp, w, w.T)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() >= t_end or len(times) >= 200:
            break
    us = statistics.mean(times) * 1e6
    return {"value": round(us, 1), "unit": "us/round", "cores": cores_used(), "kind": "oracle",
            "sample": f"{len(times)} full {w.name} rounds (clean, dispatch, clean, combine) of the single-threaded "
                      f"C oracle; host has {len(os.sched_getaffinity(0))} cores available"}


def run_reference(args, rank: int):
    import oracle
    from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs

    if rank != 0:
        return
    oracle.build()
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=args.seed)
    # size each step's token sample so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    probe = max(1, w.T // 16)
    oracle_round(inp, w, probe)
    per_token = max((time.perf_counter() - t0) / probe, 1e-7)
    budget_per_step = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(min(w.T, max(1, budget_per_step / per_token)))
    for _ in range(args.warmup):
        oracle_round(inp, w, tokens)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_round(inp, w, tokens)
        times.append(time.perf_counter() - t0)
    us_full = statistics.mean(times) * 1e6 * (w.T / tokens)
    algo = algorithmic_bytes(w, int((inp["topk_idx"] >= 0).sum()), w.T)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us_full, 2), "unit": "us/round", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic", "effective_gbs": round(algo["round"] / us_full / 1e3, 3),
        "config": {"workload": w.name, "shape": w.describe(), "seed": args.seed,
                   "sample": f"each step runs the oracle on {tokens} of {w.T} tokens per rank; value scales the "
                             f"step time to a full round"},
        "cpu_baseline": {"value": round(us_full, 2), "unit": "us/round", "cores": cores_used(), "kind": "oracle",
                         "sample": f"{tokens}/{w.T} tokens per rank per step, {args.steps} steps"},
        "e2e": {"value": round(us_full, 2), "unit": "us/round", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    from combine_routing_count_prefix_gb300 import build as cuda_build

    cuda_build.build()
    from combine_routing_count_prefix_gb300 import llmoe
    from combine_routing_count_prefix_gb300.inputs import WORKLOADS, dense_y, make_inputs

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=args.seed, dtype=args.dtype)
    tokens = w.T
    n_valid = int((inp["topk_idx"] >= 0).sum())
    es = 4 if args.dtype == "fp32" else 2
    algo = algorithmic_bytes(w, n_valid, tokens, es)

    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    x, idx, wt = dev(inp["x"]), dev(inp["topk_idx"]), dev(inp["topk_w"])
    y = dev(inp["y_pool"]).index_select(0, dev(inp["y_row_map"])).contiguous()
    out = torch.empty((w.R, tokens, w.H), dtype=torch.float32 if es == 4 else torch.int16, device="cuda")
    rb = llmoe.RankBuffers(w.T, w.H, w.R, w.E, fill=0, dtype=args.dtype)
    # a round is dispatch(set 0) + combine(set 1) with each kernel also
    # zeroing the other set's signal words (the cleans the next calls need,
    # fused: LLMOE_FLAG_CLEAN_OTHER_SET); the combine's routing is ready long
    # before the kernel that precedes it, as in a MoE layer whose router ran
    # before the experts, so it is scanned while that kernel drains
    # (LLMOE_FLAG_INPUTS_READY)
    F = llmoe.LLMOE_FLAG_CLEAN_OTHER_SET
    bs0 = rb.buf_set(0, w.K, flags=F)
    bs1 = rb.buf_set(1, w.K, flags=F | llmoe.LLMOE_FLAG_INPUTS_READY)
    # the same round as four calls with separate cleans
    bs0_plain, bs1_plain = rb.buf_set(0, w.K), rb.buf_set(1, w.K, flags=llmoe.LLMOE_FLAG_INPUTS_READY)
    # L2 flush between timed steps: write a buffer larger than L2, then read
    # another one so the written lines are evicted (and written back) before
    # the step's first event instead of inside the step
    flush_w = torch.empty(FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")
    flush_r = torch.ones(FLUSH_READ_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        flush_w.zero_()
        flush_r.sum()

    stream = torch.cuda.current_stream()
    # the C-ABI calls of a round, arguments marshalled once
    dispatch = llmoe.bind_dispatch(x, idx, bs0, stream)
    combine = llmoe.bind_combine(y, idx, wt, out, bs1, stream)
    clean0, clean1 = llmoe.bind_clean(bs0_plain, stream), llmoe.bind_clean(bs1_plain, stream)
    dispatch_plain = llmoe.bind_dispatch(x, idx, bs0_plain, stream)
    combine_plain = llmoe.bind_combine(y, idx, wt, out, bs1_plain, stream)

    combine_staged = llmoe.Bound("llmoe_combine_staged", combine.args, combine.keep)

    def step():
        dispatch()
        combine()

    def step_four_calls():
        clean0()
        dispatch_plain()
        clean1()
        combine_plain()

    # the same round captured once as a CUDA graph (two kernel nodes with a
    # programmatic edge), replayed per step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        llmoe.llmoe_dispatch(x, idx, bs0)
        llmoe.llmoe_combine(y, idx, wt, out, bs1)

    clean0()  # once, before the first round
    for _ in range(args.warmup):
        flush()
        step()
    for _ in range(3):
        step_four_calls()
    clean0()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    def new_events(n, k):
        return [[torch.cuda.Event(enable_timing=True) for _ in range(k)] for _ in range(n)]

    ev, ev4, evk = new_events(args.steps, 2), new_events(args.steps, 2), new_events(args.steps, 3)
    evs, evg, evf = new_events(args.steps, 2), new_events(args.steps, 2), new_events(args.steps, 2)
    with ClockSampler(gpu_id_for(local_rank)) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall0 = time.perf_counter()
        # timed region (value): events around each round only, so the two
        # kernels overlap their launch with the previous kernel's drain
        for e in ev:
            flush()
            e[0].record(stream)
            step()
            e[1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - wall0
        # the four-call round
        for e in ev4:
            flush()
            e[0].record(stream)
            step_four_calls()
            e[1].record(stream)
        clean0()
        # events around every kernel (roofline)
        for e in evk:
            flush()
            e[0].record(stream)
            dispatch()
            e[1].record(stream)
            combine()
            e[2].record(stream)
        # the combine alone after its own flush (the dispatch's dirty lines
        # written back first, outside the events)
        for e in evf:
            flush()
            dispatch()
            flush()
            e[0].record(stream)
            combine()
            e[1].record(stream)
        # the round replayed from its CUDA graph
        for e in evg:
            flush()
            e[0].record(stream)
            graph.replay()
            e[1].record(stream)
        # the staged combine (messages through combine_recv[e][t], then the reduction)
        for e in evs:
            flush()
            dispatch()
            e[0].record(stream)
            combine_staged()
            e[1].record(stream)
        torch.cuda.synchronize()
    staged_ms = [e[0].elapsed_time(e[1]) for e in evs]
    graph_ms = [e[0].elapsed_time(e[1]) for e in evg]
    comb_flushed_ms = [e[0].elapsed_time(e[1]) for e in evf]
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    four_ms = [e[0].elapsed_time(e[1]) for e in ev4]
    disp_ms = [e[0].elapsed_time(e[1]) for e in evk]
    comb_ms = [e[1].elapsed_time(e[2]) for e in evk]
    timed = max_over_ranks([sum(step_ms), wall], world)
    round_us = timed[0] / args.steps * 1e3

    route = run_route(llmoe, w, idx, rb, tokens, flush)
    pipe = run_pipeline(args, llmoe, w, x, idx, wt, y, rb, tokens, es)
    signaled = run_signaled(args, llmoe, w, x, idx, rb, es, flush)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, llmoe, w, inp, dense_y, rb, tokens, stream)
        e2e["value"] = max_over_ranks([e2e["value"]], world)[0]

    d_us = statistics.mean(disp_ms) * 1e3
    c_us = statistics.mean(comb_ms) * 1e3
    configs = None
    if not args.no_configs:
        # the other workloads, one at a time on freed memory; this one from the measurements above
        this = {"round_us": round(round_us, 3), "dispatch_us": round(d_us, 3), "combine_us": round(c_us, 3),
                "steps": args.steps}
        del x, idx, wt, y, out, rb, dispatch, combine, dispatch_plain, combine_plain, combine_staged, graph
        del clean0, clean1, bs0, bs1, bs0_plain, bs1_plain
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        configs = run_configs(args, llmoe, w, this, algo, n_valid, flush, world)

    if rank == 0:
        peak, peak_kind = measured_hbm_peak()
        dom, dom_us = ("dispatch", d_us) if d_us >= c_us else ("combine", c_us)
        dom_gbs = algo[dom] / dom_us / 1e3
        traffic = ncu_traffic(dom + "_kernel", w.name)
        gbs = algo["round"] * world / round_us / 1e3
        line = {
            "metric": METRIC, "value": round(round_us, 3), "unit": "us/round", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(round_us / 1e3, 6),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": args.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "shape": w.describe(), "seed": args.seed, "tokens_per_rank": tokens,
                       "unmasked_entries": n_valid, "parallelism": f"replicas{world}",
                       "l2": f"flushed before every timed step, outside the events ({FLUSH_BYTES >> 20} MB write, "
                             f"then {FLUSH_READ_BYTES >> 20} MB read so the written lines leave L2 first)",
                       "round": "llmoe_dispatch(set 0) + llmoe_combine(set 1), each zeroing the other set's "
                                "signal words (LLMOE_FLAG_CLEAN_OTHER_SET: the llmoe_clean calls fused); combine "
                                "with LLMOE_FLAG_INPUTS_READY; round_us_four_calls: clean, dispatch, clean, "
                                "combine as four calls; round_us_cuda_graph: the two-launch round captured "
                                "once as a CUDA graph and replayed",
                       "timing": "value: CUDA events around each round; per-kernel times and roofline: a second "
                                 "pass with events around every kernel, same step count; combine_us_l2_flushed: "
                                 "the combine with L2 flushed between it and the dispatch"},
            "effective_gbs": round(gbs, 1), "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "frac_of_measured_hbm": round(gbs / peak, 4),
            "algorithmic_bytes_per_round": algo["round"],
            "dispatch_us": round(d_us, 3), "combine_us": round(c_us, 3),
            "combine_us_l2_flushed": round(statistics.mean(comb_flushed_ms) * 1e3, 3),
            "round_us_four_calls": round(statistics.mean(four_ms) * 1e3, 3),
            "round_us_cuda_graph": round(statistics.mean(graph_ms) * 1e3, 3),
            "staged_combine_us": round(statistics.mean(staged_ms) * 1e3, 3),
            "staged_combine_gbs": round((algo["combine"] + 2 * n_valid * (4 + es * w.H)) /
                                        (statistics.mean(staged_ms) * 1e3) / 1e3, 1),
            "step_us_median": round(statistics.median(step_ms) * 1e3, 3),
            "wall_s": round(timed[1], 3),
            "roofline": {"kernel": dom + "_kernel", "bound": "hbm", "achieved": round(dom_gbs, 1),
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                         "traffic": traffic, "algorithmic_bytes": algo[dom]},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks.summary(),
        }
        cf_us = statistics.mean(comb_flushed_ms) * 1e3
        line["kernels"] = {  # every kernel of the round against the same measured peak
            "dispatch_kernel": {"us": round(d_us, 3), "gbs": round(algo["dispatch"] / d_us / 1e3, 1),
                                "frac": round(algo["dispatch"] / d_us / 1e3 / peak, 4)},
            "combine_kernel": {"us": round(c_us, 3), "gbs": round(algo["combine"] / c_us / 1e3, 1),
                               "frac": round(algo["combine"] / c_us / 1e3 / peak, 4)},
            "combine_kernel_l2_flushed": {"us": round(cf_us, 3), "gbs": round(algo["combine"] / cf_us / 1e3, 1),
                                          "frac": round(algo["combine"] / cf_us / 1e3 / peak, 4)}}
        line["route"] = route
        line["double_buffer"] = pipe
        line["dispatch_unpack"] = signaled
        if configs is not None:
            line["configs"] = configs
        if e2e is not None:
            line["e2e"] = e2e
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(inp, w, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def config_bytes(w, es: int) -> int:
    """Device bytes one workload needs: the rank buffers, the dense expert
    outputs y [E*R*T, H], x and the output, with 1 GB to spare."""
    from combine_routing_count_prefix_gb300 import llmoe

    layout = llmoe.llmoe_layout_bytes_dtype(w.T, w.H, w.R, w.E, llmoe.DTYPE_CODES["fp32" if es == 4 else "bf16"])
    return w.R * llmoe.round_up(layout, 256) + w.E * w.R * w.T * w.H * es + 2 * w.R * w.T * w.H * es + (1 << 30)


def run_configs(args, llmoe, main_w, main_res, main_algo, main_n, flush, world):
    """Every workload of the bench, measured as the main one is: L2 flushed
    before each round (outside the events), CUDA events around the two-launch
    round, then around each kernel.  Returns {workload: figures}; a workload
    that does not fit in free device memory reports so instead."""
    import torch

    from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs

    peak, _ = measured_hbm_peak()
    es = 4 if args.dtype == "fp32" else 2
    steps = max(3, min(args.steps, args.config_steps))
    res = {}
    for name in args.configs.split(","):
        w = WORKLOADS[name]
        r = None
        if name == main_w.name:
            r, algo, n_valid = dict(main_res), main_algo, main_n
        else:
            free, _total = torch.cuda.mem_get_info()
            need = config_bytes(w, es)
            if need <= free:
                inp = make_inputs(w, seed=args.seed, dtype=args.dtype)
                n_valid = int((inp["topk_idx"] >= 0).sum())
                algo = algorithmic_bytes(w, n_valid, w.T, es)
                r = measure_round(llmoe, w, inp, es, steps, flush)
                del inp
                torch.cuda.empty_cache()
        # every rank takes part in the maximum, measured or not
        slowest = max_over_ranks([r["round_us"] if r is not None else -1.0], world)[0]
        if r is None:
            res[name] = {"shape": w.describe(), "insufficient free HBM":
                         f"needs {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free"}
            continue
        r["round_us"] = slowest
        gbs = algo["round"] / r["round_us"] / 1e3
        r.update({"shape": w.describe(), "unmasked_entries": n_valid, "algorithmic_bytes_per_round": algo["round"],
                  "effective_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4),
                  "dispatch_frac": round(algo["dispatch"] / r["dispatch_us"] / 1e3 / peak, 4),
                  "combine_frac": round(algo["combine"] / r["combine_us"] / 1e3 / peak, 4)})
        res[name] = r
    return res


def measure_round(llmoe, w, inp, es: int, steps: int, flush) -> dict:
    """The bench round of one workload (dispatch on set 0, combine on set 1,
    cleans fused) on its own buffers: mean µs of the round, then of each
    kernel, L2 flushed before every round."""
    import torch

    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    x, idx, wt = dev(inp["x"]), dev(inp["topk_idx"]), dev(inp["topk_w"])
    y = dev(inp["y_pool"]).index_select(0, dev(inp["y_row_map"])).contiguous()
    out = torch.empty((w.R, w.T, w.H), dtype=torch.float32 if es == 4 else torch.int16, device="cuda")
    rb = llmoe.RankBuffers(w.T, w.H, w.R, w.E, fill=0, dtype="fp32" if es == 4 else "bf16")
    F = llmoe.LLMOE_FLAG_CLEAN_OTHER_SET
    bs0 = rb.buf_set(0, w.K, flags=F)
    bs1 = rb.buf_set(1, w.K, flags=F | llmoe.LLMOE_FLAG_INPUTS_READY)
    stream = torch.cuda.current_stream()
    dispatch = llmoe.bind_dispatch(x, idx, bs0, stream)
    combine = llmoe.bind_combine(y, idx, wt, out, bs1, stream)
    llmoe.llmoe_clean(rb.buf_set(0, w.K), stream)
    for _ in range(3):
        flush()
        dispatch()
        combine()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    ek = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        flush()
        e[0].record(stream)
        dispatch()
        combine()
        e[1].record(stream)
    for e in ek:
        flush()
        e[0].record(stream)
        dispatch()
        e[1].record(stream)
        combine()
        e[2].record(stream)
    torch.cuda.synchronize()
    r = {"round_us": round(statistics.mean(a.elapsed_time(b) for a, b, _ in ev) * 1e3, 3),
         "dispatch_us": round(statistics.mean(a.elapsed_time(b) for a, b, _ in ek) * 1e3, 3),
         "combine_us": round(statistics.mean(b.elapsed_time(c) for _, b, c in ek) * 1e3, 3), "steps": steps}
    del dispatch, combine, x, idx, wt, y, out, rb
    return r


def run_route(llmoe, w, idx, rb, tokens, flush, steps: int = 200):
    """llmoe_route on its own (the routing count / prefix scan that the
    dispatch and combine kernels run inside): ids read, slots and counts
    written; L2 flushed before each launch, events around it."""
    import torch

    slot = torch.empty((w.R, tokens, w.K), dtype=torch.int32, device="cuda")
    counts = torch.empty((w.E, w.R), dtype=torch.int64, device="cuda")
    bs = rb.buf_set(0, w.K)
    cur = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps + 3):
        flush()
        if i >= 3:
            evs[i - 3][0].record(cur)
        llmoe.llmoe_route(idx, slot, counts, bs, cur)
        if i >= 3:
            evs[i - 3][1].record(cur)
    torch.cuda.synchronize()
    us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    nbytes = idx.numel() * 8 + slot.numel() * 4 + counts.numel() * 8
    return {"us": round(us, 3), "algorithmic_bytes": nbytes, "steps": steps,
            "note": "events around llmoe_route alone, L2 flushed before each launch: launch- and latency-bound"}


def run_pipeline(args, llmoe, w, x, idx, wt, y, rb, tokens, es, micro_batches: int = 200):
    """Micro-batches back to back: serial on one stream (clean, dispatch,
    clean, combine on one set each) against the two-stream double-buffered
    schedule, where micro-batch b+1's dispatch overlaps micro-batch b's
    combine (sets b % 2).  No L2 flush between micro-batches: this is the
    steady state of a pipeline.  Each schedule is timed as issued from Python
    (eager) and replayed from a CUDA graph captured once (both streams join
    the capture), which takes the host's issue rate out of the figure."""
    import torch

    from combine_routing_count_prefix_gb300.pipeline import DoubleBufferPipeline

    outs = [torch.empty((w.R, tokens, w.H), dtype=torch.float32 if es == 4 else torch.int16, device="cuda")
            for _ in (0, 1)]
    bs = [rb.buf_set(s, w.K) for s in (0, 1)]

    def serial():
        cur = torch.cuda.current_stream()
        for b in range(micro_batches):
            s = b % 2
            llmoe.llmoe_clean(bs[s], cur)
            llmoe.llmoe_dispatch(x, idx, bs[s], cur)
            llmoe.llmoe_clean(bs[s], cur)
            llmoe.llmoe_combine(y, idx, wt, outs[s], bs[s], cur)

    # one schedule for eager calls, a fresh one for the capture: a captured
    # stream may only wait on events recorded inside the same capture
    pipes = {False: DoubleBufferPipeline(rb, w.K), True: DoubleBufferPipeline(rb, w.K)}

    def pipelined():
        pipe = pipes[torch.cuda.is_current_stream_capturing()]
        for b in range(micro_batches):
            pipe.dispatch(b, x, idx)
            pipe.combine(b, y, idx, wt, outs[b % 2])
        pipe.join()

    def timed(run):
        cur = torch.cuda.current_stream()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        run()
        b_.record(cur)
        torch.cuda.synchronize()
        return round(a.elapsed_time(b_) * 1e3 / micro_batches, 3)

    res = {}
    for name, fn in (("serial", serial), ("pipelined", pipelined)):
        fn()  # warm-up
        torch.cuda.synchronize()
        res[f"{name}_us_per_microbatch_eager"] = timed(fn)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        graph.replay()
        torch.cuda.synchronize()
        res[f"{name}_us_per_microbatch"] = timed(graph.replay)
        del graph
    res["micro_batches"] = micro_batches
    res["note"] = ("micro-batch b uses buffer set b % 2; pipelined: dispatches on one stream, combines on another, "
                   "b+1's dispatch overlapping b's combine; no L2 flush between micro-batches; *_us_per_microbatch: "
                   "the schedule replayed from a CUDA graph; *_eager: issued from Python call by call")
    return res


def run_signaled(args, llmoe, w, x, idx, rb, es, flush, steps: int = 200):
    """Dispatch plus unpack (received rows in the experts' input order): two
    launches (llmoe_dispatch, llmoe_unpack); the dispatch that writes the rows
    itself (llmoe_dispatch_unpack, one launch); and one cooperative launch
    whose CTAs signal each other through the count words
    (llmoe_dispatch_signaled, bounded waits).  L2 flushed before each."""
    import torch

    rows = w.E * w.R * w.T
    recv_x = torch.empty((rows, w.H), dtype=torch.float32 if es == 4 else torch.int16, device="cuda")
    recv_src = torch.empty((rows,), dtype=torch.int32, device="cuda")
    bs = rb.buf_set(0, w.K)
    ws = torch.zeros(llmoe.llmoe_signal_workspace_bytes(bs) // 4, dtype=torch.int32, device="cuda")
    cur = torch.cuda.current_stream()

    def two_launches():
        llmoe.llmoe_dispatch(x, idx, bs, cur)
        llmoe.llmoe_unpack(recv_x, recv_src, bs, cur)

    def one_launch():
        llmoe.llmoe_dispatch_signaled(x, idx, recv_x, recv_src, ws, 2_000_000_000, bs, cur)

    def with_rows():
        llmoe.llmoe_dispatch_unpack(x, idx, recv_x, recv_src, bs, cur)

    res = {}
    for name, fn in (("dispatch_then_unpack_us", two_launches), ("dispatch_unpack_us", with_rows),
                     ("signaled_us", one_launch)):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps + 3):
            flush()
            llmoe.llmoe_clean(bs, cur)
            if i >= 3:
                evs[i - 3][0].record(cur)
            fn()
            if i >= 3:
                evs[i - 3][1].record(cur)
        torch.cuda.synchronize()
        res[name] = round(statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3, 3)
    res["steps"] = steps
    res["note"] = ("events around the dispatch (+ unpack) only; the clean before each is outside; "
                   "dispatch_unpack: one launch that writes the messages, the counts and the experts' input rows; "
                   "signaled: one cooperative launch, consumers wait on the count words with a clock limit")
    return res


def pack_e2e_input(inp):
    """x, topk_idx and topk_w of one step laid end to end in one pinned host
    buffer (uint8), the layout the e2e step uploads in one copy."""
    import torch

    parts = [np.ascontiguousarray(inp[k]).view(np.uint8).reshape(-1) for k in ("x", "topk_idx", "topk_w")]
    hin = torch.empty(sum(p.size for p in parts), dtype=torch.uint8).pin_memory()
    off = 0
    for p in parts:
        hin[off:off + p.size].copy_(torch.from_numpy(p))
        off += p.size
    return hin


def run_e2e(args, llmoe, w, inp, dense_y, rb, tokens, stream):
    """Rounds through the C ABI with host buffers, per step: the inputs copied
    from pinned host memory, the result (the combine output) read back.

    e2e: one MoE layer with identity experts.  x, topk_idx and topk_w sit in
    one pinned host buffer and go up in one copy; llmoe_dispatch_unpack (set
    0) writes the messages and counts and lays the received rows out as the
    experts' input, in the receive-row order the combine reads its expert
    outputs in, and an identity expert's output is its input, so those rows
    are the combine's y; llmoe_combine (set 1) returns bf16(sum_k w_k x) per
    token, and the output comes back in one copy.
    e2e_dense_y: the bench round (dispatch + combine) with the dense expert
    outputs y [E*R*T, H] also copied from the host every step."""
    import torch

    x, idx, wts = inp["x"], inp["topk_idx"], inp["topk_w"]
    x_b, idx_b, w_b = x.nbytes, idx.nbytes, wts.nbytes  # x: whole 16-byte rows; idx: 8-byte words
    hin = pack_e2e_input(inp)
    din = torch.empty_like(hin, device="cuda")
    pay = torch.float32 if rb.msg_bytes - 4 == 4 * w.H else torch.int16
    dx = din[:x_b].view(pay).view(w.R, tokens, w.H)
    didx = din[x_b:x_b + idx_b].view(torch.int64).view(w.R, tokens, w.K)
    dw = din[x_b + idx_b:].view(torch.float32).view(w.R, tokens, w.K)
    hout = torch.empty((w.R, tokens, w.H), dtype=pay).pin_memory()
    dout = torch.empty_like(hout, device="cuda")
    rows = w.E * w.R * w.T
    recv_x = torch.empty((rows, w.H), dtype=pay, device="cuda")
    recv_src = torch.empty((rows,), dtype=torch.int32, device="cuda")
    F = llmoe.LLMOE_FLAG_CLEAN_OTHER_SET
    bs0 = rb.buf_set(0, w.K, flags=F)
    bs1 = rb.buf_set(1, w.K, flags=F | llmoe.LLMOE_FLAG_INPUTS_READY)
    d2h = hout.numel() * hout.element_size()

    def layer():
        din.copy_(hin, non_blocking=True)
        llmoe.llmoe_dispatch_unpack(dx, didx, recv_x, recv_src, bs0, stream)
        llmoe.llmoe_combine(recv_x, didx, dw, dout, bs1, stream)
        hout.copy_(dout, non_blocking=True)

    def timed(step):
        llmoe.llmoe_clean(rb.buf_set(0, w.K), stream)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        n = max(3, args.e2e_steps)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3, n

    us, n = timed(layer)
    serial = {"value": round(us, 2), "unit": "us/round", "steps": n,
              "note": "the same layer with each step's copies and kernels one after another on one stream"}
    pipe = run_e2e_pipelined(args, llmoe, w, [hin], [hout], rb, tokens, stream)
    ceil = copy_ceiling(hin, hout)
    res = {"value": pipe["value"], "unit": "us/round", "h2d_bytes_per_step": hin.numel(),
           "d2h_bytes_per_step": d2h, "steps": pipe["steps"], "launches_per_step": 2,
           "note": "one MoE layer with identity experts through the C ABI, steps back to back: x, topk_idx, topk_w "
                   "copied host->device in one copy from one pinned buffer; llmoe_dispatch_unpack (the messages, "
                   "counts and the experts' input rows, which identity experts return as their output y); "
                   "llmoe_combine over them; the output copied back.  Uploads and downloads run on their own streams into double "
                   "buffers, so step i+1's upload and step i-1's download overlap step i's kernels; value = time "
                   "from the first upload to the last download / steps",
           "serial": serial, "copy_ceiling": ceil,
           "copy_gbs": round((hin.numel() + d2h) / (pipe["copy_us_per_step"] * 1e3), 1)}
    del recv_x, recv_src
    if not args.no_e2e_dense_y:
        hy = torch.from_numpy(dense_y(inp).view(np.int16) if pay == torch.int16 else dense_y(inp)).pin_memory()
        dy = torch.empty_like(hy, device="cuda")

        def round_dense_y():
            din.copy_(hin, non_blocking=True)
            dy.copy_(hy, non_blocking=True)
            llmoe.llmoe_dispatch(dx, didx, bs0, stream)
            llmoe.llmoe_combine(dy, didx, dw, dout, bs1, stream)
            hout.copy_(dout, non_blocking=True)

        us2, n2 = timed(round_dense_y)
        res["dense_y"] = {"value": round(us2, 2), "unit": "us/round",
                          "h2d_bytes_per_step": hin.numel() + hy.numel() * hy.element_size(),
                          "d2h_bytes_per_step": d2h, "steps": n2,
                          "note": "the bench round with the dense expert outputs y [E*R*T, H] also copied "
                                  "host->device every step"}
    return res


def copy_ceiling(hin, hout, reps: int = 20) -> dict:
    """Pinned host <-> device copy rates of the e2e step's sizes, each copy
    alone on the current stream (CUDA events, mean of `reps`)."""
    import torch

    din = torch.empty_like(hin, device="cuda")
    dout = torch.empty_like(hout, device="cuda")
    cur = torch.cuda.current_stream()
    res = {}
    for name, dst, src in (("h2d", din, hin), ("d2h", hout, dout)):
        dst.copy_(src, non_blocking=True)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in evs:
            a.record(cur)
            dst.copy_(src, non_blocking=True)
            b.record(cur)
        torch.cuda.synchronize()
        us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
        nbytes = src.numel() * src.element_size()
        res[name] = {"us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1), "bytes": nbytes}
    # both directions at once, each on its own stream, as the e2e steps run them
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    for s in (s_up, s_down):
        s.wait_event(a)
    for _ in range(reps):
        with torch.cuda.stream(s_up):
            din.copy_(hin, non_blocking=True)
        with torch.cuda.stream(s_down):
            hout.copy_(dout, non_blocking=True)
    for s in (s_up, s_down):
        cur.wait_stream(s)
    b.record(cur)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / reps
    nbytes = hin.numel() * hin.element_size() + dout.numel() * dout.element_size()
    res["both"] = {"us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1), "bytes": nbytes,
                   "note": "one upload and one download at once per pair, on two streams"}
    return res


def run_e2e_pipelined(args, llmoe, w, hins, houts, rb, tokens, stream):
    """The e2e layer, steps back to back with their copies overlapped; step i
    uploads hins[i % len(hins)] and downloads into houts[i % len(houts)]
    (pinned host buffers of one size each).  Step i's upload (its own stream,
    into input buffer i % 2) waits only for the kernels of step i-2 that read
    that buffer; step i's kernels wait for its upload and for the download of
    step i-2 from output buffer i % 2; step i's download (its own stream)
    waits for its kernels.  The kernels stay on one stream in order:
    consecutive steps share the rank buffers, and one stream keeps each
    kernel's launch behind its predecessor's drain (programmatic dependent
    launch) with the cleans fused into the data kernels.  Kernels of
    consecutive steps on two streams, each step on its own buffer set, took
    108 us a layer against 103-105 with this schedule (both with dispatch
    then unpack): the cleans that schedule needs, and launches no longer
    hidden behind a predecessor, cost more than the overlap gained."""
    import torch

    hin, hout = hins[0], houts[0]
    x_b = w.R * tokens * w.H * (hout.element_size())
    idx_b = w.R * tokens * w.K * 8
    pay = hout.dtype
    din = [torch.empty_like(hin, device="cuda") for _ in (0, 1)]
    dout = [torch.empty((w.R, tokens, w.H), dtype=pay, device="cuda") for _ in (0, 1)]
    rows = w.E * w.R * w.T
    recv_x = torch.empty((rows, w.H), dtype=pay, device="cuda")
    recv_src = torch.empty((rows,), dtype=torch.int32, device="cuda")
    F = llmoe.LLMOE_FLAG_CLEAN_OTHER_SET
    bs0 = rb.buf_set(0, w.K, flags=F)
    bs1 = rb.buf_set(1, w.K, flags=F | llmoe.LLMOE_FLAG_INPUTS_READY)
    views = []
    for d in din:
        views.append((d[:x_b].view(pay).view(w.R, tokens, w.H), d[x_b:x_b + idx_b].view(torch.int64).view(w.R, tokens, w.K),
                      d[x_b + idx_b:].view(torch.float32).view(w.R, tokens, w.K)))
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    up_done = [torch.cuda.Event() for _ in (0, 1)]
    comp_done = [torch.cuda.Event() for _ in (0, 1)]
    down_done = [torch.cuda.Event() for _ in (0, 1)]

    def run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(comp_done[b])
                din[b].copy_(hins[i % len(hins)], non_blocking=True)
                up_done[b].record(s_up)
            stream.wait_event(up_done[b])
            if i >= 2:
                stream.wait_event(down_done[b])
            dx, didx, dw = views[b]
            llmoe.llmoe_dispatch_unpack(dx, didx, recv_x, recv_src, bs0, stream)
            llmoe.llmoe_combine(recv_x, didx, dw, dout[b], bs1, stream)
            comp_done[b].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(comp_done[b])
                houts[i % len(houts)].copy_(dout[b], non_blocking=True)
                down_done[b].record(s_down)

    for s in (s_up, s_down):
        s.wait_stream(stream)
    llmoe.llmoe_clean(rb.buf_set(0, w.K), stream)
    run(4)
    torch.cuda.synchronize()
    n = max(4, args.e2e_steps)
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    stream.wait_event(a)
    run(n)
    s_down.wait_event(comp_done[(n - 1) % 2])
    b_.record(s_down)
    torch.cuda.synchronize()
    us = a.elapsed_time(b_) * 1e3 / n
    # the copies alone, as this schedule issues them (for the overlap achieved),
    # into a host buffer of their own so the steps' outputs stay as they are
    hscratch = torch.empty_like(hout).pin_memory()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for i in range(n):
        din[i % 2].copy_(hin, non_blocking=True)
        hscratch.copy_(dout[i % 2], non_blocking=True)
    c1.record(stream)
    torch.cuda.synchronize()
    return {"value": round(us, 2), "steps": n, "copy_us_per_step": c0.elapsed_time(c1) * 1e3 / n}


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
