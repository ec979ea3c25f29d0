"""Where a dispatch or combine launch spends its time: a phase budget.

Builds the phase-trace variant of the library (-DLLMOE_PHASE_TRACE=1: the
same kernels with timer stamps at fixed points of every CTA's prologue and
data phase), runs each kernel alone after the bench's L2 flush, and prints
per workload, in microseconds:

- the kernel as CUDA events see it (launch, run, drain);
- the span from the first CTA's entry to the last CTA's exit (globaltimer);
- for each phase, the time from a CTA's own entry to that phase: median and
  maximum over the CTAs, median over steps;
- when the CTAs entered and left, relative to the first CTA's entry;
- two reference kernels launched the same way: an empty one, and one whose
  single thread per CTA loads one word (its stamps give the load latency).

Each kernel is measured after the bench's L2 flush ("flush"), after the
flush and a call of the same kernel on a tiny separate problem, which brings
the kernel's code back into L2 but none of this call's data ("warm-code"),
and back to back ("no-flush").

Usage (one GPU):
    python -m combine_routing_count_prefix_gb300.phase_budget [--workloads tiny,many_small,dsv3] [--steps 30]

The stamps themselves cost a few global stores per CTA; the normal build has
none of them.
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PHASES = {
    "dispatch": ["entry", "prior grid done", "route histogram built (consumer warps)", "destinations packed",
                 "consumers start (after the early wait)", "first chunk in shared memory", "consumer warp done",
                 "exit"],
    "combine": ["entry", "prior grid done (not early)", "route histogram built", "row table ready",
                "prior grid done (early)", "first unit stored", "all units stored", "exit"],
}
NPH = 8  # stamps per CTA and kind (globaltimer, then clock64)
SM_MHZ = 2070  # the GB300's maximum SM clock, for the cycle stamps
FLUSH_BYTES = 512 << 20
FLUSH_READ_BYTES = 256 << 20


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workloads", default="tiny,many_small,skewed,dsv3")
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--modes", default="flush,warm-code,no-flush")
    ap.add_argument("--dump", default="", help="directory for every CTA's stamps (an .npz per workload and mode)")
    args = ap.parse_args(argv)

    from combine_routing_count_prefix_gb300 import build as cuda_build

    # LLMOE_TRACE_LIBRARY: an already built trace library (e.g. a variant
    # compiled with other tuning macros); by default the in-tree trace build
    os.environ["LLMOE_LIBRARY"] = os.environ.get("LLMOE_TRACE_LIBRARY") or cuda_build.build(trace=True)
    import ctypes

    import torch

    from combine_routing_count_prefix_gb300 import llmoe
    from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs

    lib = llmoe._lib
    lib.llmoe_phase_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.llmoe_phase_trace_clear.argtypes = [ctypes.c_void_p]
    lib.llmoe_trace_empty.argtypes = [ctypes.c_int, ctypes.c_void_p]
    lib.llmoe_trace_load.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    max_ctas = 65536  # trace rows: the dispatch's CTAs, then the combine's from max_ctas / 2
    host = np.zeros((max_ctas, 2 * NPH), dtype=np.uint64)

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    flush_w = torch.empty(FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")
    flush_r = torch.ones(FLUSH_READ_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def traced(launch, steps, mode="flush", warm=None):
        """Events around `launch`; the stamps of every step.  mode "flush":
        the bench's L2 flush before each step; "warm-code": the flush, then
        `warm()` (the same kernel on a tiny separate problem, which brings the
        kernel's code back into L2 but not this call's data); "no-flush":
        back-to-back steps."""
        ev_us, stamps = [], []
        for i in range(steps + 2):
            if mode != "no-flush":
                flush()
            if mode == "warm-code":
                warm()
            llmoe._check(lib.llmoe_phase_trace_clear(sp), "llmoe_phase_trace_clear")
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch()
            b.record(stream)
            torch.cuda.synchronize()
            if i < 2:
                continue  # warm-up
            ev_us.append(a.elapsed_time(b) * 1e3)
            llmoe._check(lib.llmoe_phase_trace_read(host.ctypes.data, max_ctas), "llmoe_phase_trace_read")
            half = host[:max_ctas // 2], host[max_ctas // 2:]  # dispatch rows, combine rows
            stamps.append(tuple(h[h[:, 0] != 0].astype(np.int64).copy() for h in half))  # the CTAs that stamped
        return ev_us, stamps

    def summarize(name, phases, ev_us, stamps):
        """Means over steps (event times have a coarse tick; the flush between
        steps puts each step at a random phase of it, so means dither)."""
        mean = statistics.mean
        spans, enters, exits = [], [], []
        per_phase = {p: ([], [], []) for p in range(NPH)}
        for s in stamps:
            gt, cy = s[:, :NPH], s[:, NPH:]
            entry = gt[:, 0]
            t0 = entry.min()
            last = np.where(gt[:, NPH - 1] > 0, gt[:, NPH - 1], gt.max(axis=1))
            spans.append((last.max() - t0) / 1e3)
            enters.append(((entry - t0).max()) / 1e3)
            exits.append((np.median(last - t0) / 1e3, (last.max() - t0) / 1e3))
            for p in range(1, NPH):
                ok = gt[:, p] > 0
                if ok.any():
                    d = (gt[ok, p] - entry[ok]) / 1e3
                    c = (cy[ok, p] - cy[ok, 1]) / SM_MHZ + (gt[ok, 1] - gt[ok, 0]) / 1e3  # slot 0 holds the SM id
                    per_phase[p][0].append(float(np.median(d)))
                    per_phase[p][1].append(float(d.max()))
                    per_phase[p][2].append(float(np.median(c)))
        ncta = stamps[0].shape[0] if stamps else 0
        print(f"\n### {name}: {ncta} CTAs, {len(ev_us)} steps")
        print(f"- CUDA events around the launch: mean {mean(ev_us):.2f} us (min {min(ev_us):.2f})")
        print(f"- first CTA entry -> last CTA exit: {mean(spans):.2f} us; launch + drain outside it: "
              f"{mean(ev_us) - mean(spans):.2f} us")
        print(f"- last CTA entry after the first: {mean(enters):.2f} us; CTA exits after the first entry: "
              f"median CTA {mean([e[0] for e in exits]):.2f}, last {mean([e[1] for e in exits]):.2f} us")
        print(f"\n| phase | from CTA entry, median CTA (us) | slowest CTA (us) | median CTA, SM cycles at "
              f"{SM_MHZ} MHz from phase 1, plus phase 1 (us) |")
        print("|---|---|---|---|")
        order = sorted((p for p in range(1, NPH) if per_phase[p][0]), key=lambda p: statistics.mean(per_phase[p][0]))
        for p in order:
            a, b, c = per_phase[p]
            if a:
                print(f"| {phases[p]} | {mean(a):.2f} | {mean(b):.2f} | {mean(c):.2f} |")

    def timeline(name, ev_us, stamps):
        """One round on one clock: times relative to the dispatch's first CTA
        entry, means over steps."""
        mean = statistics.mean
        rows = {k: [] for k in ("d_last_entry", "d_exit_med", "d_exit_last", "c_first_entry", "c_entry_med",
                                "c_wait_min", "c_wait_med", "c_first_unit_med", "c_done_med", "c_exit_last")}
        for d, c in stamps:
            t0 = d[:, 0].min()
            rel = lambda v: (v - t0) / 1e3
            d_exit = d[:, NPH - 1]
            rows["d_last_entry"].append(rel(d[:, 0].max()))
            rows["d_exit_med"].append(rel(np.median(d_exit)))
            rows["d_exit_last"].append(rel(d_exit.max()))
            rows["c_first_entry"].append(rel(c[:, 0].min()))
            rows["c_entry_med"].append(rel(np.median(c[:, 0])))
            rows["c_wait_min"].append(rel(c[:, 4].min()))
            rows["c_wait_med"].append(rel(np.median(c[:, 4])))
            rows["c_first_unit_med"].append(rel(np.median(c[:, 5][c[:, 5] > 0])))
            rows["c_done_med"].append(rel(np.median(c[:, 6])))
            rows["c_exit_last"].append(rel(c[:, NPH - 1].max()))
        r = {k: mean(v) for k, v in rows.items()}
        print(f"\n### {name}: {len(ev_us)} steps\n- CUDA events around the round: mean {mean(ev_us):.2f} us; "
              f"first dispatch CTA entry -> last combine CTA exit: {r['c_exit_last']:.2f} us; outside it: "
              f"{mean(ev_us) - r['c_exit_last']:.2f} us")
        print("\n| event (from the first dispatch CTA's entry) | us |\n|---|---|")
        for k, label in (("d_last_entry", "last dispatch CTA entered"), ("d_exit_med", "median dispatch CTA exit"),
                         ("d_exit_last", "last dispatch CTA exit"), ("c_first_entry", "first combine CTA entered"),
                         ("c_entry_med", "median combine CTA entered"),
                         ("c_wait_min", "first combine CTA past its wait for the dispatch"),
                         ("c_wait_med", "median combine CTA past its wait"),
                         ("c_first_unit_med", "median combine CTA's first unit stored"),
                         ("c_done_med", "median combine CTA done"), ("c_exit_last", "last combine CTA exit")):
            print(f"| {label} | {r[k]:.2f} |")

    # reference kernels
    cold = torch.ones(2048 * 4096, dtype=torch.int64, device="cuda")
    sink = torch.empty(2048, dtype=torch.int64, device="cuda")
    for ctas in (1, 1024):
        for mode in ("flush", "no-flush"):
            ev, st = traced(lambda: llmoe._check(lib.llmoe_trace_empty(ctas, sp), "llmoe_trace_empty"), args.steps,
                            mode)
            print(f"\n### empty kernel, {ctas} CTAs, {mode}\n- CUDA events: mean {statistics.mean(ev):.2f} us")
            ev, st = traced(lambda: llmoe._check(lib.llmoe_trace_load(cold.data_ptr(), sink.data_ptr(), ctas, sp),
                                                 "llmoe_trace_load"), args.steps, mode)
            lat = [float(np.median((s[0][:, 1] - s[0][:, 0]) / 1e3)) for s in st]
            print(f"\n### one load per CTA, {ctas} CTAs, {mode}\n- CUDA events: mean {statistics.mean(ev):.2f} us; "
                  f"load latency (median CTA): {statistics.mean(lat):.2f} us")

    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    def problem(w):
        inp = make_inputs(w, seed=0)
        p = {"x": dev(inp["x"]), "idx": dev(inp["topk_idx"]), "wt": dev(inp["topk_w"]),
             "y": dev(inp["y_pool"]).index_select(0, dev(inp["y_row_map"])).contiguous(),
             "out": torch.empty((w.R, w.T, w.H), dtype=torch.int16, device="cuda"),
             "rb": llmoe.RankBuffers(w.T, w.H, w.R, w.E, fill=0)}
        F = llmoe.LLMOE_FLAG_CLEAN_OTHER_SET
        p["bs0"] = p["rb"].buf_set(0, w.K, flags=F)
        p["bs1"] = p["rb"].buf_set(1, w.K, flags=F | llmoe.LLMOE_FLAG_INPUTS_READY)
        llmoe.llmoe_clean(p["rb"].buf_set(0, w.K))
        return p

    tiny = problem(WORKLOADS["tiny"])
    warm_dispatch = lambda: llmoe.llmoe_dispatch(tiny["x"], tiny["idx"], tiny["bs0"], stream)
    warm_combine = lambda: llmoe.llmoe_combine(tiny["y"], tiny["idx"], tiny["wt"], tiny["out"], tiny["bs1"], stream)
    for wname in args.workloads.split(","):
        w = WORKLOADS[wname]
        p = problem(w)
        print(f"\n## {wname}: {w.describe()}")
        for mode in args.modes.split(","):
            ev, st = traced(lambda: llmoe.llmoe_dispatch(p["x"], p["idx"], p["bs0"], stream), args.steps, mode,
                            warm_dispatch)
            summarize(f"dispatch_kernel, {mode}", PHASES["dispatch"], ev, [x[0] for x in st])
            ev, st = traced(lambda: llmoe.llmoe_combine(p["y"], p["idx"], p["wt"], p["out"], p["bs1"], stream),
                            args.steps, mode, warm_combine)
            summarize(f"combine_kernel (LLMOE_FLAG_INPUTS_READY), {mode}", PHASES["combine"], ev,
                      [x[1] for x in st])

            def round_():
                llmoe.llmoe_dispatch(p["x"], p["idx"], p["bs0"], stream)
                llmoe.llmoe_combine(p["y"], p["idx"], p["wt"], p["out"], p["bs1"], stream)

            ev, st = traced(round_, args.steps, mode, lambda: (warm_dispatch(), warm_combine()))
            timeline(f"round (dispatch + combine, as the bench times it), {mode}", ev, st)
            if args.dump:
                os.makedirs(args.dump, exist_ok=True)
                # per step: [CTA, 2 * NPH] stamps (globaltimer phases, then SM cycles; cycle slot 0 = SM id)
                np.savez_compressed(os.path.join(args.dump, f"round_{wname}_{mode}.npz"),
                                    **{f"dispatch_{i}": d for i, (d, _) in enumerate(st)},
                                    **{f"combine_{i}": c for i, (_, c) in enumerate(st)})
        del p
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
