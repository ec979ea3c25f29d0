"""Each C-ABI call of the library, a few times, for a kernel profiler.

Runs the calls named by --calls on one workload, --reps times each, with the
L2 flushed (a 512 MB write, then a 256 MB read) before every call, so each
launch starts from cold caches as the bench's do.  Meant to run under
``ncu -k <kernel> -c <n>``: every kernel of the library is launched here a
known, small number of times, on a workload small enough that a capture of
all its sections ends quickly (dense16: 2.35 GB on the device).

    python -m combine_routing_count_prefix_gb300.profile_calls --workload dense16 \\
        --calls route,clean,dispatch,combine,unpack,signaled,staged,dispatch_unpack --reps 3

Kernels per call: route -> route_kernel; clean -> clean_kernel; dispatch ->
dispatch_kernel<false>; dispatch_unpack -> dispatch_kernel<true> (the dispatch
that also writes the experts' input rows); combine -> combine_kernel<payload type>; unpack ->
unpack_balanced_kernel (fewer buckets than routed entries) or unpack_kernel
(otherwise, e.g. many_small); signaled -> dispatch_signaled_kernel; staged ->
combine_put_kernel, then combine_reduce_ring_kernel (more (token, chunk) units
than consumer warps in a full wave, e.g. dense16) or combine_reduce_kernel.  Each call that reads a dispatch's
results gets one, outside the flush.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FLUSH_BYTES = 512 << 20
FLUSH_READ_BYTES = 256 << 20


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="dense16")
    ap.add_argument("--calls", default="route,clean,dispatch,combine,unpack,signaled,staged,dispatch_unpack")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)

    import torch

    from combine_routing_count_prefix_gb300 import build

    build.build()
    from combine_routing_count_prefix_gb300 import llmoe
    from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs

    torch.cuda.set_device(0)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=0)
    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    x, idx, wt = dev(inp["x"]), dev(inp["topk_idx"]), dev(inp["topk_w"])
    y = dev(inp["y_pool"]).index_select(0, dev(inp["y_row_map"])).contiguous()
    out = torch.empty((w.R, w.T, w.H), dtype=torch.int16, device="cuda")
    rb = llmoe.RankBuffers(w.T, w.H, w.R, w.E, fill=0)
    bs0, bs1 = rb.buf_set(0, w.K), rb.buf_set(1, w.K)
    flush_w = torch.empty(FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")
    flush_r = torch.ones(FLUSH_READ_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        flush_w.zero_()
        flush_r.sum()

    rows = w.E * w.R * w.T
    recv_x = recv_src = ws = slot = counts = None
    calls = args.calls.split(",")
    if "unpack" in calls or "signaled" in calls or "dispatch_unpack" in calls:
        recv_x = torch.empty((rows, w.H), dtype=torch.int16, device="cuda")
        recv_src = torch.empty((rows,), dtype=torch.int32, device="cuda")
        ws = torch.zeros(llmoe.llmoe_signal_workspace_bytes(bs0) // 4, dtype=torch.int32, device="cuda")
    if "route" in calls:
        slot = torch.empty((w.R, w.T, w.K), dtype=torch.int32, device="cuda")
        counts = torch.empty((w.E, w.R), dtype=torch.int64, device="cuda")

    def dispatched():
        llmoe.llmoe_clean(bs0)
        llmoe.llmoe_dispatch(x, idx, bs0)

    for name in calls:
        for _ in range(args.reps):
            if name == "route":
                flush()
                llmoe.llmoe_route(idx, slot, counts, bs0)
            elif name == "clean":
                flush()
                llmoe.llmoe_clean(bs0)
            elif name == "dispatch":
                llmoe.llmoe_clean(bs0)
                flush()
                llmoe.llmoe_dispatch(x, idx, bs0)
            elif name == "combine":
                llmoe.llmoe_clean(bs1)
                flush()
                llmoe.llmoe_combine(y, idx, wt, out, bs1)
            elif name == "unpack":
                dispatched()
                flush()
                llmoe.llmoe_unpack(recv_x, recv_src, bs0)
            elif name == "dispatch_unpack":
                llmoe.llmoe_clean(bs0)
                flush()
                llmoe.llmoe_dispatch_unpack(x, idx, recv_x, recv_src, bs0)
            elif name == "signaled":
                llmoe.llmoe_clean(bs0)
                flush()
                llmoe.llmoe_dispatch_signaled(x, idx, recv_x, recv_src, ws, 2_000_000_000, bs0)
            elif name == "staged":
                llmoe.llmoe_clean(bs1)
                flush()
                llmoe.llmoe_combine_staged(y, idx, wt, out, bs1)
            else:
                raise SystemExit(f"unknown call {name}")
    torch.cuda.synchronize()
    print(f"profile_calls: {args.workload}: {','.join(calls)} x {args.reps}")


if __name__ == "__main__":
    main()
