"""Two-stream double-buffered micro-batch schedule over the C-ABI calls.

LLMoEBufferLayout holds two buffer sets so that consecutive micro-batches do
not share buffers (LL_MoE_Buffers.hpp, "Two sets of LLMoEBuffer for double
buffering").  Here micro-batch b uses set b % 2 for both its dispatch and its
combine.  Dispatches run on one stream and combines on another, so micro-batch
b+1's dispatch (set (b+1) % 2) runs while micro-batch b's combine (set b % 2)
is still running.  CUDA events order what must be ordered:

- a combine waits for its own micro-batch's dispatch (the expert outputs it
  reads are computed from that dispatch's receive buffer);
- a dispatch waits for the combine that last used its set (two micro-batches
  earlier), because both write the same signal words;
- each call also waits for the work already enqueued on the caller's current
  stream (its inputs).

Each call is preceded by an llmoe_clean of its set on its own stream.  The
dispatch's counts are therefore zeroed before the combine of the same
micro-batch writes its flags, and whatever consumes the counts must be
enqueued, on the combine stream, before ``combine()`` is called.  The other
set is in use by the concurrent kernel, so this schedule never uses
LLMOE_FLAG_CLEAN_OTHER_SET.

This module only orders calls; every step of the data path runs in the
library's kernels.
"""
from __future__ import annotations

import torch

from . import llmoe


class DoubleBufferPipeline:
    def __init__(self, rank_buffers: "llmoe.RankBuffers", num_topk: int, num_tokens: int | None = None,
                 err=None, dispatch_stream: torch.cuda.Stream | None = None,
                 combine_stream: torch.cuda.Stream | None = None):
        self.rb = rank_buffers
        self.bs = [rank_buffers.buf_set(s, num_topk, num_tokens, err) for s in (0, 1)]
        self.sd = dispatch_stream or torch.cuda.Stream()
        self.sc = combine_stream or torch.cuda.Stream()
        self.dispatched = [torch.cuda.Event() for _ in (0, 1)]
        self.combined = [torch.cuda.Event() for _ in (0, 1)]
        self.used = [False, False]

    def dispatch(self, b: int, x, topk_idx, after=None) -> None:
        """Micro-batch b's dispatch into set b % 2, on the dispatch stream.
        `after()`, if given, is enqueued on the dispatch stream right after the
        dispatch (e.g. the expert kernels reading the receive rows and counts)."""
        s = b % 2
        self.sd.wait_stream(torch.cuda.current_stream())  # the caller's earlier work (e.g. x) comes first
        with torch.cuda.stream(self.sd):
            if self.used[s]:
                self.sd.wait_event(self.combined[s])
            llmoe.llmoe_clean(self.bs[s], self.sd)
            llmoe.llmoe_dispatch(x, topk_idx, self.bs[s], self.sd)
            if after is not None:
                after()
            self.dispatched[s].record(self.sd)
        self.used[s] = True

    def combine(self, b: int, y, topk_idx, topk_w, out, after=None) -> None:
        """Micro-batch b's combine on set b % 2, on the combine stream, after
        its dispatch.  `after()`, if given, is enqueued on the combine stream
        right after the combine (e.g. whatever reads the flag words)."""
        s = b % 2
        self.sc.wait_stream(torch.cuda.current_stream())  # the caller's earlier work (e.g. y) comes first
        with torch.cuda.stream(self.sc):
            self.sc.wait_event(self.dispatched[s])
            llmoe.llmoe_clean(self.bs[s], self.sc)
            llmoe.llmoe_combine(y, topk_idx, topk_w, out, self.bs[s], self.sc)
            if after is not None:
                after()
            self.combined[s].record(self.sc)

    def join(self, stream: torch.cuda.Stream | None = None) -> None:
        """Make `stream` (default: the current stream) wait for all issued work."""
        stream = stream or torch.cuda.current_stream()
        stream.wait_stream(self.sd)
        stream.wait_stream(self.sc)
