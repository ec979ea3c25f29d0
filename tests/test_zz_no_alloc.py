"""The allocation-free signaled dispatch (llmoe_dispatch_signaled_static).

Callers that cannot allocate device memory at the call (a plugin given only
raw pointers by a framework that owns all allocations, or a latency-critical
loop that must not cudaMalloc) use this variant: its workspace is a fixed
array inside the library.  This file sorts last so that a run stopping at the
first failure has run every other test; it also passes on its own.  Its
results must equal those of llmoe_dispatch_signaled with a caller-allocated
workspace, bit for bit, on two calls in a row, and the CPU oracle's
messages, counts and unpacked rows.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from combine_routing_count_prefix_gb300 import build

    build.build()
    from combine_routing_count_prefix_gb300 import llmoe

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    oracle.build()
    return llmoe


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()


def outputs(L, w):
    rb = L.RankBuffers(w.T, w.H, w.R, w.E, guard=256, fill=0xA5)
    rows = w.E * w.R * w.T
    recv_x = torch.full((rows, w.H), 0x7FC1, dtype=torch.int16, device="cuda")
    recv_src = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")  # returned: the buf set points at it
    return rb, rb.buf_set(0, w.K, err=err), recv_x, recv_src, err


@pytest.mark.parametrize("name", ["skewed", "dsv3"])
def test_static_workspace_matches_caller_workspace(L, name):
    w = WORKLOADS[name]
    rb_a, bs_a, rx_a, rs_a, err_a = outputs(L, w)  # caller-allocated workspace
    rb_b, bs_b, rx_b, rs_b, err_b = outputs(L, w)  # the library's fixed workspace
    ws = torch.zeros(L.llmoe_signal_workspace_bytes(bs_a) // 4, dtype=torch.int32, device="cuda")
    for call in range(2):  # two calls in a row, on different inputs
        inp = make_inputs(w, seed=90 + call)
        x, idx = dev(inp["x"]), dev(inp["topk_idx"])
        for t in (rs_a, rs_b):
            t.fill_(-7)
        L.llmoe_clean(bs_a)
        L.llmoe_dispatch_signaled(x, idx, rx_a, rs_a, ws, 2_000_000_000, bs_a)
        L.llmoe_clean(bs_b)
        L.llmoe_dispatch_signaled_static(x, idx, rx_b, rs_b, 2_000_000_000, bs_b)
        torch.cuda.synchronize()
        assert L.llmoe_get_error(bs_a) == 0 and L.llmoe_get_error(bs_b) == 0
        assert torch.equal(rx_a, rx_b), f"call {call}: unpacked rows differ"
        assert torch.equal(rs_a, rs_b), f"call {call}: source tokens differ"
        assert torch.equal(rb_a.storage, rb_b.storage), f"call {call}: rank buffers differ"
        assert (rs_b >= 0).sum().item() == int((inp["topk_idx"] >= 0).sum())
        check_against_oracle(rb_b, rx_b, rs_b, inp, w)


def check_against_oracle(rb, recv_x, recv_src, inp, w):
    """Messages, count words and unpacked rows equal the CPU oracle's."""
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, num_max_tokens=w.T)
    got = rb.recv_rows(0)[dev(d["row_rank"]), dev(d["row_index"])].cpu().numpy()
    assert np.array_equal(got, d["msgs"]), "dispatch messages differ from the oracle"
    assert np.array_equal(rb.signal_words(0).cpu().numpy(), d["count_words"]), "count words differ"
    u = oracle.unpack(inp["x"], inp["topk_idx"], w.E, num_max_tokens=w.T)
    rows = u["rows"]
    gx, gs = recv_x.cpu().numpy(), recv_src.cpu().numpy()
    assert np.array_equal(gx[rows].view(np.uint16), u["recv_x"][rows]), "unpacked rows differ from the oracle"
    assert np.array_equal(gs[rows], u["recv_src"][rows]), "unpacked source tokens differ from the oracle"


@pytest.mark.parametrize("name", ["skewed", "dsv3"])
def test_static_workspace_matches_oracle_after_a_timed_out_call(L, name):
    """A call whose consumers give up at once (a one-cycle spin limit, so most
    of them time out), then a normal call: the second call's results are the
    oracle's, whatever the first left behind."""
    w = WORKLOADS[name]
    rb, bs, recv_x, recv_src, err = outputs(L, w)
    inp = make_inputs(w, seed=93)
    x, idx = dev(inp["x"]), dev(inp["topk_idx"])
    L.llmoe_clean(bs)
    L.llmoe_dispatch_signaled_static(x, idx, recv_x, recv_src, 1, bs)
    torch.cuda.synchronize()
    assert L.llmoe_get_error(bs, reset=True) in (L.LLMOE_DEV_OK, L.LLMOE_DEV_TIMEOUT)
    recv_src.fill_(-7)
    L.llmoe_clean(bs)
    L.llmoe_dispatch_signaled_static(x, idx, recv_x, recv_src, 2_000_000_000, bs)
    torch.cuda.synchronize()
    assert L.llmoe_get_error(bs) == 0
    check_against_oracle(rb, recv_x, recv_src, inp, w)


def test_static_workspace_rejects_too_many_ranks(L):
    # rejected on the host before anything is queued (the pointers are never
    # dereferenced)
    w = WORKLOADS["tiny"].with_(R=L.LLMOE_STATIC_MAX_RANKS + 1, E=L.LLMOE_STATIC_MAX_RANKS + 1, K=1, T=1, H=8)
    bs = L.llmoe_buf_set_t(base=1 << 20, rank_stride=1 << 20, num_max_tokens=w.T, num_tokens=w.T, hidden=w.H,
                           num_ranks=w.R, num_experts=w.E, num_topk=w.K, set=0, err=None, flags=0, dtype=0)
    A = 1 << 24
    with pytest.raises(L.LLMoEError) as ei:
        L.llmoe_dispatch_signaled_static(A, A, A, A, 1000, bs)
    assert ei.value.status == L.LLMOE_ERR_INVALID_ARGUMENT
