"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every test feeds the same seeded inputs to both.  Bars:
- dispatch: every written message (header + payload) and every recv-count
  word bit-exact; every other byte of the rank buffers untouched (canary);
- combine: every output element within 1 bf16 ulp (ordinal distance of the
  bit patterns <= 1) of the oracle, and in fact bit-exact since both sides
  round the same products and sums in the same order; flag words exact;
- route: slots and counts exact.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

CANARY = 0xA5
CANARY_WORD = int(np.array([0xA5A5A5A5A5A5A5A5], dtype=np.uint64).view(np.int64)[0])
OUT_CANARY = 0x7FC1  # a NaN pattern: an unwritten output element fails


@pytest.fixture(scope="module")
def L():
    from combine_routing_count_prefix_gb300 import build

    build.build()
    from combine_routing_count_prefix_gb300 import llmoe

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    oracle.build()
    return llmoe


def dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def y_dev(inp) -> torch.Tensor:
    pool = dev(inp["y_pool"])
    return pool.index_select(0, dev(inp["y_row_map"])).contiguous()


def ordinal(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def all_equal_chunked(t: torch.Tensor, value: int, chunk=1 << 31) -> bool:
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk):
        if not bool((flat[s:s + chunk] == value).all()):
            return False
    return True


def ulp_distance(got: np.ndarray, ref: np.ndarray, dtype: str) -> np.ndarray:
    """Ordinal distance between the bit patterns of two float arrays."""
    if dtype == "fp32":
        g, r = got.view(np.uint32).astype(np.int64), ref.view(np.uint32).astype(np.int64)
        og = np.where(g & 0x80000000, -(g & 0x7FFFFFFF), g)
        orf = np.where(r & 0x80000000, -(r & 0x7FFFFFFF), r)
        return np.abs(og - orf)
    return np.abs(ordinal(got.view(np.uint16)) - ordinal(ref.view(np.uint16)))


class Round:
    """One clean / dispatch / clean / combine round on fresh canary-filled buffers."""

    def __init__(self, L, w: Workload, seed=0, tokens=None, dispatch_set=0, inp=None, validate=True, dtype="bf16"):
        self.L, self.w, self.dtype = L, w, dtype
        self.inp = inp if inp is not None else make_inputs(w, seed=seed, tokens=tokens, dtype=dtype)
        self.T_call = self.inp["x"].shape[1]
        self.rb = L.RankBuffers(w.T, w.H, w.R, w.E, guard=256, fill=CANARY, dtype=dtype)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda") if validate else None
        self.ds, self.cs = dispatch_set, 1 - dispatch_set
        self.bs_d = self.rb.buf_set(self.ds, w.K, self.T_call, self.err)
        self.bs_c = self.rb.buf_set(self.cs, w.K, self.T_call, self.err)
        self.x, self.idx, self.wt = dev(self.inp["x"]), dev(self.inp["topk_idx"]), dev(self.inp["topk_w"])
        self.y = y_dev(self.inp)
        if dtype == "fp32":
            self.out = torch.full((w.R, self.T_call, w.H), float("nan"), dtype=torch.float32, device="cuda")
        else:
            self.out = torch.full((w.R, self.T_call, w.H), OUT_CANARY, dtype=torch.int16, device="cuda")

    def run(self):
        L = self.L
        L.llmoe_clean(self.bs_d)
        L.llmoe_dispatch(self.x, self.idx, self.bs_d)
        L.llmoe_clean(self.bs_c)
        L.llmoe_combine(self.y, self.idx, self.wt, self.out, self.bs_c)
        torch.cuda.synchronize()
        return self

    def error(self):
        return self.L.llmoe_get_error(self.bs_d) if self.err is not None else 0

    def check_dispatch(self, d=None):
        w, inp = self.w, self.inp
        if d is None:
            d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, num_max_tokens=w.T, dtype=self.dtype)
        recv = self.rb.recv_rows(self.ds)
        rr, ri = dev(d["row_rank"]), dev(d["row_index"])
        got = recv[rr, ri].cpu().numpy() if d["n"] else np.zeros((0, self.rb.msg_bytes), np.uint8)
        assert got.shape == d["msgs"].shape
        bad = np.nonzero((got != d["msgs"]).any(axis=1))[0]
        assert bad.size == 0, f"{bad.size} of {d['n']} messages differ; first at entry {bad[:5]}"
        assert np.array_equal(self.rb.signal_words(self.ds).cpu().numpy(), d["count_words"])
        return d

    def check_combine(self):
        w, inp = self.w, self.inp
        ref, flags = oracle.combine((inp["y_pool"], inp["y_row_map"]), inp["topk_idx"], inp["topk_w"], w.H, w.E,
                                    num_max_tokens=w.T, dtype=self.dtype)
        dist = ulp_distance(self.out.cpu().numpy(), ref, self.dtype)
        assert dist.max(initial=0) <= 1, f"max ulp distance {dist.max()}"
        assert int((dist != 0).sum()) == 0, f"{int((dist != 0).sum())} elements differ by 1 ulp"
        assert np.array_equal(self.rb.signal_words(self.cs).cpu().numpy(), flags)

    def check_canary(self, d):
        """Nothing outside the written messages and signal words changed."""
        recv = self.rb.recv_rows(self.ds)
        if d["n"]:
            recv[dev(d["row_rank"]), dev(d["row_index"])] = CANARY
        self.rb.signal_words(0).fill_(CANARY_WORD)
        self.rb.signal_words(1).fill_(CANARY_WORD)
        assert all_equal_chunked(self.rb.storage, CANARY)


def full_check(r: Round):
    r.run()
    assert r.error() == 0
    d = r.check_dispatch()
    r.check_combine()
    r.check_canary(d)


# ---------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "many_small"])
def test_workload_full_size(L, name):
    full_check(Round(L, WORKLOADS[name], seed=0))


def test_workload_large(L):
    w = WORKLOADS["large"]
    need = L.round_up(L.llmoe_layout_bytes(w.T, w.H, w.R, w.E) + 256, 256) * w.R + w.E * w.R * w.T * w.H * 2
    free, _ = torch.cuda.mem_get_info()
    assert free > need + (8 << 30), f"large workload needs {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free"
    full_check(Round(L, w, seed=0))


# ---------------------------------------------------------------------------
# shape sweep: odd hidden sizes (every row phase, partial warp chunks), one
# rank, many ranks, top-1 .. top-8, masks, fewer tokens than the layout
# ---------------------------------------------------------------------------

SWEEP = []
for R, Lx in [(1, 8), (2, 4), (32, 1), (3, 5)]:
    for K in (1, 2, 8):
        if K > R * Lx:
            continue
        for H in (8, 56, 264):
            for T in (1, 3, 37):
                SWEEP.append((R, R * Lx, K, H, T))


@pytest.mark.parametrize("R,E,K,H,T", SWEEP)
def test_shape_sweep(L, R, E, K, H, T):
    w = Workload("sweep", R, T, H, E, K, mask_p=0.3 if K > 1 else 0.0)
    full_check(Round(L, w, seed=R * 1000 + E * 10 + K + H + T))


@pytest.mark.parametrize("tokens", [0, 1, 5, 127])
def test_fewer_tokens_than_layout(L, tokens):
    w = WORKLOADS["dsv3"].with_(H=512)
    full_check(Round(L, w, seed=tokens, tokens=tokens))


def test_repeat_after_smaller_call_on_same_buffers(L):
    w = WORKLOADS["skewed"]
    r = Round(L, w, seed=1).run()
    assert r.error() == 0
    r.check_dispatch()
    r.check_combine()
    small = make_inputs(w, seed=2, tokens=9)
    r2 = Round.__new__(Round)
    r2.__dict__.update(r.__dict__)
    r2.inp, r2.T_call = small, 9
    r2.bs_d = r.rb.buf_set(0, w.K, 9, r.err)
    r2.bs_c = r.rb.buf_set(1, w.K, 9, r.err)
    r2.x, r2.idx, r2.wt = dev(small["x"]), dev(small["topk_idx"]), dev(small["topk_w"])
    r2.y = y_dev(small)
    r2.out = torch.full((w.R, 9, w.H), OUT_CANARY, dtype=torch.int16, device="cuda")
    r2.run()
    assert r2.error() == 0
    r2.check_dispatch()
    r2.check_combine()


def test_all_tokens_masked(L):
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=0)
    inp["topk_idx"][:] = -1
    r = Round(L, w, inp=inp)
    full_check(r)
    assert not (r.out != 0).any()


def test_maximum_topk_and_experts(L):
    w = Workload("max", 8, 4, 8, 8192, 32, mask_p=0.05)
    full_check(Round(L, w, seed=5))


def test_long_prefix_many_tokens_per_cta(L):
    # enough tokens that each CTA takes the maximum token block
    w = Workload("long", 8, 4864, 8, 16, 3, routing="zipf", zipf_s=1.2, mask_p=0.1)
    full_check(Round(L, w, seed=6))


@pytest.mark.parametrize("dtype,tokens", [("bf16", None), ("fp32", None), ("bf16", 599)])
def test_split_grids_several_tokens_per_cta(L, dtype, tokens):
    # more tokens than one wave of CTAs (several tokens per CTA), so the
    # dispatch gives each token block one CTA per ring chunk of its rows and
    # the combine two CTAs per block; rows of 3 (bf16) or 6 (fp32) ring chunks
    # and 11 or 21 512 B chunks, so the shares are uneven; Zipf routing, masks,
    # and a ragged call
    w = Workload("split", 8, 600, 2600, 16, 3, routing="zipf", zipf_s=1.2, mask_p=0.1)
    full_check(Round(L, w, seed=7, tokens=tokens, dtype=dtype))


def test_hot_expert_single_bucket(L):
    # every token of every rank picks expert 0: one bucket per source holds T rows
    w = WORKLOADS["skewed"].with_(H=256)
    inp = make_inputs(w, seed=3)
    inp["topk_idx"][:, :, 0] = 0
    inp["topk_idx"][:, :, 1:] = np.where(inp["topk_idx"][:, :, 1:] == 0, -1, inp["topk_idx"][:, :, 1:])
    full_check(Round(L, w, inp=inp))


@pytest.mark.parametrize("name", ["tiny", "many_small"])
def test_dispatch_into_set_one(L, name):
    full_check(Round(L, WORKLOADS[name], seed=4, dispatch_set=1))


def test_validation_off_gives_same_results(L):
    full_check(Round(L, WORKLOADS["skewed"].with_(H=1024), seed=8, validate=False))


# ---------------------------------------------------------------------------
# route scan on its own
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "many_small", "large"])
def test_route_scan(L, name):
    w = WORKLOADS[name].with_(H=8)
    inp = make_inputs(w, seed=11)
    slot_ref, cnt_ref = oracle.route(inp["topk_idx"], w.E)
    idx = dev(inp["topk_idx"])
    slot = torch.full(idx.shape, -7, dtype=torch.int32, device="cuda")
    counts = torch.full((w.E, w.R), -7, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bs = L.llmoe_buf_set_t(base=None, rank_stride=0, num_max_tokens=w.T, num_tokens=w.T, hidden=w.H,
                           num_ranks=w.R, num_experts=w.E, num_topk=w.K, set=0, err=err.data_ptr())
    L.llmoe_route(idx, slot, counts, bs)
    assert L.llmoe_get_error(bs) == 0
    assert np.array_equal(slot.cpu().numpy(), slot_ref)
    assert np.array_equal(counts.cpu().numpy(), cnt_ref)


# ---------------------------------------------------------------------------
# the two buffer sets are independent; a round replays in a CUDA graph
# ---------------------------------------------------------------------------

def test_combine_leaves_dispatch_set_alone(L):
    w = WORKLOADS["many_small"]
    r = Round(L, w, seed=9)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)
    torch.cuda.synchronize()
    snap = r.rb.storage.clone()
    L.llmoe_clean(r.bs_c)
    L.llmoe_combine(r.y, r.idx, r.wt, r.out, r.bs_c)
    torch.cuda.synchronize()
    r.rb.signal_words(1).copy_(snap.view(torch.int64).as_strided(r.rb.signal_words(1).shape,
                                                                  r.rb.signal_words(1).stride(),
                                                                  r.rb.signal_words(1).storage_offset()))
    assert torch.equal(snap, r.rb.storage)


def test_round_in_cuda_graph(L):
    w = WORKLOADS["skewed"]
    r = Round(L, w, seed=10)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        r.run()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.llmoe_clean(r.bs_d)
        L.llmoe_dispatch(r.x, r.idx, r.bs_d)
        L.llmoe_clean(r.bs_c)
        L.llmoe_combine(r.y, r.idx, r.wt, r.out, r.bs_c)
    r.rb.storage.fill_(CANARY)
    r.out.fill_(OUT_CANARY)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert r.error() == 0
    d = r.check_dispatch()
    r.check_combine()
    r.check_canary(d)


# ---------------------------------------------------------------------------
# validate mode: bad input is reported, skipped, and stays in bounds
# ---------------------------------------------------------------------------

def test_stale_signal_reported(L):
    w = WORKLOADS["tiny"]
    r = Round(L, w, seed=0)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)
    assert L.llmoe_get_error(r.bs_d) == L.LLMOE_DEV_OK
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)  # no clean in between
    assert L.llmoe_get_error(r.bs_d, reset=True) == L.LLMOE_DEV_STALE_SIGNAL
    assert L.llmoe_get_error(r.bs_d) == L.LLMOE_DEV_OK
    L.llmoe_clean(r.bs_c)
    L.llmoe_combine(r.y, r.idx, r.wt, r.out, r.bs_c)
    L.llmoe_combine(r.y, r.idx, r.wt, r.out, r.bs_c)
    assert L.llmoe_get_error(r.bs_c, reset=True) == L.LLMOE_DEV_STALE_SIGNAL


@pytest.mark.parametrize("bad", [8, 9, 1 << 40, -2, -(1 << 40)])
def test_out_of_range_expert_reported_and_skipped(L, bad):
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=1)
    inp["topk_idx"][1, 3, 1] = bad
    r = Round(L, w, inp=inp).run()
    assert r.error() == L.LLMOE_DEV_BAD_EXPERT
    masked = inp["topk_idx"].copy()
    masked[1, 3, 1] = -1
    d = oracle.dispatch(inp["x"], masked, w.E, num_max_tokens=w.T)
    r.check_dispatch(d)
    r.check_canary(d)


def test_duplicate_expert_reported_in_bounds(L):
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=2)
    inp["topk_idx"][0, :, 1] = inp["topk_idx"][0, :, 0]  # every token of rank 0 repeats its expert
    r = Round(L, w, inp=inp).run()
    assert r.error() in (L.LLMOE_DEV_DUPLICATE, L.LLMOE_DEV_SLOT_RANGE)
    # only receive rows and signal words may have changed
    for s in (0, 1):
        r.rb.recv_rows(s).fill_(CANARY)
        r.rb.signal_words(s).fill_(CANARY_WORD)
    assert all_equal_chunked(r.rb.storage, CANARY)


def test_error_word_reset(L):
    err = torch.full((1,), 3, dtype=torch.int32, device="cuda")
    bs = L.llmoe_buf_set_t(base=None, rank_stride=0, num_max_tokens=1, num_tokens=1, hidden=8, num_ranks=1,
                           num_experts=1, num_topk=1, set=0, err=err.data_ptr())
    assert L.llmoe_get_error(bs, reset=True) == 3
    assert int(err.item()) == 0


def test_invalid_call_launches_nothing(L):
    w = WORKLOADS["tiny"]
    r = Round(L, w, seed=0)
    bad = r.rb.buf_set(0, w.K, w.T, r.err)
    bad.hidden = 12
    with pytest.raises(L.LLMoEError) as ei:
        L.llmoe_dispatch(r.x, r.idx, bad)
    assert ei.value.status == L.LLMOE_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert all_equal_chunked(r.rb.storage, CANARY)


# ---------------------------------------------------------------------------
# LLMOE_FLAG_INPUTS_READY: routing read before the previous kernel drains
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "skewed", "dsv3"])
def test_inputs_ready_flag_same_results(L, name):
    w = WORKLOADS[name]
    r = Round(L, w, seed=12)
    r.bs_d = r.rb.buf_set(r.ds, w.K, r.T_call, r.err, flags=L.LLMOE_FLAG_INPUTS_READY)
    r.bs_c = r.rb.buf_set(r.cs, w.K, r.T_call, r.err, flags=L.LLMOE_FLAG_INPUTS_READY)
    full_check(r)


def test_inputs_ready_flag_in_cuda_graph_after_producer(L):
    # the combine's y is written by the kernel right before it: the flag must
    # still make the combine wait for y (only the routing is read early)
    w = WORKLOADS["many_small"]
    r = Round(L, w, seed=13)
    r.bs_c = r.rb.buf_set(r.cs, w.K, r.T_call, r.err, flags=L.LLMOE_FLAG_INPUTS_READY)
    y_final = r.y.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        r.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.llmoe_clean(r.bs_d)
        L.llmoe_dispatch(r.x, r.idx, r.bs_d)
        L.llmoe_clean(r.bs_c)
        r.y.copy_(y_final)  # the expert outputs land right before the combine
        L.llmoe_combine(r.y, r.idx, r.wt, r.out, r.bs_c)
    for _ in range(3):
        r.y.zero_()
        r.rb.storage.fill_(CANARY)
        r.out.fill_(OUT_CANARY)
        g.replay()
    torch.cuda.synchronize()
    assert r.error() == 0
    d = r.check_dispatch()
    r.check_combine()
    r.check_canary(d)


# ---------------------------------------------------------------------------
# LLMOE_FLAG_CLEAN_OTHER_SET: two-launch rounds with the cleans fused
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "skewed", "dsv3"])
def test_fused_clean_rounds(L, name):
    w = WORKLOADS[name]
    r = Round(L, w, seed=14)
    F = L.LLMOE_FLAG_CLEAN_OTHER_SET | L.LLMOE_FLAG_INPUTS_READY
    bs_d = r.rb.buf_set(0, w.K, r.T_call, r.err, flags=F)
    bs_c = r.rb.buf_set(1, w.K, r.T_call, r.err, flags=F)
    r.rb.signal_words(1).fill_(CANARY_WORD)  # the first dispatch must clean set 1
    L.llmoe_clean(r.rb.buf_set(0, w.K, r.T_call, r.err))
    for rep in range(3):
        L.llmoe_dispatch(r.x, r.idx, bs_d)
        torch.cuda.synchronize()
        assert not r.rb.signal_words(1).any(), "dispatch did not clean the other set"
        r.check_dispatch()
        L.llmoe_combine(r.y, r.idx, r.wt, r.out, bs_c)
        torch.cuda.synchronize()
        assert not r.rb.signal_words(0).any(), "combine did not clean the other set"
        r.check_combine()
        assert L.llmoe_get_error(bs_d) == 0  # no stale signal on any repeat


# ---------------------------------------------------------------------------
# staged combine: messages through combine_recv[e][t], then the reduction
# ---------------------------------------------------------------------------

def run_staged(L, r: Round):
    L.llmoe_clean(r.bs_c)
    L.llmoe_combine_staged(r.y, r.idx, r.wt, r.out, r.bs_c)
    torch.cuda.synchronize()
    assert L.llmoe_get_error(r.bs_c) == 0
    w, inp = r.w, r.inp
    st = oracle.combine_staged((inp["y_pool"], inp["y_row_map"]), inp["topk_idx"], inp["topk_w"], w.H, w.E,
                               num_max_tokens=w.T, dtype=r.dtype)
    recv = r.rb.recv_rows(r.cs)
    if st["n"]:
        got = recv[dev(st["msg_rank"]), dev(st["msg_row"])].cpu().numpy()
        bad = np.nonzero((got != st["msgs"]).any(axis=1))[0]
        assert bad.size == 0, f"{bad.size} of {st['n']} staged messages differ"
    dist = ulp_distance(r.out.cpu().numpy(), st["out"], r.dtype)
    assert dist.max(initial=0) <= 1 and int((dist != 0).sum()) == 0
    assert np.array_equal(r.rb.signal_words(r.cs).cpu().numpy(), st["flag_words"])
    # nothing but those messages and the signal words was written
    if st["n"]:
        recv[dev(st["msg_rank"]), dev(st["msg_row"])] = CANARY
    r.rb.signal_words(0).fill_(CANARY_WORD)
    r.rb.signal_words(1).fill_(CANARY_WORD)
    assert all_equal_chunked(r.rb.storage, CANARY)
    return st


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "many_small", "large"])
def test_staged_combine(L, name):
    run_staged(L, Round(L, WORKLOADS[name], seed=31))


@pytest.mark.parametrize("R,E,K,H,T", [(1, 8, 2, 8, 3), (3, 15, 8, 56, 37), (32, 32, 1, 264, 3), (2, 8, 8, 264, 1),
                                       (8, 64, 6, 4096, 9)])
def test_staged_combine_shapes(L, R, E, K, H, T):
    w = Workload("staged", R, T, H, E, K, mask_p=0.3 if K > 1 else 0.0)
    run_staged(L, Round(L, w, seed=R + E + K + H + T))


# Sizes at which the reduce runs through its shared-memory ring (more (token,
# chunk) units than consumer warps in a full wave): rows with a partial last
# 512 B chunk, masked entries, the largest top-k, fp16 / fp32 payloads and a
# call with fewer tokens than the layout holds.
@pytest.mark.parametrize("R,E,K,H,T,tokens,dtype", [(4, 12, 5, 1000, 500, None, "bf16"),
                                                    (2, 64, 32, 520, 300, None, "bf16"),
                                                    (4, 8, 3, 260, 1000, 999, "fp32"),
                                                    (8, 16, 4, 1032, 250, None, "fp16")])
def test_staged_combine_ring_shapes(L, R, E, K, H, T, tokens, dtype):
    w = Workload("staged_ring", R, T, H, E, K, mask_p=0.3)
    run_staged(L, Round(L, w, seed=R + E + K + H + T + 7, tokens=tokens, dtype=dtype))


def test_staged_combine_fewer_tokens_and_set_one(L):
    w = WORKLOADS["dsv3"].with_(H=1024)
    run_staged(L, Round(L, w, seed=33, tokens=77, dispatch_set=1))


def test_staged_equals_direct_on_gpu(L):
    w = WORKLOADS["skewed"]
    r = Round(L, w, seed=34)
    L.llmoe_clean(r.bs_c)
    L.llmoe_combine(r.y, r.idx, r.wt, r.out, r.bs_c)
    direct = r.out.clone()
    r.out.fill_(OUT_CANARY)
    L.llmoe_clean(r.bs_c)
    L.llmoe_combine_staged(r.y, r.idx, r.wt, r.out, r.bs_c)
    torch.cuda.synchronize()
    assert torch.equal(direct, r.out)


# ---------------------------------------------------------------------------
# payload types other than bf16 (LLMoEBufferLayout<T>)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "many_small"])
def test_payload_types_round(L, name, dtype):
    full_check(Round(L, WORKLOADS[name], seed=51, dtype=dtype))


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed"])
def test_payload_types_staged(L, name, dtype):
    run_staged(L, Round(L, WORKLOADS[name], seed=52, dtype=dtype))


@pytest.mark.parametrize("dtype,H", [("fp32", 4), ("fp32", 12), ("fp32", 36), ("fp16", 8), ("fp16", 56),
                                     ("fp32", 2052)])
@pytest.mark.parametrize("R,E,K,T", [(1, 8, 2, 3), (3, 15, 8, 37), (32, 32, 1, 3)])
def test_payload_types_shapes(L, dtype, H, R, E, K, T):
    w = Workload("typed", R, T, H, E, K, mask_p=0.3 if K > 1 else 0.0)
    r = Round(L, w, seed=R + E + K + H + T, dtype=dtype)
    full_check(r)
    run_staged(L, Round(L, w, seed=R + E + K + H + T + 1, dtype=dtype))


# ---------------------------------------------------------------------------
# two-stream double buffering: micro-batch b on set b % 2, b+1's dispatch
# overlapping b's combine
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,H,graph", [("tiny", 256, False), ("skewed", 512, False), ("many_small", 256, False),
                                          ("skewed", 512, True)])
def test_double_buffer_pipeline(L, name, H, graph):
    # graph: the whole two-stream schedule captured once as a CUDA graph (both
    # streams join the capture) and replayed twice
    from combine_routing_count_prefix_gb300.pipeline import DoubleBufferPipeline

    w = WORKLOADS[name].with_(H=H)
    M = 7
    batches = [make_inputs(w, seed=60 + b) for b in range(M)]
    rb = L.RankBuffers(w.T, w.H, w.R, w.E, guard=256, fill=CANARY)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pipe = DoubleBufferPipeline(rb, w.K, err=err)
    dev_in = [(dev(b["x"]), dev(b["topk_idx"]), dev(b["topk_w"]), y_dev(b)) for b in batches]
    outs = [torch.full((w.R, w.T, w.H), OUT_CANARY, dtype=torch.int16, device="cuda") for _ in range(M)]
    snaps, flags = [None] * M, [None] * M

    def schedule():
        for b in range(M):
            x, idx, wt, y = dev_in[b]
            s = b % 2

            def snap_dispatch(b=b, s=s):
                snaps[b] = (rb.recv_rows(s).clone(), rb.signal_words(s).clone())

            def snap_flags(b=b, s=s):
                flags[b] = rb.signal_words(s).clone()

            pipe.dispatch(b, x, idx, after=snap_dispatch)
            pipe.combine(b, y, idx, wt, outs[b], after=snap_flags)
        pipe.join()

    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            schedule()
        for _ in range(2):
            g.replay()
    else:
        schedule()
    torch.cuda.synchronize()
    assert L.llmoe_get_error(pipe.bs[0]) == 0
    for b in range(M):
        inp = batches[b]
        d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, num_max_tokens=w.T)
        recv, counts = snaps[b]
        got = recv[dev(d["row_rank"]), dev(d["row_index"])].cpu().numpy()
        assert np.array_equal(got, d["msgs"]), f"micro-batch {b}: dispatch messages differ"
        assert np.array_equal(counts.cpu().numpy(), d["count_words"])
        ref, fl = oracle.combine((inp["y_pool"], inp["y_row_map"]), inp["topk_idx"], inp["topk_w"], w.H, w.E)
        assert np.array_equal(outs[b].cpu().numpy().view(np.uint16), ref), f"micro-batch {b}: combine differs"
        assert np.array_equal(flags[b].cpu().numpy(), fl)


# ---------------------------------------------------------------------------
# unpack, and the dispatch whose CTAs signal each other (bounded waits)
# ---------------------------------------------------------------------------

def unpack_buffers(w, dtype="bf16"):
    rows = w.E * w.R * w.T
    if dtype == "fp32":
        recv_x = torch.full((rows, w.H), float("nan"), dtype=torch.float32, device="cuda")
    else:
        recv_x = torch.full((rows, w.H), OUT_CANARY, dtype=torch.int16, device="cuda")
    recv_src = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    return recv_x, recv_src


def check_unpack(r: Round, recv_x, recv_src):
    w, inp = r.w, r.inp
    u = oracle.unpack(inp["x"], inp["topk_idx"], w.E, num_max_tokens=w.T, dtype=r.dtype)
    got_x = recv_x.cpu().numpy()
    got_src = recv_src.cpu().numpy()
    rows = u["rows"]
    assert np.array_equal(got_x[rows].view(np.uint8), u["recv_x"][rows].view(np.uint8))
    assert np.array_equal(got_src[rows], u["recv_src"][rows])
    untouched = np.ones(got_src.shape[0], dtype=bool)
    untouched[rows] = False
    assert (got_src[untouched] == -7).all()
    if r.dtype == "fp32":
        assert np.isnan(got_x[untouched]).all()
    else:
        assert (got_x[untouched].view(np.uint16) == OUT_CANARY).all()


@pytest.mark.parametrize("name,dtype", [("tiny", "bf16"), ("dsv3", "bf16"), ("skewed", "bf16"), ("many_small", "bf16"),
                                        ("skewed", "fp32"), ("many_small", "fp16"), ("large", "bf16")])
def test_unpack_after_dispatch(L, name, dtype):
    w = WORKLOADS[name]
    r = Round(L, w, seed=81, dtype=dtype)
    recv_x, recv_src = unpack_buffers(w, dtype)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)
    L.llmoe_unpack(recv_x, recv_src, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    check_unpack(r, recv_x, recv_src)


@pytest.mark.parametrize("name,dtype", [("tiny", "bf16"), ("dsv3", "bf16"), ("skewed", "bf16"), ("many_small", "bf16"),
                                        ("skewed", "fp32"), ("large", "bf16")])
def test_dispatch_signaled(L, name, dtype):
    w = WORKLOADS[name]
    r = Round(L, w, seed=82, dtype=dtype)
    recv_x, recv_src = unpack_buffers(w, dtype)
    ws = torch.zeros(L.llmoe_signal_workspace_bytes(r.bs_d) // 4, dtype=torch.int32, device="cuda")
    for rep in range(3):
        L.llmoe_clean(r.bs_d)
        L.llmoe_dispatch_signaled(r.x, r.idx, recv_x, recv_src, ws, 2_000_000_000, r.bs_d)
        torch.cuda.synchronize()
        assert r.error() == 0
        assert not ws.any(), "the workspace is left zero"
        d = r.check_dispatch()  # messages and plain counts, as llmoe_dispatch leaves them
        check_unpack(r, recv_x, recv_src)
    r.check_canary(d)


# odd shapes for both unpack kernels (balanced when buckets are fewer than
# routed entries, else per bucket) and the signalled dispatch: payloads of
# 1, 7, 33, 125 and 385 quads (partial chunks, a row shorter than one step,
# rows ending mid-step), every message phase, masks, one to 32 ranks
UNPACK_SHAPES = [s for s in SWEEP if s[4] == 37] + [(2, 8, 3, 1000, 41, "bf16"), (3, 15, 4, 3080, 19, "bf16"),
                                                    (2, 8, 2, 252, 23, "fp32"), (4, 8, 3, 264, 9, "fp16")]
UNPACK_SHAPES = [s if len(s) == 6 else (*s, "bf16") for s in UNPACK_SHAPES]


@pytest.mark.parametrize("R,E,K,H,T,dtype", UNPACK_SHAPES)
def test_unpack_shapes(L, R, E, K, H, T, dtype):
    w = Workload("unpack_shape", R, T, H, E, K, mask_p=0.3 if K > 1 else 0.0)
    r = Round(L, w, seed=R * 100 + E + K + H + T, dtype=dtype)
    recv_x, recv_src = unpack_buffers(w, dtype)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)
    L.llmoe_unpack(recv_x, recv_src, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    check_unpack(r, recv_x, recv_src)
    recv_x2, recv_src2 = unpack_buffers(w, dtype)
    ws = torch.zeros(L.llmoe_signal_workspace_bytes(r.bs_d) // 4, dtype=torch.int32, device="cuda")
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_signaled(r.x, r.idx, recv_x2, recv_src2, ws, 2_000_000_000, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    check_unpack(r, recv_x2, recv_src2)
    recv_x3, recv_src3 = unpack_buffers(w, dtype)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_unpack(r.x, r.idx, recv_x3, recv_src3, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    check_unpack(r, recv_x3, recv_src3)


# the dispatch that writes the experts' input rows itself: messages, counts
# and rows equal llmoe_dispatch followed by llmoe_unpack (oracle), nothing
# else in the rank buffers written; repeated on the same buffers
@pytest.mark.parametrize("name,dtype", [("tiny", "bf16"), ("dsv3", "bf16"), ("skewed", "bf16"), ("many_small", "bf16"),
                                        ("skewed", "fp32"), ("many_small", "fp16"), ("dense16", "bf16")])
def test_dispatch_unpack(L, name, dtype):
    w = WORKLOADS[name]
    r = Round(L, w, seed=87, dtype=dtype)
    recv_x, recv_src = unpack_buffers(w, dtype)
    for rep in range(2):
        L.llmoe_clean(r.bs_d)
        L.llmoe_dispatch_unpack(r.x, r.idx, recv_x, recv_src, r.bs_d)
        torch.cuda.synchronize()
        assert r.error() == 0
        d = r.check_dispatch()
        check_unpack(r, recv_x, recv_src)
    r.check_canary(d)


@pytest.mark.parametrize("bad", [8, 1 << 40, -2])
def test_dispatch_unpack_bad_expert_reported_and_skipped(L, bad):
    # an id outside [-1, E): reported in validate mode, and neither a message
    # nor a row is written for it
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=1)
    inp["topk_idx"][1, 3, 1] = bad
    r = Round(L, w, inp=inp)
    recv_x, recv_src = unpack_buffers(w)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_unpack(r.x, r.idx, recv_x, recv_src, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == L.LLMOE_DEV_BAD_EXPERT
    masked = inp["topk_idx"].copy()
    masked[1, 3, 1] = -1
    d = oracle.dispatch(inp["x"], masked, w.E, num_max_tokens=w.T)
    r.check_dispatch(d)
    r.inp = dict(inp, topk_idx=masked)
    check_unpack(r, recv_x, recv_src)
    r.check_canary(d)


def test_dispatch_unpack_in_cuda_graph(L):
    # captured once, replayed on canary-filled buffers
    w = WORKLOADS["skewed"]
    r = Round(L, w, seed=89)
    recv_x, recv_src = unpack_buffers(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        L.llmoe_clean(r.bs_d)
        L.llmoe_dispatch_unpack(r.x, r.idx, recv_x, recv_src, r.bs_d)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.llmoe_clean(r.bs_d)
        L.llmoe_dispatch_unpack(r.x, r.idx, recv_x, recv_src, r.bs_d)
    r.rb.storage.fill_(CANARY)
    recv_x2, recv_src2 = unpack_buffers(w)
    recv_x.copy_(recv_x2)
    recv_src.copy_(recv_src2)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert r.error() == 0
    d = r.check_dispatch()
    check_unpack(r, recv_x, recv_src)
    r.check_canary(d)


@pytest.mark.parametrize("name,tokens,dispatch_set", [("dsv3", 1, 1), ("dsv3", 37, 0), ("skewed", 0, 1),
                                                      ("many_small", 9, 0), ("large", 599, 1)])
def test_dispatch_unpack_fewer_tokens_flags_and_set(L, name, tokens, dispatch_set):
    # a ragged call on either set, with both flags; then the identity-expert
    # layer over its rows
    w = WORKLOADS[name]
    r = Round(L, w, seed=88, tokens=tokens, dispatch_set=dispatch_set)
    recv_x, recv_src = unpack_buffers(w)
    F = L.LLMOE_FLAG_CLEAN_OTHER_SET | L.LLMOE_FLAG_INPUTS_READY
    bs = r.rb.buf_set(r.ds, w.K, r.T_call, r.err, flags=F)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_unpack(r.x, r.idx, recv_x, recv_src, bs)
    torch.cuda.synchronize()
    assert r.error() == 0
    assert not r.rb.signal_words(r.cs).any(), "the other set was cleaned"
    r.check_dispatch()
    check_unpack(r, recv_x, recv_src)
    if tokens:
        L.llmoe_combine(recv_x, r.idx, r.wt, r.out, r.bs_c)
        torch.cuda.synchronize()
        u = oracle.unpack(r.inp["x"], r.inp["topk_idx"], w.E, num_max_tokens=w.T)
        ref, _ = oracle.combine(u["recv_x"], r.inp["topk_idx"], r.inp["topk_w"], w.H, w.E, num_max_tokens=w.T)
        assert np.array_equal(r.out.cpu().numpy().view(np.uint16), ref)


@pytest.mark.parametrize("name,dtype", [("tiny", "bf16"), ("dsv3", "bf16"), ("skewed", "bf16"), ("many_small", "fp16")])
def test_identity_expert_layer(L, name, dtype):
    # dispatch -> unpack -> combine over the unpacked rows: an identity expert
    # returns its input, so the unpacked rows are the combine's y (the
    # end-to-end layer the benchmark times); both fused cleans on
    w = WORKLOADS[name]
    r = Round(L, w, seed=85, dtype=dtype)
    recv_x, recv_src = unpack_buffers(w, dtype)
    F = L.LLMOE_FLAG_CLEAN_OTHER_SET
    bs0 = r.rb.buf_set(0, w.K, r.T_call, r.err, flags=F)
    bs1 = r.rb.buf_set(1, w.K, r.T_call, r.err, flags=F | L.LLMOE_FLAG_INPUTS_READY)
    L.llmoe_clean(r.bs_d)
    for rep in range(2):
        L.llmoe_dispatch(r.x, r.idx, bs0)
        L.llmoe_unpack(recv_x, recv_src, bs0)
        L.llmoe_combine(recv_x, r.idx, r.wt, r.out, bs1)
        torch.cuda.synchronize()
        assert r.error() == 0
        u = oracle.unpack(r.inp["x"], r.inp["topk_idx"], w.E, num_max_tokens=w.T, dtype=dtype)
        ref, flags = oracle.combine(u["recv_x"], r.inp["topk_idx"], r.inp["topk_w"], w.H, w.E, num_max_tokens=w.T,
                                    dtype=dtype)
        dist = ulp_distance(r.out.cpu().numpy(), ref, dtype)
        assert dist.max(initial=0) == 0, f"{int((dist != 0).sum())} elements differ"
        assert np.array_equal(r.rb.signal_words(1).cpu().numpy(), flags)
        assert not r.rb.signal_words(0).any(), "the combine zeroed the dispatch set's counts"


@pytest.mark.parametrize("name,tokens", [("dsv3", 1), ("dsv3", 37), ("skewed", 0), ("many_small", 9)])
def test_unpack_fewer_tokens_than_layout(L, name, tokens):
    # a ragged call: num_tokens < num_max_tokens; rows still index with the
    # layout's T, through both unpack kernels, the signalled dispatch and the
    # identity-expert layer
    w = WORKLOADS[name]
    r = Round(L, w, seed=86 + tokens, tokens=tokens)
    recv_x, recv_src = unpack_buffers(w)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)
    L.llmoe_unpack(recv_x, recv_src, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    u = oracle.unpack(r.inp["x"], r.inp["topk_idx"], w.E, num_max_tokens=w.T)
    got_x, got_src = recv_x.cpu().numpy(), recv_src.cpu().numpy()
    rows = u["rows"]
    assert np.array_equal(got_x[rows].view(np.uint8), u["recv_x"][rows].view(np.uint8))
    assert np.array_equal(got_src[rows], u["recv_src"][rows])
    untouched = np.ones(got_src.shape[0], dtype=bool)
    untouched[rows] = False
    assert (got_src[untouched] == -7).all()
    # the signalled dispatch on the same call
    recv_x2, recv_src2 = unpack_buffers(w)
    ws = torch.zeros(L.llmoe_signal_workspace_bytes(r.bs_d) // 4, dtype=torch.int32, device="cuda")
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_signaled(r.x, r.idx, recv_x2, recv_src2, ws, 2_000_000_000, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    assert torch.equal(recv_src2, recv_src)
    assert np.array_equal(recv_x2.cpu().numpy()[rows], got_x[rows])
    # combine over the unpacked rows (identity experts)
    L.llmoe_clean(r.bs_c)
    L.llmoe_combine(recv_x, r.idx, r.wt, r.out, r.bs_c)
    torch.cuda.synchronize()
    assert r.error() == 0
    ref, flags = oracle.combine(u["recv_x"], r.inp["topk_idx"], r.inp["topk_w"], w.H, w.E, num_max_tokens=w.T)
    assert np.array_equal(r.out.cpu().numpy().view(np.uint16), ref)
    assert np.array_equal(r.rb.signal_words(r.cs).cpu().numpy(), flags)


def test_unpack_more_buckets_than_the_balanced_prefix_holds(L):
    # E * R = 16,384 buckets, beyond the balanced kernel's shared prefix
    # (8,192), with more routed entries (65,536) than buckets: the per-bucket
    # kernel runs although buckets hold several rows each
    w = Workload("many_buckets", 2, 1024, 8, 8192, 32, mask_p=0.1)
    r = Round(L, w, seed=87)
    recv_x, recv_src = unpack_buffers(w)
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch(r.x, r.idx, r.bs_d)
    L.llmoe_unpack(recv_x, recv_src, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    check_unpack(r, recv_x, recv_src)


def test_dispatch_signaled_times_out_without_signals(L):
    # completion counters that never reach the last CTA: no source ever
    # raises its signal words, so every consumer wait runs out
    w = WORKLOADS["tiny"]
    r = Round(L, w, seed=83)
    recv_x, recv_src = unpack_buffers(w)
    ws = torch.full((L.llmoe_signal_workspace_bytes(r.bs_d) // 4,), 1 << 30, dtype=torch.int32, device="cuda")
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_signaled(r.x, r.idx, recv_x, recv_src, ws, 200_000, r.bs_d)
    torch.cuda.synchronize()
    assert L.llmoe_get_error(r.bs_d, reset=True) == L.LLMOE_DEV_TIMEOUT
    assert (recv_src == -7).all(), "no bucket is unpacked without its signal"
    # zeroed again, the same buffers work
    ws.zero_()
    L.llmoe_clean(r.bs_d)
    L.llmoe_dispatch_signaled(r.x, r.idx, recv_x, recv_src, ws, 2_000_000_000, r.bs_d)
    torch.cuda.synchronize()
    assert r.error() == 0
    r.check_dispatch()
    check_unpack(r, recv_x, recv_src)


def test_dispatch_signaled_refuses_a_grid_that_cannot_be_resident(L):
    w = Workload("wide", 8, 100_000, 8, 8, 1)
    rb = L.RankBuffers(w.T, w.H, w.R, w.E)
    bs = rb.buf_set(0, w.K)
    x = torch.zeros((w.R, w.T, w.H), dtype=torch.int16, device="cuda")
    idx = torch.zeros((w.R, w.T, w.K), dtype=torch.int64, device="cuda")
    recv_x = torch.zeros((w.E * w.R * w.T, w.H), dtype=torch.int16, device="cuda")
    recv_src = torch.zeros((w.E * w.R * w.T,), dtype=torch.int32, device="cuda")
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(L.LLMoEError) as ei:
        L.llmoe_dispatch_signaled(x, idx, recv_x, recv_src, ws, 1000, bs)
    assert ei.value.status == L.LLMOE_ERR_INVALID_ARGUMENT
