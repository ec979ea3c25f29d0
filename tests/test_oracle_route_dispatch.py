"""Pins for the oracle's route scan and dispatch.

- Slots and counts: brute force over every routing of tiny shapes, checked
  against a second formulation (collect the unmasked entries, stable-sort them
  by (owner rank, local expert, source rank, token), rank inside each group).
- Dispatch: round trip (every written message's header names its source token
  and its payload is that token's row, bit for bit), every unmasked entry
  written exactly once, headers strictly ascending inside a bucket, slots
  filling [0, count), count conservation (sum of recv-count words = number of
  unmasked entries), each bucket <= T.
"""
import itertools

import numpy as np
import pytest

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs


def sort_formulation(idx, E):
    """Slots and counts via a stable sort: independent of the oracle's scan."""
    R, T, K = idx.shape
    L = E // R if E % R == 0 else None
    entries = []
    for src in range(R):
        for t in range(T):
            for k in range(K):
                e = int(idx[src, t, k])
                if e >= 0:
                    key = (e // L, e % L) if L else (e, 0)
                    entries.append((key, src, t, k, e))
    entries.sort(key=lambda z: (z[0], z[1], z[2]))
    slot = np.full((R, T, K), -1, dtype=np.int64)
    cnt = np.zeros((E, R), dtype=np.int64)
    for (key, src, t, k, e) in entries:
        slot[src, t, k] = cnt[e, src]
        cnt[e, src] += 1
    return slot, cnt


def token_choices(E, K):
    """Every top-k row: distinct non-negative experts, -1 anywhere."""
    out = []
    for combo in itertools.product(range(-1, E), repeat=K):
        pos = [c for c in combo if c >= 0]
        if len(pos) == len(set(pos)):
            out.append(combo)
    return out


@pytest.mark.parametrize("K", [1, 2])
@pytest.mark.parametrize("T", [1, 2, 3])
def test_route_brute_force(oracle_lib, K, T):
    E, R = 4, 2
    rows = token_choices(E, K)
    seqs = list(itertools.product(range(len(rows)), repeat=T))
    rng = np.random.default_rng(T * 10 + K)
    if len(seqs) > 4000:  # K=2, T=3: 9261 sequences for rank 0
        pass
    for n, seq in enumerate(seqs):
        other = seqs[(n * 7919 + 13) % len(seqs)] if rng.random() < 0.5 else seq
        idx = np.array([[rows[i] for i in seq], [rows[i] for i in other]], dtype=np.int64)
        slot, cnt = oracle.route(idx, E)
        s2, c2 = sort_formulation(idx, E)
        assert np.array_equal(slot.astype(np.int64), s2), (idx, slot, s2)
        assert np.array_equal(cnt, c2)


def test_route_rejects_bad_ids(oracle_lib):
    idx = np.array([[[0, 1], [2, 4]]], dtype=np.int64)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.route(idx, 4)
    assert ei.value.code == oracle.BAD_EXPERT
    idx = np.array([[[0, -2]]], dtype=np.int64)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.route(idx, 4)
    assert ei.value.code == oracle.BAD_EXPERT
    idx = np.array([[[3, 3]]], dtype=np.int64)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.route(idx, 4)
    assert ei.value.code == oracle.DUPLICATE
    # -1 twice is two masked entries, not a duplicate
    oracle.route(np.array([[[-1, -1]]], dtype=np.int64), 4)


def check_dispatch(x, idx, E, T_max, d):
    R, T, H = x.shape
    K = idx.shape[2]
    L = E // R
    valid = idx >= 0
    n = int(valid.sum())
    assert d["n"] == n
    # conservation and bounds of the count words
    cw = d["count_words"]
    assert cw.shape == (R, E)
    assert int(cw.sum()) == n
    assert cw.min() >= 0 and cw.max() <= T
    for src in range(R):
        assert int(cw[:, src::R].sum()) == int(valid[src].sum())  # words le*R + src
    # each message: header = token, payload = x row, at a row of its bucket
    seen = set()
    hdr = d["msgs"][:, :4].copy().view(np.int32)[:, 0]
    payload = d["msgs"][:, 4:].copy().view(np.uint16)
    buckets = {}
    j = 0
    for src in range(R):
        for t in range(T):
            for k in range(K):
                e = int(idx[src, t, k])
                if e < 0:
                    continue
                dst, le = e // L, e % L
                assert d["row_rank"][j] == dst
                row = int(d["row_index"][j])
                base = (le * R + src) * T_max
                assert base <= row < base + T_max
                assert hdr[j] == t
                assert np.array_equal(payload[j], x[src, t])
                key = (dst, row)
                assert key not in seen
                seen.add(key)
                buckets.setdefault((dst, le, src), []).append((row - base, t))
                j += 1
    assert j == n
    for (dst, le, src), lst in buckets.items():
        slots = sorted(s for s, _ in lst)
        assert slots == list(range(len(lst)))
        assert cw[dst, le * R + src] == len(lst)
        toks = [t for _, t in sorted(lst)]
        assert all(a < b for a, b in zip(toks, toks[1:]))


@pytest.mark.parametrize("name", ["tiny", "skewed", "many_small"])
def test_dispatch_round_trip(oracle_lib, name):
    w = WORKLOADS[name]
    if name != "tiny":
        w = w.with_(H=64)  # keep the CPU test light; routing is unchanged
    inp = make_inputs(w, seed=3)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E)
    check_dispatch(inp["x"], inp["topk_idx"], w.E, w.T, d)


def test_dispatch_fewer_tokens_than_layout(oracle_lib):
    w = WORKLOADS["tiny"].with_(T=16)
    inp = make_inputs(w, seed=5, tokens=5)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, num_max_tokens=16)
    check_dispatch(inp["x"], inp["topk_idx"], w.E, 16, d)
    assert d["row_index"].max() < w.E * w.T


def test_dispatch_brute_force_small(oracle_lib):
    E, R, H = 4, 2, 8
    rows = token_choices(E, 2)
    rng = np.random.default_rng(7)
    for n in range(600):
        T = 1 + n % 3
        seq = rng.integers(0, len(rows), size=(R, T))
        idx = np.array([[rows[i] for i in r] for r in seq], dtype=np.int64)
        x = rng.integers(0, 2**16, size=(R, T, H), dtype=np.uint16)
        d = oracle.dispatch(x, idx, E, num_max_tokens=3)
        check_dispatch(x, idx, E, 3, d)


def test_dispatch_all_masked_and_empty(oracle_lib):
    x = np.zeros((2, 4, 8), dtype=np.uint16)
    idx = np.full((2, 4, 2), -1, dtype=np.int64)
    d = oracle.dispatch(x, idx, 4)
    assert d["n"] == 0 and not d["count_words"].any()
    d = oracle.dispatch(np.zeros((2, 0, 8), dtype=np.uint16), np.zeros((2, 0, 2), dtype=np.int64), 4,
                        num_max_tokens=4)
    assert d["n"] == 0 and not d["count_words"].any()


def test_clean(oracle_lib):
    words = oracle.clean(3, 5)
    assert words.shape == (3, 5) and not words.any()
