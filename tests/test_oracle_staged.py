"""Pins for the oracle's staged combine (combine send / recv roles).

- The reduction read back from the returned messages equals the direct
  combine over the expert outputs, bit for bit (two formulations of the same
  sum), on every workload shape and with masks.
- Every message is [t][the expert output row of that entry], found by a
  linear search for the entry's receive slot rather than the oracle's slots.
- Rows are combine_recv[e][t]: unique per source rank, inside E * T_max rows,
  and the row of entry (src, t, k) is e * T_max + t.
- Flag words equal the plain combine's.
"""
import numpy as np
import pytest

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs


@pytest.mark.parametrize("name,H", [("tiny", 256), ("skewed", 32), ("many_small", 16), ("dsv3", 16)])
def test_staged_equals_direct_combine(oracle_lib, name, H):
    w = WORKLOADS[name].with_(H=H)
    inp = make_inputs(w, seed=21)
    ys = (inp["y_pool"], inp["y_row_map"])
    st = oracle.combine_staged(ys, inp["topk_idx"], inp["topk_w"], w.H, w.E)
    out, flags = oracle.combine(ys, inp["topk_idx"], inp["topk_w"], w.H, w.E)
    assert np.array_equal(st["out"], out)
    assert np.array_equal(st["flag_words"], flags)
    assert st["n"] == int((inp["topk_idx"] >= 0).sum())


def test_staged_messages(oracle_lib):
    w = WORKLOADS["skewed"].with_(H=8, T=24)
    inp = make_inputs(w, seed=22)
    y = inp["y_pool"][inp["y_row_map"]]
    idx = inp["topk_idx"]
    st = oracle.combine_staged(y, idx, inp["topk_w"], w.H, w.E)
    R, T, K = idx.shape
    hdr = st["msgs"][:, :4].copy().view(np.int32)[:, 0]
    pay = st["msgs"][:, 4:].copy().view(np.uint16)
    j = 0
    seen = set()
    for src in range(R):
        for t in range(T):
            for k in range(K):
                e = int(idx[src, t, k])
                if e < 0:
                    continue
                assert st["msg_rank"][j] == src and st["msg_row"][j] == e * w.T + t
                assert (src, st["msg_row"][j]) not in seen
                seen.add((src, st["msg_row"][j]))
                slot = sum(1 for tt in range(t) if e in idx[src, tt])  # earlier tokens of src choosing e
                assert hdr[j] == t
                assert np.array_equal(pay[j], y[e * R * w.T + src * w.T + slot])
                j += 1
    assert j == st["n"] and st["msg_row"].max() < w.E * w.T
