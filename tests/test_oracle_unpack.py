"""Pins for the oracle's unpack (the received rows as the experts' input).

Two formulations must agree: the unpack computed from x and the routing, and
the dispatch's messages moved to row rank * (L * R * T) + receive row with
their headers.  Each expert's rows also follow the combine's reading order:
feeding the unpacked rows back as identity experts makes the combine return
the weighted sum of x.
"""
import numpy as np
import pytest

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs


@pytest.mark.parametrize("name,H,dtype", [("tiny", 256, "bf16"), ("skewed", 24, "fp16"), ("many_small", 8, "fp32"),
                                          ("dsv3", 16, "bf16")])
def test_unpack_equals_relocated_messages(oracle_lib, name, H, dtype):
    w = WORKLOADS[name].with_(H=H)
    inp = make_inputs(w, seed=71, dtype=dtype)
    u = oracle.unpack(inp["x"], inp["topk_idx"], w.E, dtype=dtype)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, dtype=dtype)
    grow = d["row_rank"] * (w.L * w.R * w.T) + d["row_index"]
    assert np.array_equal(np.sort(grow), np.sort(u["rows"]))
    npdt = np.float32 if dtype == "fp32" else np.uint16
    expect = np.zeros_like(u["recv_x"])
    expect[grow] = d["msgs"][:, 4:].copy().view(npdt).reshape(-1, w.H)
    assert np.array_equal(expect.view(np.uint8), u["recv_x"].view(np.uint8))
    src = np.full(w.E * w.R * w.T, -1, dtype=np.int32)
    src[grow] = d["msgs"][:, :4].copy().view(np.int32)[:, 0]
    assert np.array_equal(src, u["recv_src"])


def test_unpack_is_the_combine_order(oracle_lib):
    w = WORKLOADS["skewed"].with_(H=16, K=1, mask_p=0.0)
    inp = make_inputs(w, seed=72)
    u = oracle.unpack(inp["x"], inp["topk_idx"], w.E)
    out, _ = oracle.combine(u["recv_x"], inp["topk_idx"], np.ones_like(inp["topk_w"]), w.H, w.E)
    assert np.array_equal(out, inp["x"])
