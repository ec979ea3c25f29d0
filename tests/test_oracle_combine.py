"""Pins for the oracle's combine and its bf16 rounding.

- bf16 round-to-nearest-even: hand-built tie / carry / subnormal / overflow
  bit patterns, and agreement with PyTorch's float32 -> bfloat16 cast (a
  library routine) on 2^20 random finite floats.
- combine: (i) top-1 with weight 1 over identity experts (expert output =
  the dispatched row) returns x bit for bit; (ii) one-hot weights return the
  chosen expert's row; (iii) constant expert rows give sum_k w_k c_{e_k}
  computed without any row addressing; (iv) identity experts with K > 1 give
  bf16(sum_k w_k x) computed without slots; (v) the accumulation order is
  ascending k and a product is rounded before it is added (cases where the
  other choices give a different bf16); (vi) masked entries contribute
  nothing; a fully masked token is +0.0; the flag words count rows per expert.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs


def f32_bits(u):
    return np.array([u], dtype=np.uint32).view(np.float32)[0]


@pytest.mark.parametrize("bits,expect", [
    (0x3F808000, 0x3F80),  # tie, kept part even -> stays
    (0x3F818000, 0x3F82),  # tie, kept part odd -> up to even
    (0x3F808001, 0x3F81),  # just above the tie
    (0x3F807FFF, 0x3F80),  # just below the tie
    (0x3FFF8000, 0x4000),  # tie, odd, carry into the exponent (-> 2.0)
    (0x7F7FFFFF, 0x7F80),  # largest float rounds to +inf
    (0x7F800000, 0x7F80),  # +inf
    (0xFF800000, 0xFF80),  # -inf
    (0xBF808000, 0xBF80),  # negative tie, even
    (0xBF818000, 0xBF82),  # negative tie, odd
    (0x00008000, 0x0000),  # subnormal tie to zero (even)
    (0x00018000, 0x0002),  # subnormal tie, odd -> up
    (0x80000000, 0x8000),  # -0.0
    (0x3F800000, 0x3F80),  # exact
])
def test_bf16_rne_bit_patterns(oracle_lib, bits, expect):
    assert oracle.f32_to_bf16(f32_bits(bits)) == expect


def test_bf16_nan_stays_nan(oracle_lib):
    b = oracle.f32_to_bf16(f32_bits(0x7F800001))
    assert (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


def test_bf16_matches_torch_cast(oracle_lib):
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2**32, size=2**20, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    # also values in the data path's range
    f = np.concatenate([f, rng.standard_normal(2**18).astype(np.float32)])
    ours = oracle.f32_to_bf16_array(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_widen_exact(oracle_lib):
    for b in (0x0000, 0x8000, 0x3F80, 0xC0A0, 0x0001, 0x7F7F):
        assert np.float32(oracle.bf16_to_f32(b)).view(np.uint32) == np.uint32(b << 16)


def identity_expert_y(d, E, R, T_max, H):
    """Dense expert outputs where every used row equals its dispatched payload."""
    L = E // R
    y = np.zeros((E * R * T_max, H), dtype=np.uint16)
    grow = d["row_rank"] * (L * R * T_max) + d["row_index"]
    y[grow] = d["msgs"][:, 4:].copy().view(np.uint16).reshape(-1, H)
    return y


def bf16_vals(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


def test_top1_weight1_identity_returns_x(oracle_lib):
    w = WORKLOADS["many_small"].with_(K=1, H=64)
    inp = make_inputs(w, seed=2)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E)
    y = identity_expert_y(d, w.E, w.R, w.T, w.H)
    ones = np.ones_like(inp["topk_w"])
    out, flags = oracle.combine(y, inp["topk_idx"], ones, w.H, w.E)
    assert np.array_equal(out, inp["x"])


def test_one_hot_weights_return_expert_row(oracle_lib):
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=4)
    y = inp["y_pool"][inp["y_row_map"]]
    slot, _ = oracle.route(inp["topk_idx"], w.E)
    rng = np.random.default_rng(0)
    R, T, K = inp["topk_idx"].shape
    pick = rng.integers(0, K, size=(R, T))
    wts = np.zeros((R, T, K), dtype=np.float32)
    wts[np.arange(R)[:, None], np.arange(T)[None, :], pick] = 1.0
    out, _ = oracle.combine(y, inp["topk_idx"], wts, w.H, w.E)
    # the expected row found by a linear search for the (src, t) entry of
    # expert e among the used rows, not by the oracle's row formula
    for src in range(R):
        for t in range(T):
            e = inp["topk_idx"][src, t, pick[src, t]]
            # slot = number of earlier tokens of src that chose e
            s = sum(1 for tt in range(t) if e in inp["topk_idx"][src, tt])
            row = y[e * R * w.T + src * w.T + s]
            assert np.array_equal(bf16_vals(out[src, t]), bf16_vals(row))


def test_constant_expert_rows(oracle_lib):
    w = WORKLOADS["skewed"].with_(H=16)
    inp = make_inputs(w, seed=6)
    R, T, K = inp["topk_idx"].shape
    # each expert's rows hold one constant c_e
    c = np.float32(np.linspace(-3, 3, w.E)).astype(np.float32)
    cb = torch.from_numpy(c).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = np.repeat(cb, R * w.T)[:, None].repeat(w.H, axis=1)
    out, flags = oracle.combine(y, inp["topk_idx"], inp["topk_w"], w.H, w.E)
    cv = bf16_vals(cb)
    for src in range(R):
        for t in range(T):
            acc = np.float32(0.0)
            for k in range(K):
                e = inp["topk_idx"][src, t, k]
                if e >= 0:
                    acc = np.float32(acc + np.float32(inp["topk_w"][src, t, k] * cv[e]))
            expect = torch.tensor([acc]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
            assert np.all(out[src, t] == expect)
    # flags: rank src, word e = tokens of src that chose e
    for src in range(R):
        for e in range(w.E):
            assert flags[src, e] == int((inp["topk_idx"][src] == e).any(axis=1).sum())


def test_identity_experts_weighted_sum(oracle_lib):
    w = WORKLOADS["dsv3"].with_(H=32, T=16)
    inp = make_inputs(w, seed=8)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E)
    y = identity_expert_y(d, w.E, w.R, w.T, w.H)
    out, _ = oracle.combine(y, inp["topk_idx"], inp["topk_w"], w.H, w.E)
    xv = bf16_vals(inp["x"])
    R, T, K = inp["topk_idx"].shape
    acc = np.zeros((R, T, w.H), dtype=np.float32)
    for k in range(K):
        p = (inp["topk_w"][:, :, k:k + 1] * xv).astype(np.float32)
        p = np.where((inp["topk_idx"][:, :, k] >= 0)[..., None], p, np.float32(0))
        acc = (acc + p).astype(np.float32)
    expect = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, expect)


def one_token_combine(ys, ws):
    """One rank, one token, K = len(ys) experts 0..K-1, H = 1."""
    K = len(ys)
    yb = torch.tensor(ys, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = np.zeros((K, 1), dtype=np.uint16)
    y[:, 0] = yb
    idx = np.arange(K, dtype=np.int64).reshape(1, 1, K)
    out, _ = oracle.combine(y, idx, np.array(ws, dtype=np.float32).reshape(1, 1, K), 1, K)
    return int(out[0, 0, 0])


def bf16_of(v):
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0])


def test_ascending_k_order(oracle_lib):
    # (256 + -256) + 2^-20 = 2^-20, while 256 + (-256 + 2^-20) = 0 in fp32
    # and the reversed order (2^-20 + -256) + 256 = 0 as well.
    assert one_token_combine([256.0, -256.0, 2.0 ** -20], [1.0, 1.0, 1.0]) == bf16_of(2.0 ** -20)
    assert one_token_combine([2.0 ** -20, -256.0, 256.0], [1.0, 1.0, 1.0]) == 0


def test_product_rounded_before_add(oracle_lib):
    # acc = fl(-w*y) then acc + fl(w*y) = +0 exactly; a fused multiply-add
    # would leave the product's rounding error (non-zero).
    w = np.float32(0.1)
    y = 1.0078125  # bf16-exact, w*y needs more than 24 bits
    assert float(np.float32(w) * np.float32(y)) != float(np.float64(w) * np.float64(y))
    assert one_token_combine([-y, y], [w, w]) == 0x0000


def test_masked_entries_and_all_masked(oracle_lib):
    y = np.array([[bf16_of(1.5)], [bf16_of(-2.0)], [bf16_of(4.0)]], dtype=np.uint16)
    idx = np.array([[[0, -1, 2]]], dtype=np.int64)
    out, flags = oracle.combine(y, idx, np.array([[[0.5, 100.0, 0.25]]], dtype=np.float32), 1, 3)
    assert out[0, 0, 0] == bf16_of(0.5 * 1.5 + 0.25 * 4.0)
    assert list(flags[0]) == [1, 0, 1]
    idx = np.full((1, 1, 3), -1, dtype=np.int64)
    out, flags = oracle.combine(y, idx, np.ones((1, 1, 3), dtype=np.float32), 1, 3)
    assert out[0, 0, 0] == 0x0000 and not flags.any()


def test_pool_row_map_equals_dense(oracle_lib):
    w = WORKLOADS["many_small"].with_(H=16)
    inp = make_inputs(w, seed=1, pool_rows=1000)
    dense = inp["y_pool"][inp["y_row_map"]]
    a, fa = oracle.combine(dense, inp["topk_idx"], inp["topk_w"], w.H, w.E)
    b, fb = oracle.combine((inp["y_pool"], inp["y_row_map"]), inp["topk_idx"], inp["topk_w"], w.H, w.E)
    assert np.array_equal(a, b) and np.array_equal(fa, fb)
