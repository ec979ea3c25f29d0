"""Pins for the oracle's payload types other than bf16 (LLMoEBufferLayout<T>
with T = fp16 or fp32).

- binary16 round to nearest even: hand-built ties, carries, subnormals,
  overflow and specials, and agreement with numpy's float32 -> float16 cast
  (a library routine) on 2^20 random floats; widening checked on all 65,536
  binary16 patterns against numpy.
- dispatch of fp16 / fp32 payloads: round trip of every message.
- combine: one-hot weights return the expert row; constant rows give
  sum_k w_k c_{e_k} computed without rows; identity experts give
  T(sum_k w_k x); the staged combine equals the direct one.
"""
import numpy as np
import pytest

import oracle
from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs


def f32(bits):
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


@pytest.mark.parametrize("value,expect", [
    (1.0, 0x3C00), (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (1e30, 0x7C00),
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (3 * 2.0 ** -25, 0x0002), (2.0 ** -14, 0x0400),
    (1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02), (2047.5, 0x67FF + 1), (-0.0, 0x8000),
    (-1.5, 0xBE00), (2.0 ** -14 - 2.0 ** -25, 0x0400),
])
def test_f16_rne_patterns(oracle_lib, value, expect):
    assert oracle.f32_to_f16(value) == expect


def test_f16_specials(oracle_lib):
    assert oracle.f32_to_f16(f32(0x7F800000)) == 0x7C00
    assert oracle.f32_to_f16(f32(0xFF800000)) == 0xFC00
    h = oracle.f32_to_f16(f32(0x7FC00000))
    assert (h & 0x7C00) == 0x7C00 and (h & 0x3FF) != 0


def test_f16_matches_numpy(oracle_lib):
    rng = np.random.default_rng(5)
    u = rng.integers(0, 2**32, size=2**20, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    f = np.concatenate([f, rng.standard_normal(2**16).astype(np.float32),
                        (rng.standard_normal(2**16) * 1e-5).astype(np.float32),
                        (rng.standard_normal(2**16) * 3e4).astype(np.float32)])
    ours = oracle.f32_to_f16_array(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_widen_all_patterns(oracle_lib):
    for h in range(0, 65536, 7):
        v = oracle.f16_to_f32(h)
        ref = np.array([h], dtype=np.uint16).view(np.float16)[0].astype(np.float32)
        if np.isnan(ref):
            assert np.isnan(v)
        else:
            assert np.float32(v).view(np.uint32) == ref.view(np.uint32)


def values(a, dtype):
    return a.view(np.float16).astype(np.float32) if dtype == "fp16" else a.astype(np.float32)


def to_type(acc, dtype):
    return acc.astype(np.float16).view(np.uint16) if dtype == "fp16" else acc.astype(np.float32)


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_dispatch_round_trip_typed(oracle_lib, dtype):
    w = WORKLOADS["skewed"].with_(H=24)
    inp = make_inputs(w, seed=41, dtype=dtype)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, dtype=dtype)
    es = 2 if dtype == "fp16" else 4
    assert d["msgs"].shape[1] == 4 + es * w.H
    hdr = d["msgs"][:, :4].copy().view(np.int32)[:, 0]
    j = 0
    idx = inp["topk_idx"]
    for src in range(w.R):
        for t in range(w.T):
            for k in range(w.K):
                if idx[src, t, k] < 0:
                    continue
                assert hdr[j] == t
                assert d["msgs"][j, 4:].tobytes() == inp["x"][src, t].tobytes()
                j += 1
    assert j == d["n"] and int(d["count_words"].sum()) == d["n"]


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_combine_typed_closed_forms(oracle_lib, dtype):
    w = WORKLOADS["many_small"].with_(H=16)
    inp = make_inputs(w, seed=42, dtype=dtype)
    R, T, K = inp["topk_idx"].shape
    y = inp["y_pool"][inp["y_row_map"]]
    # one-hot weights: out is the chosen expert's row
    pick = np.random.default_rng(1).integers(0, K, size=(R, T))
    wts = np.zeros((R, T, K), dtype=np.float32)
    wts[np.arange(R)[:, None], np.arange(T)[None, :], pick] = 1.0
    out, _ = oracle.combine(y, inp["topk_idx"], wts, w.H, w.E, dtype=dtype)
    for src in range(R):
        for t in range(T):
            e = inp["topk_idx"][src, t, pick[src, t]]
            s = sum(1 for tt in range(t) if e in inp["topk_idx"][src, tt])
            assert np.array_equal(values(out[src, t], dtype), values(y[e * R * w.T + src * w.T + s], dtype))
    # constant rows: sum_k w_k c_e without any row addressing
    c = np.linspace(-2, 2, w.E).astype(np.float32)
    cq = to_type(c, dtype)
    yc = np.repeat(cq, R * w.T)[:, None].repeat(w.H, axis=1)
    out, _ = oracle.combine(yc, inp["topk_idx"], inp["topk_w"], w.H, w.E, dtype=dtype)
    cv = values(cq, dtype)
    for src in range(R):
        for t in range(T):
            acc = np.float32(0)
            for k in range(K):
                e = inp["topk_idx"][src, t, k]
                if e >= 0:
                    acc = np.float32(acc + np.float32(inp["topk_w"][src, t, k] * cv[e]))
            assert np.all(out[src, t] == to_type(np.array([acc], dtype=np.float32), dtype)[0])


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_identity_experts_and_staged_typed(oracle_lib, dtype):
    w = WORKLOADS["dsv3"].with_(H=16, T=12)
    inp = make_inputs(w, seed=43, dtype=dtype)
    d = oracle.dispatch(inp["x"], inp["topk_idx"], w.E, dtype=dtype)
    npdt = np.uint16 if dtype == "fp16" else np.float32
    y = np.zeros((w.E * w.R * w.T, w.H), dtype=npdt)
    grow = d["row_rank"] * (w.L * w.R * w.T) + d["row_index"]
    y[grow] = d["msgs"][:, 4:].copy().view(npdt).reshape(-1, w.H)
    out, flags = oracle.combine(y, inp["topk_idx"], inp["topk_w"], w.H, w.E, dtype=dtype)
    xv = values(inp["x"], dtype)
    acc = np.zeros((w.R, w.T, w.H), dtype=np.float32)
    for k in range(w.K):
        p = (inp["topk_w"][:, :, k:k + 1] * xv).astype(np.float32)
        p = np.where((inp["topk_idx"][:, :, k] >= 0)[..., None], p, np.float32(0))
        acc = (acc + p).astype(np.float32)
    assert np.array_equal(out, to_type(acc, dtype))
    st = oracle.combine_staged(y, inp["topk_idx"], inp["topk_w"], w.H, w.E, dtype=dtype)
    assert np.array_equal(st["out"], out) and np.array_equal(st["flag_words"], flags)
