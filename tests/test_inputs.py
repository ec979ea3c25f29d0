"""The seeded workload generator draws what its description says."""
import numpy as np

from combine_routing_count_prefix_gb300.inputs import WORKLOADS, make_inputs


def test_deterministic():
    w = WORKLOADS["tiny"]
    a, b = make_inputs(w, seed=0), make_inputs(w, seed=0)
    for k in a:
        assert np.array_equal(a[k], b[k])
    c = make_inputs(w, seed=1)
    assert not np.array_equal(a["x"], c["x"])


def test_uniform_routing_distinct_and_complete():
    w = WORKLOADS["many_small"].with_(H=8)
    inp = make_inputs(w, seed=0)
    idx = inp["topk_idx"].reshape(-1, w.K)
    assert idx.min() >= 0 and idx.max() < w.E
    assert all(len(set(r)) == w.K for r in idx.tolist())
    wts = inp["topk_w"].reshape(-1, w.K)
    assert np.allclose(wts.sum(1), 1.0, atol=1e-6) and (wts > 0).all()


def test_zipf_masked_routing():
    w = WORKLOADS["skewed"].with_(H=8)
    inp = make_inputs(w, seed=0)
    idx = inp["topk_idx"].reshape(-1, w.K)
    frac = (idx < 0).mean()
    assert 0.07 < frac < 0.13
    for r in idx.tolist():
        pos = [e for e in r if e >= 0]
        assert len(pos) == len(set(pos))
    counts = np.bincount(idx[idx >= 0], minlength=w.E)
    assert counts[0] == counts.max() and counts[0] > 3 * counts[-8:].mean()


def test_row_map_hashed_when_large():
    w = WORKLOADS["dsv3"].with_(H=8)
    inp = make_inputs(w, seed=0)
    m = inp["y_row_map"]
    assert m.shape == (w.E * w.R * w.T,) and m.min() >= 0 and m.max() < inp["y_pool"].shape[0]
    # no systematic aliasing at the strides a row-addressing bug would use
    for stride in (1, w.T, w.R * w.T, 16 * w.R * w.T):
        assert (m[:-stride] == m[stride:]).mean() < 0.01


def test_fewer_tokens_per_call():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=0, tokens=3)
    assert inp["x"].shape == (2, 3, 256) and inp["topk_idx"].shape == (2, 3, 2)
    assert inp["y_row_map"].shape == (w.E * w.R * w.T,)
