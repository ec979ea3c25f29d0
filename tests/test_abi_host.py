"""The C-ABI library without a GPU: it builds, loads, exports every function
include/llmoe.h declares, its host-only layout calls agree with the oracle,
and its argument checks reject bad calls before anything is launched."""
import ctypes
import os
import random
import re
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from combine_routing_count_prefix_gb300 import build

    build.build()
    from combine_routing_count_prefix_gb300 import llmoe

    return llmoe


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"LLMOE_API\s+[\w\s\*]+?\b(llmoe_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    out = subprocess.run(["nm", "-D", "--defined-only", lib._SO], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(lib._lib, n)
    assert set(lib.EXPORTS) == set(names)
    # nothing else of ours leaks out
    ours = {n for n in exported if n.startswith("llmoe")}
    assert ours == set(names)


def test_layout_bytes_matches_oracle(lib):
    rnd = random.Random(99)
    dims = [(8, 256, 2, 8), (128, 7168, 8, 256), (1024, 7168, 8, 256), (16, 2048, 32, 128), (128, 4096, 8, 64)]
    dims += [(rnd.randint(1, 4096), rnd.randint(1, 16384), rnd.randint(1, 64), rnd.randint(1, 2048))
             for _ in range(3000)]
    dims += [(1, 1, 1, 1), (3, 5, 2, 3), (0, 8, 1, 1), (2**31 - 1, 2**31 - 1, 1, 2**31 - 1)]
    for T, H, R, E in dims:
        assert lib.llmoe_layout_bytes(T, H, R, E) == oracle.size_hint(T, H, R, E), (T, H, R, E)


def test_layout_offsets_match_oracle(lib):
    for T, H, R, E in [(8, 256, 2, 8), (128, 7168, 8, 256), (7, 56, 3, 9), (1, 8, 1, 1)]:
        rc, L = oracle.layout(T, H, R, E)
        assert rc == oracle.OK
        for s in (0, 1):
            assert lib.llmoe_layout_offsets(T, H, R, E, s) == (
                L.dispatch_send[s], L.dispatch_recv[s], L.dispatch_recv_count[s])
    with pytest.raises(lib.LLMoEError):
        lib.llmoe_layout_offsets(8, 256, 2, 8, 2)
    with pytest.raises(lib.LLMoEError):
        lib.llmoe_layout_offsets(1, 1, 1, 1, 0)  # the layout's % 4 assertion


def bs_for(lib, **kw):
    base = dict(base=1 << 20, rank_stride=1 << 20, num_max_tokens=8, num_tokens=8, hidden=256, num_ranks=2,
                num_experts=8, num_topk=2, set=0, err=None)
    base.update(kw)
    return lib.llmoe_buf_set_t(**base)


BAD = [
    dict(num_max_tokens=0), dict(num_tokens=9), dict(num_tokens=-1), dict(hidden=12), dict(hidden=0),
    dict(num_ranks=0), dict(num_experts=9), dict(num_experts=1), dict(num_topk=0), dict(num_topk=9),
    dict(num_experts=16384, num_ranks=2), dict(num_topk=33, num_experts=64), dict(set=2), dict(set=-1),
    dict(base=None), dict(base=(1 << 20) + 8), dict(rank_stride=1000), dict(rank_stride=(1 << 20) + 8),
    dict(rank_stride=1024), dict(err=(1 << 20) + 2),
]


@pytest.mark.parametrize("kw", BAD)
def test_invalid_buf_set_rejected_before_launch(lib, kw):
    bs = bs_for(lib, **kw)
    A = 1 << 24
    calls = [
        lambda: lib._lib.llmoe_dispatch(A, A, ctypes.byref(bs), None),
        lambda: lib._lib.llmoe_combine(A, A, A, 2 * A, ctypes.byref(bs), None),
        lambda: lib._lib.llmoe_clean(ctypes.byref(bs), None),
        lambda: lib._lib.llmoe_dispatch_unpack(A, A, 2 * A, 3 * A, ctypes.byref(bs), None),
    ]
    for c in calls:
        assert c() == lib.LLMOE_ERR_INVALID_ARGUMENT


def test_invalid_pointers_rejected_before_launch(lib):
    bs = bs_for(lib)
    A = 1 << 24
    L = lib._lib
    assert L.llmoe_dispatch(None, A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch(A + 4, A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch(A, A + 4, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_combine(A, A, A, None, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_combine(A, A, A + 2, 2 * A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    # out overlapping y
    assert L.llmoe_combine(A, A, A, A + 4096, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_route(A, A, None, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch(A, A, None, None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    # the dispatch with the experts' rows: recv_x / recv_src missing or misaligned
    assert L.llmoe_dispatch_unpack(A, A, None, 3 * A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch_unpack(A, A, 2 * A, None, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch_unpack(A, A, 2 * A + 8, 3 * A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch_unpack(A, A, 2 * A, 3 * A + 2, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert L.llmoe_dispatch_unpack(None, A, 2 * A, 3 * A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    code = ctypes.c_int32()
    assert L.llmoe_get_error(ctypes.byref(bs), None, ctypes.byref(code), 0) == lib.LLMOE_ERR_INVALID_USAGE


def test_status_strings(lib):
    assert lib.llmoe_status_string(0) == "success"
    assert lib.llmoe_status_string(4) == "invalid argument"
    assert lib.llmoe_status_string(77) == "unknown status"


def test_layout_bytes_dtype_matches_oracle(lib):
    rnd = random.Random(7)
    for _ in range(2000):
        T, H, R, E = rnd.randint(1, 2048), rnd.randint(1, 8192), rnd.randint(1, 64), rnd.randint(1, 1024)
        for code, es in ((0, 2), (1, 2), (2, 4)):
            assert lib.llmoe_layout_bytes_dtype(T, H, R, E, code) == oracle.size_hint(T, H, R, E, es)
    assert lib.llmoe_layout_bytes_dtype(8, 256, 2, 8, 3) == 0
    assert lib.llmoe_layout_bytes_dtype(8, 256, 2, 8, -1) == 0
    for code, es in ((0, 2), (1, 2), (2, 4)):
        rc, L = oracle.layout(16, 96, 4, 32, es)
        for s in (0, 1):
            assert lib.llmoe_layout_offsets_dtype(16, 96, 4, 32, code, s) == (
                L.dispatch_send[s], L.dispatch_recv[s], L.dispatch_recv_count[s])


@pytest.mark.parametrize("kw", [dict(dtype=3), dict(dtype=-1), dict(dtype=2, hidden=6), dict(dtype=1, hidden=12),
                                dict(dtype=2, hidden=2)])
def test_invalid_dtype_rejected_before_launch(lib, kw):
    bs = bs_for(lib, **kw)
    A = 1 << 24
    assert lib._lib.llmoe_dispatch(A, A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
    assert lib._lib.llmoe_combine(A, A, A, 2 * A, ctypes.byref(bs), None) == lib.LLMOE_ERR_INVALID_ARGUMENT
