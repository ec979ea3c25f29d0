"""Pins for the oracle's layout (LL_MoE_Buffers.hpp, LLMoEBufferLayout).

The oracle transcribes the constructor's steps.  It is pinned here by things
other than those steps: hand-computed worked values, the closed form the steps
reduce to when num_experts >= 1 (the combine send region E*T*msg is then never
smaller than the dispatch send region T*msg, so total = 4*E*T*msg + 16*E), the
aliasing that clean_meta() asserts, and the region geometry.
"""
import os
import random

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_worked_values.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, *vals = line.split()
        rows.append((name, [int(v) for v in vals]))
    return rows


@pytest.mark.parametrize("name,vals", _golden_rows())
def test_worked_values(oracle_lib, name, vals):
    T, H, R, E, msg, send, recv, sig, total, s0s, s0r, s0g, s1s, s1r, s1g = vals
    rc, L = oracle.layout(T, H, R, E)
    assert rc == oracle.OK
    assert (L.msg_bytes, L.send_bytes, L.recv_bytes, L.sig_bytes, L.total_bytes) == (msg, send, recv, sig, total)
    assert (L.dispatch_send[0], L.dispatch_recv[0], L.dispatch_recv_count[0]) == (s0s, s0r, s0g)
    assert (L.dispatch_send[1], L.dispatch_recv[1], L.dispatch_recv_count[1]) == (s1s, s1r, s1g)
    assert oracle.size_hint(T, H, R, E) == total


def test_closed_form_sweep(oracle_lib):
    rnd = random.Random(1234)
    for _ in range(3000):
        T = rnd.randint(1, 5000)
        H = rnd.randint(1, 20000)
        R = rnd.randint(1, 64)
        E = rnd.randint(1, 1024)
        eb = rnd.choice([1, 2, 4])
        m = 4 + H * eb
        rc, L = oracle.layout(T, H, R, E, eb)
        if (E * T * m) % 4 != 0:
            assert rc == oracle.ASSERT
            continue
        assert rc == oracle.OK
        S = E * T * m
        assert L.total_bytes == 4 * E * T * m + 16 * E
        for i in (0, 1):
            assert L.dispatch_send[i] == S * i
            assert L.dispatch_recv[i] == 2 * S + S * i
            assert L.dispatch_recv_count[i] == 4 * S + 8 * E * i
        assert L.num_sig_elems == E


def test_num_ranks_unused(oracle_lib):
    # num_ranks is [[maybe_unused]] in the constructor: it never changes a size.
    base = oracle.size_hint(128, 7168, 8, 256)
    for R in (1, 2, 3, 8, 32, 1000):
        assert oracle.size_hint(128, 7168, R, 256) == base


def test_combine_roles_alias_dispatch_roles(oracle_lib):
    # clean_meta() asserts dispatch_recv_count == combine_recv_flag; the
    # pointer assignment gives combine send/recv the dispatch send/recv
    # addresses of the same set.
    for dims in [(8, 256, 2, 8), (128, 7168, 8, 256), (3, 56, 1, 5)]:
        rc, L = oracle.layout(*dims)
        assert rc == oracle.OK
        for i in (0, 1):
            assert L.combine_recv_flag[i] == L.dispatch_recv_count[i]
            assert L.combine_send[i] == L.dispatch_send[i]
            assert L.combine_recv[i] == L.dispatch_recv[i]


def test_regions_tile_the_buffer(oracle_lib):
    # six regions, disjoint, in order, covering [0, total) exactly
    for dims in [(8, 256, 2, 8), (16, 2048, 32, 128), (1, 8, 1, 1), (7, 56, 3, 9)]:
        rc, L = oracle.layout(*dims)
        assert rc == oracle.OK
        spans = [
            (L.dispatch_send[0], L.send_bytes), (L.dispatch_send[1], L.send_bytes),
            (L.dispatch_recv[0], L.recv_bytes), (L.dispatch_recv[1], L.recv_bytes),
            (L.dispatch_recv_count[0], L.sig_bytes), (L.dispatch_recv_count[1], L.sig_bytes),
        ]
        pos = 0
        for off, size in spans:
            assert off == pos
            pos += size
        assert pos == L.total_bytes


def test_assertion_and_errors(oracle_lib):
    # bf16 payload: msg = 4 + 2H; with H odd and E*T odd the region is 2 mod 4
    rc, _ = oracle.layout(1, 1, 1, 1, 2)
    assert rc == oracle.ASSERT
    assert oracle.size_hint(1, 1, 1, 1) == 0
    assert oracle.layout(3, 5, 2, 3, 2)[0] == oracle.ASSERT
    assert oracle.layout(2, 5, 2, 3, 2)[0] == oracle.OK
    for bad in [(0, 8, 1, 1), (1, 0, 1, 1), (1, 8, 0, 1), (1, 8, 1, 0), (-1, 8, 1, 1)]:
        assert oracle.layout(*bad)[0] == oracle.BAD_ARG
    # 2^31-1 tokens x 2^31-1 hidden x 2^31-1 experts overflows 64 bits
    big = 2**31 - 1
    assert oracle.layout(big, big, 1, big)[0] == oracle.OVERFLOW
