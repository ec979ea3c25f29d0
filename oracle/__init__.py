"""CPU oracle for the low-latency MoE dispatch / combine data path.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library and its
Python binding never import this package, and the two share no source.

The arithmetic lives in ``llmoe_oracle.c`` (plain C, single-threaded, built
with ``-ffp-contract=off``); this module compiles it with gcc on first use and
marshals numpy arrays through ctypes.  Each wrapper cites the passage its C
function follows:

- ``layout`` / ``size_hint``: LL_MoE_Buffers.hpp, LLMoEBufferLayout
  constructor and get_rdma_size_hint.
- ``route``: the per-(expert, source-rank) counts and ascending-token slots.
- ``dispatch``: LL_MoE_Buffers.hpp, LLMoEBuffer dispatch recv buffer
  ([num_experts * num_tokens] messages of one int header plus ``hidden``
  values) and recv-count words.
- ``combine``: the K-row gather, fp32 ``w * y`` in ascending k, bf16 store;
  LLMoEBuffer combine recv-flag words.
- ``combine_staged``: the combine through the combine receive buffers
  (LLMoEBuffer combine send / recv roles): messages [t | y row] at
  combine_recv[e][t] of the source rank, then the reduction from them.
- ``unpack``: the received rows in the experts' input order (each local
  expert's receive rows contiguous, the order the combine reads y in).
- ``clean``: LLMoEBuffer::clean_meta.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "llmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_LOCK = threading.Lock()
_lib = None

OK, BAD_EXPERT, DUPLICATE = 0, 1, 2

# payload element types of LLMoEBufferLayout<T>: (code, bytes, numpy dtype of the stored values)
DTYPES = {"bf16": (0, 2, np.uint16), "fp16": (1, 2, np.uint16), "fp32": (2, 4, np.float32)}
BAD_ARG, ASSERT, OVERFLOW = -1, -2, -3

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


class Layout(ctypes.Structure):
    _fields_ = [
        ("total_bytes", ctypes.c_uint64),
        ("msg_bytes", ctypes.c_uint64),
        ("send_bytes", ctypes.c_uint64),
        ("recv_bytes", ctypes.c_uint64),
        ("sig_bytes", ctypes.c_uint64),
        ("dispatch_send", ctypes.c_uint64 * 2),
        ("dispatch_recv", ctypes.c_uint64 * 2),
        ("dispatch_recv_count", ctypes.c_uint64 * 2),
        ("combine_send", ctypes.c_uint64 * 2),
        ("combine_recv", ctypes.c_uint64 * 2),
        ("combine_recv_flag", ctypes.c_uint64 * 2),
        ("num_sig_elems", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        out = {}
        for name, _ in self._fields_:
            v = getattr(self, name)
            out[name] = list(v) if hasattr(v, "__len__") else int(v)
        return out


def lib():
    global _lib
    with _LOCK:
        if _lib is None:
            so = build()
            L = ctypes.CDLL(so)
            P = ctypes.c_void_p
            i = ctypes.c_int
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f32.restype = ctypes.c_float
            L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            L.oracle_f32_to_bf16.restype = ctypes.c_uint16
            L.oracle_f32_to_bf16_array.argtypes = [P, P, ctypes.c_int64]
            L.oracle_f32_to_bf16_array.restype = None
            L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f32.restype = ctypes.c_float
            L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            L.oracle_f32_to_f16.restype = ctypes.c_uint16
            L.oracle_f32_to_f16_array.argtypes = [P, P, ctypes.c_int64]
            L.oracle_f32_to_f16_array.restype = None
            L.oracle_layout.argtypes = [i, i, i, i, i, ctypes.POINTER(Layout)]
            L.oracle_layout.restype = i
            L.oracle_size_hint.argtypes = [i, i, i, i, i]
            L.oracle_size_hint.restype = ctypes.c_uint64
            L.oracle_route.argtypes = [i, i, i, i, P, P, P]
            L.oracle_route.restype = i
            L.oracle_dispatch.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P, P]
            L.oracle_dispatch.restype = i
            L.oracle_combine.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P]
            L.oracle_combine.restype = i
            L.oracle_combine_staged.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P, P, P, P]
            L.oracle_combine_staged.restype = i
            L.oracle_unpack.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P]
            L.oracle_unpack.restype = i
            L.oracle_clean.argtypes = [i, i, P]
            L.oracle_clean.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def bf16_to_f32(b: int) -> float:
    return float(lib().oracle_bf16_to_f32(int(b)))


def f32_to_bf16(f: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(np.float32(f))))


def f16_to_f32(h: int) -> float:
    return float(lib().oracle_f16_to_f32(int(h)))


def f32_to_f16(f: float) -> int:
    return int(lib().oracle_f32_to_f16(float(np.float32(f))))


def f32_to_f16_array(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_bf16_array(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


# --------------------------------------------------------------------------
# layout
# --------------------------------------------------------------------------

def layout(num_tokens: int, hidden: int, num_ranks: int, num_experts: int, elem_bytes: int = 2):
    """(status, Layout) for one rank's buffer (LLMoEBufferLayout constructor)."""
    L = Layout()
    rc = lib().oracle_layout(num_tokens, hidden, num_ranks, num_experts, elem_bytes, ctypes.byref(L))
    return rc, L


def size_hint(num_max_tokens: int, hidden: int, num_ranks: int, num_experts: int, elem_bytes: int = 2) -> int:
    """get_rdma_size_hint: total bytes of one rank's buffer, 0 if no layout."""
    return int(lib().oracle_size_hint(num_max_tokens, hidden, num_ranks, num_experts, elem_bytes))


# --------------------------------------------------------------------------
# route / dispatch / combine / clean
# --------------------------------------------------------------------------

def route(topk_idx: np.ndarray, num_experts: int):
    """Slots [R, T, K] (int32, -1 where masked) and counts [E, R] (int64)."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    R, T, K = idx.shape
    slot = np.empty((R, T, K), dtype=np.int32)
    cnt = np.empty((num_experts, R), dtype=np.int64)
    rc = lib().oracle_route(R, T, K, num_experts, _ptr(idx), _ptr(slot), _ptr(cnt))
    if rc != OK:
        raise OracleError(rc, "route")
    return slot, cnt


def dispatch(x: np.ndarray, topk_idx: np.ndarray, num_experts: int, num_max_tokens: int | None = None,
             dtype: str = "bf16"):
    """Expected dispatch result, compact.

    x: [R, T, H] payload values (uint16 bit patterns for bf16 / fp16,
    float32 for fp32); topk_idx: int64 [R, T, K].
    Returns dict with row_rank [n], row_index [n], msgs uint8 [n, 4 + H*size]
    (in (src, t, k) order over unmasked entries) and count_words int64 [R, E]
    (rank r's E recv-count words).
    """
    code, es, npdt = DTYPES[dtype]
    x = np.ascontiguousarray(x, dtype=npdt)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    R, T, H = x.shape
    K = idx.shape[2]
    assert idx.shape[:2] == (R, T)
    T_max = T if num_max_tokens is None else num_max_tokens
    cap = max(R * T * K, 1)
    row_rank = np.empty(cap, dtype=np.int64)
    row_index = np.empty(cap, dtype=np.int64)
    msgs = np.empty((cap, 4 + es * H), dtype=np.uint8)
    count_words = np.empty((R, num_experts), dtype=np.int64)
    n = ctypes.c_int64(0)
    rc = lib().oracle_dispatch(R, T_max, T, H, num_experts, K, code, _ptr(x), _ptr(idx), _ptr(row_rank),
                               _ptr(row_index), _ptr(msgs), _ptr(count_words), ctypes.addressof(n))
    if rc != OK:
        raise OracleError(rc, "dispatch")
    n = n.value
    return {"row_rank": row_rank[:n], "row_index": row_index[:n], "msgs": msgs[:n],
            "count_words": count_words, "n": n}


def combine(y_rows, topk_idx: np.ndarray, topk_w: np.ndarray, hidden: int, num_experts: int,
            num_max_tokens: int | None = None, dtype: str = "bf16"):
    """Expected combine result.

    y_rows: either an array [E * R * T_max, H] (dense expert outputs in
    receive-row order) or a pair (pool [P, H], row_map int64 [E * R * T_max])
    meaning row r is pool[row_map[r]]; values as for ``dispatch``.
    Returns (out [R, T, H] in the payload type's storage, flag_words int64 [R, E]).
    """
    code, es, npdt = DTYPES[dtype]
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    R, T, K = idx.shape
    assert w.shape == (R, T, K)
    T_max = T if num_max_tokens is None else num_max_tokens
    ptrs, keep = _row_pointers(y_rows, hidden, num_experts * R * T_max, dtype)
    out = np.empty((R, T, hidden), dtype=npdt)
    flag_words = np.empty((R, num_experts), dtype=np.int64)
    rc = lib().oracle_combine(R, T_max, T, hidden, num_experts, K, code, _ptr(ptrs), _ptr(idx), _ptr(w),
                              _ptr(out), _ptr(flag_words))
    del keep
    if rc != OK:
        raise OracleError(rc, "combine")
    return out, flag_words


def _row_pointers(y_rows, hidden: int, nrows: int, dtype: str = "bf16"):
    _, es, npdt = DTYPES[dtype]
    if isinstance(y_rows, tuple):
        pool, row_map = y_rows
        pool = np.ascontiguousarray(pool, dtype=npdt)
        row_map = np.ascontiguousarray(row_map, dtype=np.int64)
        assert pool.shape[1] == hidden and row_map.shape == (nrows,)
        return (pool.ctypes.data + row_map * (es * hidden)).astype(np.uint64), pool
    dense = np.ascontiguousarray(y_rows, dtype=npdt)
    assert dense.shape == (nrows, hidden)
    return (dense.ctypes.data + np.arange(nrows, dtype=np.uint64) * np.uint64(es * hidden)).astype(np.uint64), dense


def combine_staged(y_rows, topk_idx: np.ndarray, topk_w: np.ndarray, hidden: int, num_experts: int,
                   num_max_tokens: int | None = None, dtype: str = "bf16"):
    """Expected staged combine: dict with msg_rank [n], msg_row [n] (row of
    the source rank's combine receive region), msgs uint8 [n, 4 + H*size],
    out [R, T, H], flag_words int64 [R, E]."""
    code, es, npdt = DTYPES[dtype]
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    R, T, K = idx.shape
    T_max = T if num_max_tokens is None else num_max_tokens
    ptrs, keep = _row_pointers(y_rows, hidden, num_experts * R * T_max, dtype)
    cap = max(R * T * K, 1)
    msg_rank = np.empty(cap, dtype=np.int64)
    msg_row = np.empty(cap, dtype=np.int64)
    msgs = np.empty((cap, 4 + es * hidden), dtype=np.uint8)
    out = np.empty((R, T, hidden), dtype=npdt)
    flag_words = np.empty((R, num_experts), dtype=np.int64)
    n = ctypes.c_int64(0)
    rc = lib().oracle_combine_staged(R, T_max, T, hidden, num_experts, K, code, _ptr(ptrs), _ptr(idx), _ptr(w),
                                     _ptr(msg_rank), _ptr(msg_row), _ptr(msgs), _ptr(out), _ptr(flag_words),
                                     ctypes.addressof(n))
    del keep
    if rc != OK:
        raise OracleError(rc, "combine_staged")
    n = n.value
    return {"msg_rank": msg_rank[:n], "msg_row": msg_row[:n], "msgs": msgs[:n], "out": out,
            "flag_words": flag_words, "n": n}


def unpack(x: np.ndarray, topk_idx: np.ndarray, num_experts: int, num_max_tokens: int | None = None,
           dtype: str = "bf16"):
    """Expected unpack: dict with rows [n] (written rows of recv_x, in (src,
    t, k) order), recv_x [E * R * T_max, H] (unwritten rows zero) and
    recv_src int32 [E * R * T_max] (unwritten -1)."""
    code, es, npdt = DTYPES[dtype]
    x = np.ascontiguousarray(x, dtype=npdt)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    R, T, H = x.shape
    K = idx.shape[2]
    T_max = T if num_max_tokens is None else num_max_tokens
    nrows = num_experts * R * T_max
    recv_x = np.zeros((nrows, H), dtype=npdt)
    recv_src = np.full(nrows, -1, dtype=np.int32)
    rows = np.empty(max(R * T * K, 1), dtype=np.int64)
    n = ctypes.c_int64(0)
    rc = lib().oracle_unpack(R, T_max, T, H, num_experts, K, code, _ptr(x), _ptr(idx), _ptr(recv_x), _ptr(recv_src),
                             _ptr(rows), ctypes.addressof(n))
    if rc != OK:
        raise OracleError(rc, "unpack")
    return {"rows": rows[:n.value], "recv_x": recv_x, "recv_src": recv_src, "n": n.value}


def clean(num_ranks: int, num_experts: int) -> np.ndarray:
    """The set's signal words after a clean: [R, E] int64."""
    words = np.full((num_ranks, num_experts), -7, dtype=np.int64)
    lib().oracle_clean(num_ranks, num_experts, _ptr(words))
    return words
