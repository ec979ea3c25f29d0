"""Python binding of libllmoe.so (include/llmoe.h).

Argument marshalling only: every step of the data path runs in the CUDA
kernels of the library.  Importing this module loads the library and raises
ImportError when it has not been built; there is no CPU or PyTorch fallback.

The functions carry the C names.  Tensor arguments are CUDA ``torch.Tensor``s
(contiguous, of the dtype the C call documents) or raw device addresses given
as ``int``; ``stream`` defaults to PyTorch's current stream.  ``RankBuffers``
allocates the R rank buffers with PyTorch (one device allocation) and hands
out ``llmoe_buf_set_t`` structs for either buffer set.
"""
from __future__ import annotations

import ctypes
import os

import torch

# LLMOE_LIBRARY selects another build of the same library (the phase-trace
# build of phase_budget.py); by default the in-tree libllmoe.so
_SO = os.environ.get("LLMOE_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build",
                                                       "libllmoe.so")
if not os.path.exists(_SO):
    raise ImportError(f"{_SO} is missing: build it with combine_routing_count_prefix_gb300.build.build()")
_lib = ctypes.CDLL(_SO)

LLMOE_SUCCESS = 0
LLMOE_ERR_CUDA = 1
LLMOE_ERR_INVALID_ARGUMENT = 4
LLMOE_ERR_INVALID_USAGE = 5

LLMOE_DEV_OK = 0
LLMOE_DEV_BAD_EXPERT = 1
LLMOE_DEV_DUPLICATE = 2
LLMOE_DEV_STALE_SIGNAL = 3
LLMOE_DEV_SLOT_RANGE = 4
LLMOE_DEV_TIMEOUT = 5
LLMOE_DEV_BAD_MESSAGE = 6

LLMOE_FLAG_INPUTS_READY = 1
LLMOE_FLAG_CLEAN_OTHER_SET = 2

LLMOE_STATIC_MAX_RANKS = 1024

LLMOE_MAX_TOPK = 32
LLMOE_MAX_EXPERTS = 8192

EXPORTS = ("llmoe_layout_bytes", "llmoe_layout_bytes_dtype", "llmoe_layout_offsets", "llmoe_layout_offsets_dtype",
           "llmoe_route", "llmoe_dispatch", "llmoe_combine", "llmoe_combine_staged", "llmoe_unpack",
           "llmoe_dispatch_unpack",
           "llmoe_signal_workspace_bytes", "llmoe_dispatch_signaled", "llmoe_dispatch_signaled_static", "llmoe_clean",
           "llmoe_get_error",
           "llmoe_status_string")

LLMOE_DTYPE_BF16, LLMOE_DTYPE_FP16, LLMOE_DTYPE_FP32 = 0, 1, 2
DTYPE_CODES = {"bf16": LLMOE_DTYPE_BF16, "fp16": LLMOE_DTYPE_FP16, "fp32": LLMOE_DTYPE_FP32}
DTYPE_BYTES = {LLMOE_DTYPE_BF16: 2, LLMOE_DTYPE_FP16: 2, LLMOE_DTYPE_FP32: 4}


class llmoe_buf_set_t(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_void_p),
        ("rank_stride", ctypes.c_uint64),
        ("num_max_tokens", ctypes.c_int32),
        ("num_tokens", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("num_ranks", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("num_topk", ctypes.c_int32),
        ("set", ctypes.c_int32),
        ("err", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("dtype", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_BS = ctypes.POINTER(llmoe_buf_set_t)
_lib.llmoe_layout_bytes.argtypes = [_I, _I, _I, _I]
_lib.llmoe_layout_bytes.restype = ctypes.c_size_t
_lib.llmoe_layout_offsets.argtypes = [_I, _I, _I, _I, _I, _P, _P, _P]
_lib.llmoe_layout_offsets.restype = _I
_lib.llmoe_layout_bytes_dtype.argtypes = [_I, _I, _I, _I, _I]
_lib.llmoe_layout_bytes_dtype.restype = ctypes.c_size_t
_lib.llmoe_layout_offsets_dtype.argtypes = [_I, _I, _I, _I, _I, _I, _P, _P, _P]
_lib.llmoe_layout_offsets_dtype.restype = _I
_lib.llmoe_route.argtypes = [_P, _P, _P, _BS, _P]
_lib.llmoe_route.restype = _I
_lib.llmoe_dispatch.argtypes = [_P, _P, _BS, _P]
_lib.llmoe_dispatch.restype = _I
_lib.llmoe_combine.argtypes = [_P, _P, _P, _P, _BS, _P]
_lib.llmoe_combine.restype = _I
_lib.llmoe_combine_staged.argtypes = [_P, _P, _P, _P, _BS, _P]
_lib.llmoe_combine_staged.restype = _I
_lib.llmoe_unpack.argtypes = [_P, _P, _BS, _P]
_lib.llmoe_unpack.restype = _I
_lib.llmoe_dispatch_unpack.argtypes = [_P, _P, _P, _P, _BS, _P]
_lib.llmoe_dispatch_unpack.restype = _I
_lib.llmoe_signal_workspace_bytes.argtypes = [_BS]
_lib.llmoe_signal_workspace_bytes.restype = ctypes.c_size_t
_lib.llmoe_dispatch_signaled.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int64, _BS, _P]
_lib.llmoe_dispatch_signaled.restype = _I
_lib.llmoe_dispatch_signaled_static.argtypes = [_P, _P, _P, _P, ctypes.c_int64, _BS, _P]
_lib.llmoe_dispatch_signaled_static.restype = _I
_lib.llmoe_clean.argtypes = [_BS, _P]
_lib.llmoe_clean.restype = _I
_lib.llmoe_get_error.argtypes = [_BS, _P, ctypes.POINTER(ctypes.c_int32), _I]
_lib.llmoe_get_error.restype = _I
_lib.llmoe_status_string.argtypes = [_I]
_lib.llmoe_status_string.restype = ctypes.c_char_p


class LLMoEError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call}: {llmoe_status_string(status)} ({status})")
        self.status = status


def _check(rc: int, call: str) -> None:
    if rc != LLMOE_SUCCESS:
        raise LLMoEError(rc, call)


_DTYPES = {
    "payload": (torch.bfloat16, torch.float16, torch.int16, torch.uint16, torch.float32),
    "bf16": (torch.bfloat16, torch.int16, torch.uint16),
    "i64": (torch.int64,),
    "i32": (torch.int32,),
    "f32": (torch.float32,),
}


def _addr(t, kind: str) -> int:
    """Device address of a tensor argument (or an int passed through)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a CUDA tensor or an address, got {type(t).__name__}")
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    if t.dtype not in _DTYPES[kind]:
        raise TypeError(f"expected dtype {_DTYPES[kind][0]}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def llmoe_status_string(status: int) -> str:
    return _lib.llmoe_status_string(status).decode()


def llmoe_layout_bytes(num_max_tokens: int, hidden: int, num_ranks: int, num_experts: int) -> int:
    return int(_lib.llmoe_layout_bytes(num_max_tokens, hidden, num_ranks, num_experts))


def llmoe_layout_offsets(num_max_tokens: int, hidden: int, num_ranks: int, num_experts: int, set: int):
    send, recv, sig = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.llmoe_layout_offsets(num_max_tokens, hidden, num_ranks, num_experts, set, ctypes.byref(send),
                                     ctypes.byref(recv), ctypes.byref(sig)), "llmoe_layout_offsets")
    return send.value, recv.value, sig.value


def llmoe_layout_bytes_dtype(num_max_tokens: int, hidden: int, num_ranks: int, num_experts: int, dtype: int) -> int:
    return int(_lib.llmoe_layout_bytes_dtype(num_max_tokens, hidden, num_ranks, num_experts, dtype))


def llmoe_layout_offsets_dtype(num_max_tokens: int, hidden: int, num_ranks: int, num_experts: int, dtype: int,
                               set: int):
    send, recv, sig = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.llmoe_layout_offsets_dtype(num_max_tokens, hidden, num_ranks, num_experts, dtype, set,
                                           ctypes.byref(send), ctypes.byref(recv), ctypes.byref(sig)),
           "llmoe_layout_offsets_dtype")
    return send.value, recv.value, sig.value


def llmoe_route(topk_idx, slot, counts, bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_route(_addr(topk_idx, "i64"), _addr(slot, "i32"), _addr(counts, "i64"), ctypes.byref(bs),
                            _stream(stream)), "llmoe_route")


def llmoe_dispatch(x, topk_idx, bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_dispatch(_addr(x, "payload"), _addr(topk_idx, "i64"), ctypes.byref(bs), _stream(stream)),
           "llmoe_dispatch")


def llmoe_combine(y, topk_idx, topk_w, out, bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_combine(_addr(y, "payload"), _addr(topk_idx, "i64"), _addr(topk_w, "f32"), _addr(out, "payload"),
                              ctypes.byref(bs), _stream(stream)), "llmoe_combine")


def llmoe_combine_staged(y, topk_idx, topk_w, out, bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_combine_staged(_addr(y, "payload"), _addr(topk_idx, "i64"), _addr(topk_w, "f32"),
                                     _addr(out, "payload"), ctypes.byref(bs), _stream(stream)), "llmoe_combine_staged")


def llmoe_unpack(recv_x, recv_src, bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_unpack(_addr(recv_x, "payload"), _addr(recv_src, "i32"), ctypes.byref(bs), _stream(stream)),
           "llmoe_unpack")


def llmoe_dispatch_unpack(x, topk_idx, recv_x, recv_src, bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_dispatch_unpack(_addr(x, "payload"), _addr(topk_idx, "i64"), _addr(recv_x, "payload"),
                                      _addr(recv_src, "i32"), ctypes.byref(bs), _stream(stream)),
           "llmoe_dispatch_unpack")


def llmoe_signal_workspace_bytes(bs: llmoe_buf_set_t) -> int:
    return int(_lib.llmoe_signal_workspace_bytes(ctypes.byref(bs)))


def llmoe_dispatch_signaled(x, topk_idx, recv_x, recv_src, workspace, spin_limit: int, bs: llmoe_buf_set_t,
                            stream=None) -> None:
    _check(_lib.llmoe_dispatch_signaled(_addr(x, "payload"), _addr(topk_idx, "i64"), _addr(recv_x, "payload"),
                                        _addr(recv_src, "i32"), _addr(workspace, "i32"), int(spin_limit),
                                        ctypes.byref(bs), _stream(stream)), "llmoe_dispatch_signaled")


def llmoe_dispatch_signaled_static(x, topk_idx, recv_x, recv_src, spin_limit: int, bs: llmoe_buf_set_t,
                                   stream=None) -> None:
    """llmoe_dispatch_signaled with the library's own fixed device workspace,
    for callers that cannot allocate one (at most LLMOE_STATIC_MAX_RANKS
    ranks; calls must not overlap on the GPU)."""
    _check(_lib.llmoe_dispatch_signaled_static(_addr(x, "payload"), _addr(topk_idx, "i64"),
                                               _addr(recv_x, "payload"), _addr(recv_src, "i32"), int(spin_limit),
                                               ctypes.byref(bs), _stream(stream)), "llmoe_dispatch_signaled_static")


def llmoe_clean(bs: llmoe_buf_set_t, stream=None) -> None:
    _check(_lib.llmoe_clean(ctypes.byref(bs), _stream(stream)), "llmoe_clean")


def llmoe_get_error(bs: llmoe_buf_set_t, stream=None, reset: bool = False) -> int:
    code = ctypes.c_int32(-1)
    _check(_lib.llmoe_get_error(ctypes.byref(bs), _stream(stream), ctypes.byref(code), int(reset)),
           "llmoe_get_error")
    return code.value


class Bound:
    """One C-ABI call with its arguments marshalled once, for tight loops:
    calling it issues the call and raises on a non-zero status."""

    __slots__ = ("fn", "args", "name", "keep")

    def __init__(self, name: str, args: tuple, keep=()):
        self.fn = getattr(_lib, name)
        self.args = args
        self.name = name
        self.keep = keep  # objects the marshalled pointers refer to

    def __call__(self) -> None:
        rc = self.fn(*self.args)
        if rc != LLMOE_SUCCESS:
            raise LLMoEError(rc, self.name)


def bind_dispatch(x, topk_idx, bs: llmoe_buf_set_t, stream=None) -> Bound:
    return Bound("llmoe_dispatch", (_addr(x, "payload"), _addr(topk_idx, "i64"), ctypes.byref(bs), _stream(stream)),
                 (x, topk_idx, bs))


def bind_combine(y, topk_idx, topk_w, out, bs: llmoe_buf_set_t, stream=None) -> Bound:
    return Bound("llmoe_combine", (_addr(y, "payload"), _addr(topk_idx, "i64"), _addr(topk_w, "f32"),
                                   _addr(out, "payload"), ctypes.byref(bs), _stream(stream)),
                 (y, topk_idx, topk_w, out, bs))


def bind_clean(bs: llmoe_buf_set_t, stream=None) -> Bound:
    return Bound("llmoe_clean", (ctypes.byref(bs), _stream(stream)), (bs,))


def round_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


class RankBuffers:
    """R rank buffers of one LLMoEBufferLayout<bf16> each, in one allocation.

    rank_stride is the layout size rounded up to 256 bytes plus ``guard``
    bytes, so a test can fill the gaps with a canary and check them.
    """

    def __init__(self, num_max_tokens: int, hidden: int, num_ranks: int, num_experts: int,
                 device="cuda", guard: int = 0, fill: int | None = None, dtype: str = "bf16"):
        self.T, self.H, self.R, self.E = num_max_tokens, hidden, num_ranks, num_experts
        self.dtype = DTYPE_CODES[dtype]
        self.layout_bytes = llmoe_layout_bytes_dtype(num_max_tokens, hidden, num_ranks, num_experts, self.dtype)
        if self.layout_bytes == 0:
            raise LLMoEError(LLMOE_ERR_INVALID_ARGUMENT, "llmoe_layout_bytes_dtype")
        self.rank_stride = round_up(self.layout_bytes + guard, 256)
        self.storage = torch.empty(self.rank_stride * num_ranks, dtype=torch.uint8, device=device)
        if fill is not None:
            self.storage.fill_(fill)
        self.offsets = [llmoe_layout_offsets_dtype(num_max_tokens, hidden, num_ranks, num_experts, self.dtype, s)
                        for s in (0, 1)]

    @property
    def msg_bytes(self) -> int:
        return 4 + DTYPE_BYTES[self.dtype] * self.H

    def buf_set(self, set: int, num_topk: int, num_tokens: int | None = None, err=None,
                flags: int = 0) -> llmoe_buf_set_t:
        return llmoe_buf_set_t(
            base=self.storage.data_ptr(), rank_stride=self.rank_stride, num_max_tokens=self.T,
            num_tokens=self.T if num_tokens is None else num_tokens, hidden=self.H, num_ranks=self.R,
            num_experts=self.E, num_topk=num_topk, set=set, err=None if err is None else _addr(err, "i32"),
            flags=flags, dtype=self.dtype)

    def rank_view(self, r: int) -> torch.Tensor:
        return self.storage[r * self.rank_stride:(r + 1) * self.rank_stride]

    def recv_rows(self, set: int) -> torch.Tensor:
        """[R, E * T, 4 + 2H] uint8 view of every rank's receive region."""
        off = self.offsets[set][1]
        rows = self.E * self.T
        return self.storage.as_strided((self.R, rows, self.msg_bytes), (self.rank_stride, self.msg_bytes, 1),
                                       storage_offset=off)

    def signal_words(self, set: int) -> torch.Tensor:
        """[R, E] int64 view of every rank's signal words of a set."""
        off = self.offsets[set][2]
        assert off % 8 == 0 and self.rank_stride % 8 == 0
        w = self.storage.view(torch.int64)
        return w.as_strided((self.R, self.E), (self.rank_stride // 8, 1), storage_offset=off // 8)
