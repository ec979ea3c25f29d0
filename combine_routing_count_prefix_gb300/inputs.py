"""Seeded synthetic inputs for the MoE dispatch / combine data path.

This module only draws inputs: token activations ``x``, routing ``topk_idx``,
routing weights ``topk_w`` and the expert outputs ``y``.  It holds none of the
dispatch / combine arithmetic (no slots, no counts, no placement), so the CUDA
path and the CPU oracle can both be fed from it without sharing any of the
method.

All draws come from one CPU ``torch.Generator`` seeded per call, in a fixed
order: x, routing, weights, mask, expert-output pool.  Payload values are
fp32 draws in the payload type: bf16 and fp16 cast by PyTorch (round to
nearest even) and handed out as their uint16 bit patterns, fp32 as is.

Workloads (tokens per rank T, hidden H, experts E over R simulated ranks,
top-k K):

=============  ==  ====  =====  ===  =  ====================================
name           R   T     H      E    K  routing / values
=============  ==  ====  =====  ===  =  ====================================
tiny           2   8     256    8    2  uniform distinct; x ~ N(0,1)
dsv3           8   128   7168   256  8  DeepSeek-V3-shaped decode; uniform
skewed         8   128   4096   64   6  Zipf(1.2) w/o replacement, 10% -1
many_small     32  16    2048   128  4  uniform; x ~ U(-1,1)
large          8   1024  7168   256  8  uniform; worst-case layout ~120 GB
dense16        8   256   7168   16   8  uniform; small layout (2.4 GB with
                                        y), kernel traffic above L2 size:
                                        the profiling case for the dsv3
                                        kernels (same row length and top-k)
=============  ==  ====  =====  ===  =  ====================================

Expert outputs ``y`` are the dense [E * R * T_max, H] bf16 matrix the combine
reads (one row per receive row).  Only the rows the routing uses are read, so
``y`` is described compactly by a pool of N(0,1) rows and a row map
(``y[r] = pool[row_map[r]]``): when the matrix has at most ``POOL_ROWS`` rows
the map is the identity; otherwise it is a SplitMix64 hash of the row index
(no stride of rows shares content systematically).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

POOL_ROWS = 16384


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int  # simulated ranks (segments)
    T: int  # max tokens per rank (the layout's num_tokens)
    H: int  # hidden
    E: int  # experts
    K: int  # top-k
    routing: str = "uniform"  # "uniform" | "zipf"
    zipf_s: float = 0.0
    mask_p: float = 0.0
    x_dist: str = "normal"  # "normal" | "uniform"

    @property
    def L(self) -> int:
        return self.E // self.R

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def describe(self) -> str:
        extra = f", zipf s={self.zipf_s}" if self.routing == "zipf" else ""
        mask = f", {self.mask_p:.0%} masked" if self.mask_p else ""
        return (f"R={self.R} T={self.T} H={self.H} E={self.E} K={self.K}, {self.routing}{extra}{mask}, "
                f"x~{'N(0,1)' if self.x_dist == 'normal' else 'U(-1,1)'}")


WORKLOADS = {
    "tiny": Workload("tiny", 2, 8, 256, 8, 2),
    "dsv3": Workload("dsv3", 8, 128, 7168, 256, 8),
    "skewed": Workload("skewed", 8, 128, 4096, 64, 6, routing="zipf", zipf_s=1.2, mask_p=0.10),
    "many_small": Workload("many_small", 32, 16, 2048, 128, 4, x_dist="uniform"),
    "large": Workload("large", 8, 1024, 7168, 256, 8),
    "dense16": Workload("dense16", 8, 256, 7168, 16, 8),
}


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _payload(t: torch.Tensor, dtype: str) -> np.ndarray:
    """fp32 draws as the payload type: bf16 / fp16 bit patterns (uint16, cast
    by PyTorch with round to nearest even) or fp32 values."""
    if dtype == "bf16":
        return _bf16_bits(t)
    if dtype == "fp16":
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp32":
        return t.numpy().astype(np.float32)
    raise ValueError(dtype)


def splitmix64(v: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Steele, Lea, Flood 2014) on uint64 words."""
    z = v.astype(np.uint64) + np.uint64(0x9E3779B97F4A7C15)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def make_inputs(w: Workload, seed: int = 0, tokens: int | None = None, pool_rows: int = POOL_ROWS,
                dtype: str = "bf16") -> dict:
    """Draw one round's inputs.

    tokens: tokens per rank in this call (default T); the layout and the
    expert-output matrix stay sized for T.
    dtype: payload type of x and y ("bf16", "fp16" as uint16 bit patterns,
    "fp32" as float32).
    Returns numpy arrays: x [R, tokens, H], topk_idx int64 [R, tokens, K]
    (-1 = masked), topk_w float32 [R, tokens, K], y_pool [P, H],
    y_row_map int64 [E * R * T].
    """
    n_tok = w.T if tokens is None else tokens
    assert 0 <= n_tok <= w.T and w.E % w.R == 0 and 1 <= w.K <= w.E
    g = torch.Generator().manual_seed(seed)
    R, H, E, K = w.R, w.H, w.E, w.K
    rows = R * n_tok

    # x
    if w.x_dist == "normal":
        xf = torch.randn(rows * H, generator=g, dtype=torch.float32)
    else:
        xf = torch.rand(rows * H, generator=g, dtype=torch.float32) * 2.0 - 1.0
    x = _payload(xf, dtype).reshape(R, n_tok, H)
    del xf

    # routing: K distinct experts per token
    if rows == 0:
        idx = torch.empty((0, K), dtype=torch.int64)
    elif w.routing == "uniform":
        idx = torch.rand(rows, E, generator=g).argsort(dim=1)[:, :K].contiguous()
    elif w.routing == "zipf":
        p = (torch.arange(E, dtype=torch.float64) + 1.0) ** (-w.zipf_s)
        idx = torch.multinomial(p.expand(rows, E), K, replacement=False, generator=g)
    else:
        raise ValueError(w.routing)

    # weights: softmax over the K choices, fp32
    wts = torch.softmax(torch.randn(rows, K, generator=g, dtype=torch.float32), dim=1)

    # mask: each top-k entry independently dropped to -1
    if w.mask_p > 0 and rows > 0:
        drop = torch.rand(rows, K, generator=g) < w.mask_p
        idx = idx.masked_fill(drop, -1)

    # expert-output pool and row map
    nrows = E * R * w.T
    P = min(nrows, pool_rows)
    pool = _payload(torch.randn(P * H, generator=g, dtype=torch.float32), dtype).reshape(P, H)
    if nrows <= pool_rows:
        row_map = np.arange(nrows, dtype=np.int64)
    else:
        h = splitmix64(np.arange(nrows, dtype=np.uint64) ^ np.uint64(seed * 0x5851F42D4C957F2D & (2**64 - 1)))
        row_map = (h % np.uint64(P)).astype(np.int64)

    return {
        "x": np.ascontiguousarray(x),
        "topk_idx": idx.reshape(R, n_tok, K).numpy().astype(np.int64),
        "topk_w": wts.reshape(R, n_tok, K).numpy().astype(np.float32),
        "y_pool": np.ascontiguousarray(pool),
        "y_row_map": row_map,
    }


def dense_y(inp: dict) -> np.ndarray:
    """The expert-output matrix [E * R * T, H] materialised on the host."""
    return inp["y_pool"][inp["y_row_map"]]
