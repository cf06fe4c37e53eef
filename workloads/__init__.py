"""Seeded synthetic inputs for the softmax and softmax+TopK workloads.

This module only draws numbers: it holds none of the softmax arithmetic, so
both the float64 oracle (tests) and the CUDA library (tests, bench) consume
the very same tensors from here without sharing any of the method's code.

Workloads (rows x cols, dtype, distribution, seed):

  softmax_64x1024_f32         64 x 1024 fp32, N(0, 1),                       seed 1001
  softmax_4096x32000_f32      4096 x 32000 fp32, N(0, 2),                    seed 1002
  softmax_8192x128256_bf16    8192 x 128256 bf16, N(0, 3); per row 4 spikes
                              of exactly +40.0 and 1% of entries -inf,       seed 1003
  topk_256x50257_f32          256 x 50257 fp32, N(0, 4) (K in {8, 64}),      seed 1004
  causal_1048576x128_f32      1048576 x 128 fp32, N(0, 1), x[r, c] = -inf
                              for c > r % 128,                               seed 1005
  increasing_65536x4096_f32   65536 x 4096 fp32, each row sorted N(0, 1)
                              draws made strictly increasing,                seed 1006
  softmax_4096x50257_f32      4096 x 50257 fp32, N(0, 2),                    seed 1009
                              (rows that are not a whole number of 16-byte
                              vectors: every row starts at another offset
                              inside its 16-byte block; the row length of the
                              TopK workload, used as a softmax case)

Attention (batch x heads x seq_len x head_dim, Q, K, V bf16, all N(0, 1)):

  attention_4x16x4096x128_bf16  64 (batch, head) slices of 4096 x 128,       seed 1007
                                with and without the causal mask
  attention_1x2x300x64_bf16     small case for the oracle (ragged tile),     seed 1008

Readings of the workload text:
  * "N(0, s)": s is the standard deviation, x = s * randn.
  * "4 spikes at +40 at random positions": row r gets one spike in each quarter
    of its columns, at a uniformly drawn offset inside the quarter, so the 4
    positions are distinct by construction; the spike value is exactly 40.0
    (representable in bf16), making 4 exact ties for the row maximum.
  * "1% entries set to -inf": every non-spike entry is -inf independently with
    probability 0.01; spikes are never masked, so no row is all -inf.
  * "strictly increasing rows": sort N(0, 1) draws ascending, then lift any
    repeated value to the next representable float above its left neighbour.

All draws use a ``torch.Generator`` seeded with the workload seed on the
device the tensor is made on.  CPU and CUDA generators give different
streams; a test therefore makes one tensor and hands that same tensor to the
oracle (after a host copy) and to the library.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    cols: int
    dtype: str            # "f32" or "bf16": the input element type
    sigma: float = 1.0
    seed: int = 0
    kind: str = "normal"  # normal | spikes | causal | increasing
    ks: tuple = field(default_factory=tuple)  # K values for the TopK workload
    op: str = "softmax"   # softmax | topk

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, rows: int | None = None, cols: int | None = None) -> "Workload":
        """The same recipe on a smaller (rows, cols) grid, for parity tests."""
        return replace(self, rows=rows or self.rows, cols=cols or self.cols)


WORKLOADS = {
    w.name: w for w in [
        Workload("softmax_64x1024_f32", 64, 1024, "f32", 1.0, 1001),
        Workload("softmax_4096x32000_f32", 4096, 32000, "f32", 2.0, 1002),
        Workload("softmax_8192x128256_bf16", 8192, 128256, "bf16", 3.0, 1003, kind="spikes"),
        Workload("topk_256x50257_f32", 256, 50257, "f32", 4.0, 1004, ks=(8, 64), op="topk"),
        Workload("causal_1048576x128_f32", 1048576, 128, "f32", 1.0, 1005, kind="causal"),
        Workload("increasing_65536x4096_f32", 65536, 4096, "f32", 1.0, 1006, kind="increasing"),
        Workload("softmax_4096x50257_f32", 4096, 50257, "f32", 2.0, 1009),
    ]
}

SPIKE_VALUE = 40.0
SPIKES_PER_ROW = 4
NEG_INF_FRACTION = 0.01
CAUSAL_PERIOD = 128


def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make(w: Workload, device="cpu", seed: int | None = None, row_offset: int = 0) -> torch.Tensor:
    """Draw the [rows, cols] input of workload ``w`` on ``device``.

    ``row_offset`` shifts the row numbering used by the causal mask, so a
    slice of a large causal workload can be drawn on its own.
    """
    device = torch.device(device)
    g = _generator(device, w.seed if seed is None else seed)
    rows, cols = w.rows, w.cols
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    if w.sigma != 1.0:
        x.mul_(w.sigma)
    if w.kind == "spikes":
        _plant_spikes_and_mask(x, g)
    elif w.kind == "causal":
        r = torch.arange(row_offset, row_offset + rows, device=device) % CAUSAL_PERIOD
        c = torch.arange(cols, device=device)
        x.masked_fill_(c[None, :] > r[:, None], float("-inf"))
    elif w.kind == "increasing":
        x = strictly_increasing(torch.sort(x, dim=1).values)
    return x.to(w.torch_dtype)


def _plant_spikes_and_mask(x: torch.Tensor, g: torch.Generator) -> None:
    rows, cols = x.shape
    dev = x.device
    mask = torch.rand(rows, cols, generator=g, device=dev) < NEG_INF_FRACTION
    x.masked_fill_(mask, float("-inf"))
    quarter = max(cols // SPIKES_PER_ROW, 1)
    for q in range(min(SPIKES_PER_ROW, cols)):
        width = quarter if q < SPIKES_PER_ROW - 1 else cols - q * quarter
        pos = q * quarter + torch.randint(0, width, (rows,), generator=g, device=dev)
        x.scatter_(1, pos[:, None], SPIKE_VALUE)


def strictly_increasing(x: torch.Tensor) -> torch.Tensor:
    """Lift repeated values of ascending rows until every row strictly increases."""
    x = x.clone()
    while True:
        dup = x[:, 1:] <= x[:, :-1]
        if not bool(dup.any()):
            return x
        nxt = torch.nextafter(x[:, :-1], torch.full_like(x[:, :-1], float("inf")))
        x[:, 1:] = torch.where(dup, nxt, x[:, 1:])


def plant_ties(x: torch.Tensor, g_seed: int = 7, per_row: int = 6) -> torch.Tensor:
    """Copy each row's maximum to ``per_row`` other random positions (exact ties)."""
    x = x.clone()
    rows, cols = x.shape
    g = _generator(x.device, g_seed)
    pos = torch.randint(0, cols, (rows, per_row), generator=g, device=x.device)
    top = x.max(dim=1, keepdim=True).values.expand(rows, per_row)
    x.scatter_(1, pos, top.contiguous())
    return x


@dataclass(frozen=True)
class AttentionWorkload:
    name: str
    batch: int
    heads: int
    seq_len: int
    head_dim: int
    seed: int = 0

    @property
    def bh(self) -> int:
        return self.batch * self.heads

    def scaled(self, batch: int | None = None, heads: int | None = None,
               seq_len: int | None = None) -> "AttentionWorkload":
        return replace(self, batch=batch or self.batch, heads=heads or self.heads,
                       seq_len=seq_len or self.seq_len)


ATTENTION_WORKLOADS = {
    w.name: w for w in [
        AttentionWorkload("attention_4x16x4096x128_bf16", 4, 16, 4096, 128, 1007),
        AttentionWorkload("attention_1x2x300x64_bf16", 1, 2, 300, 64, 1008),
    ]
}


def make_attention(w: AttentionWorkload, device="cpu", seed: int | None = None):
    """Draw (Q, K, V), each [batch * heads, seq_len, head_dim] bf16 N(0, 1)."""
    device = torch.device(device)
    g = _generator(device, w.seed if seed is None else seed)
    shape = (w.bh, w.seq_len, w.head_dim)
    return tuple(torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
                 for _ in range(3))
