"""Seeded synthetic attention inputs, shared by the CPU oracle tests and the CUDA path.

This module holds no attention arithmetic: it only draws numbers, rounds them to
bf16 and picks which query rows a comparison looks at.  Both sides of every
parity check read their inputs from here and from nowhere else.

Workloads (all tensors are ``[B, H, N, d]``, row-major, bf16):

* ``page``   B1 H1 N64 d16 causal: the worked example of the aiml.sh page
  "Speed up long contexts with FlashAttention" (``lab.py``, ``make_qkv`` and
  ``build_report``): one ``random.Random(42)`` stream drawing q, then k, then v,
  row-major, each value ``uniform(-0.8, 0.8)``.
* ``n1k``    B1 H32 N1024 d128 causal, iid U(-0.8, 0.8).
* ``n4k``    B1 H32 N4096 d128, causal and non-causal, iid U(-0.8, 0.8).
* ``b8n8k``  B8 H32 N8192 d128 causal, iid U(-0.8, 0.8)  (the throughput shape
  of the chipfoundryservices.com "edge/flashattention" model, ``inputs``).
* ``n32k``   B1 H32 N32768 d128 causal, Q,K ~ N(0, 3^2), V ~ N(0, 1): large
  logits that stress the running-max subtraction and the rescale.

The bf16 bit patterns are the contract: whatever draws them, the CPU oracle
and the GPU kernel consume the same bits.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple  # the mask settings this workload is run with
    dist: str      # "page", "uniform" or "normal3"
    seed: int
    # row selection for the oracle comparison (see ``select_rows``)
    rows: str = "all"
    rows_per_head: int = 0
    full_heads: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        """1/sqrt(d), computed in double and rounded once to fp32 (the value both sides use)."""
        return float(np.float32(1.0 / math.sqrt(self.d)))


WORKLOADS = {
    "page": Workload("page", 1, 1, 64, 16, (True,), "page", 42, rows="all"),
    "n1k": Workload("n1k", 1, 32, 1024, 128, (True,), "uniform", 1002, rows="all"),
    "n4k": Workload("n4k", 1, 32, 4096, 128, (True, False), "uniform", 1003,
                    rows="heads+sample", rows_per_head=512, full_heads=4),
    "b8n8k": Workload("b8n8k", 8, 32, 8192, 128, (True,), "uniform", 1004,
                      rows="sample+ends", rows_per_head=256),
    "n32k": Workload("n32k", 1, 32, 32768, 128, (True,), "normal3", 1005,
                     rows="sample+ends", rows_per_head=128),
}


def make_qkv_page(seq_len: int, head_dim: int, seed: int = 42):
    """The page's generator as fp64 lists (unrounded).

    One ``random.Random(seed)`` stream; all of q is drawn first, then k, then v;
    each matrix row-major; every value ``uniform(-0.8, 0.8)``.  The draw order is
    part of the page's worked example (its printed sample rows depend on it).
    """
    rng = random.Random(seed)
    mats = []
    for _ in range(3):
        mats.append([[rng.uniform(-0.8, 0.8) for _c in range(head_dim)]
                     for _r in range(seq_len)])
    return mats[0], mats[1], mats[2]


def _to_bf16(x: torch.Tensor) -> torch.Tensor:
    # round-to-nearest-even, which is what Tensor.to(bfloat16) does
    return x.to(torch.bfloat16).contiguous()


def make_inputs(w: Workload, B: int | None = None, H: int | None = None,
                N: int | None = None, d: int | None = None, seed: int | None = None):
    """Return (q, k, v) as CPU bf16 tensors of shape [B, H, N, d].

    Overriding B/H/N/d/seed keeps the workload's distribution at another size
    (used for ragged-tail and edge-case parity tests).
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    d = w.d if d is None else d
    seed = w.seed if seed is None else seed
    shape = (B, H, N, d)
    if w.dist == "page":
        if (B, H) != (1, 1):
            raise ValueError("the page generator describes one head")
        q, k, v = make_qkv_page(N, d, seed)
        return tuple(_to_bf16(torch.tensor(m, dtype=torch.float64).view(shape))
                     for m in (q, k, v))
    g = torch.Generator().manual_seed(seed)
    if w.dist == "uniform":
        out = []
        for _ in range(3):
            t = torch.rand(shape, generator=g, dtype=torch.float32)
            out.append(_to_bf16(t.mul_(1.6).sub_(0.8)))
        return tuple(out)
    if w.dist == "normal3":
        q = torch.randn(shape, generator=g, dtype=torch.float32).mul_(3.0)
        k = torch.randn(shape, generator=g, dtype=torch.float32).mul_(3.0)
        v = torch.randn(shape, generator=g, dtype=torch.float32)
        return _to_bf16(q), _to_bf16(k), _to_bf16(v)
    raise ValueError(f"unknown distribution {w.dist!r}")


def select_rows(w: Workload, B: int | None = None, H: int | None = None,
                N: int | None = None, seed: int | None = None) -> np.ndarray:
    """Query rows the oracle checks, as an int64 array of (bh, i) pairs sorted by (bh, i).

    * ``all``          every row of every head;
    * ``heads+sample`` every row of ``full_heads`` seeded heads, plus
      ``rows_per_head`` seeded distinct rows from each other head;
    * ``sample+ends``  rows 0 and N-1 of every head plus seeded distinct rows
      up to ``rows_per_head`` per head.
    The selection uses its own generator (seed + 7919), independent of the data.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    seed = (w.seed if seed is None else seed) + 7919
    BH = B * H
    g = torch.Generator().manual_seed(seed)
    pairs = []
    if w.rows == "all":
        for bh in range(BH):
            pairs.extend((bh, i) for i in range(N))
    elif w.rows == "heads+sample":
        full = set(torch.randperm(BH, generator=g)[: w.full_heads].tolist())
        for bh in range(BH):
            if bh in full or N <= w.rows_per_head:
                pairs.extend((bh, i) for i in range(N))
            else:
                rows = torch.randperm(N, generator=g)[: w.rows_per_head]
                pairs.extend((bh, int(i)) for i in sorted(rows.tolist()))
    elif w.rows == "sample+ends":
        for bh in range(BH):
            if N <= w.rows_per_head:
                pairs.extend((bh, i) for i in range(N))
                continue
            inner = torch.randperm(N - 2, generator=g)[: w.rows_per_head - 2] + 1
            rows = sorted({0, N - 1, *inner.tolist()})
            pairs.extend((bh, int(i)) for i in rows)
    else:
        raise ValueError(w.rows)
    return np.asarray(pairs, dtype=np.int64).reshape(-1, 2)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a CPU bf16 tensor, as a flat uint16 numpy array."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
