"""Seeded synthetic inputs and block masks for block-sparse attention.

This module holds no attention arithmetic: it only draws the random tensors
and builds the boolean block masks and their BSR encoding.  Both the CUDA
path (through the C-ABI) and the CPU oracle consume what it produces, so it
is the one piece of code the two sides share.

Mask shapes follow the attention workloads of the trnsparse pages
("trnsparse 0.7.0 -> 0.9.0" diff, ``benchmarks/bench_native_trn2.py``,
``block_mask`` / ``mask_bsr_from_block_mask``): a boolean ``nb x nb`` block
mask is turned into block-row pointers and block-column indices in row-major
order, so the columns of one block-row ascend and never repeat.  The band
radii, dilation and density values are the ones of the five workloads this
library is measured on (listed in ``WORKLOADS``).

Tensors are drawn with ``torch.Generator().manual_seed(seed)`` and
``torch.randn`` in the order Q, K, V, dO, as the pages' bench does
(``section_attn``), then scaled by ``std`` and rounded to the operand dtype.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

BLOCK = 128


def block_mask(kind: str, nb: int, *, radius: int = 1, p: float = 0.0, seed: int = 1) -> np.ndarray:
    """Boolean ``[nb, nb]`` block mask; entry (m, n) is True iff block (m, n) is stored.

    kinds:
      ``local``    |m - n| <= radius
      ``dilated``  |m - n| <= radius and (m - n) even
      ``global``   |m - n| <= radius, plus all of block row 0 and block column 0
      ``random``   diagonal always kept; every off-diagonal block kept iid with
                   probability ``p`` (one ``torch.rand`` draw seeded with ``seed``)
      ``full``     every block
      ``diag``     the diagonal only
    """
    m = np.arange(nb)[:, None]
    n = np.arange(nb)[None, :]
    d = m - n
    if kind == "local":
        bm = np.abs(d) <= radius
    elif kind == "dilated":
        bm = (np.abs(d) <= radius) & (d % 2 == 0)
    elif kind == "global":
        bm = np.abs(d) <= radius
        bm[0, :] = True
        bm[:, 0] = True
    elif kind == "random":
        g = torch.Generator().manual_seed(seed)
        u = torch.rand(nb, nb, generator=g, dtype=torch.float64).numpy()
        bm = u < p
        bm[np.arange(nb), np.arange(nb)] = True
    elif kind == "full":
        bm = np.ones((nb, nb), dtype=bool)
    elif kind == "diag":
        bm = np.eye(nb, dtype=bool)
    else:
        raise ValueError(f"unknown mask kind {kind!r}")
    return np.ascontiguousarray(bm.astype(bool))


def bsr_from_block_mask(bm: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Row-major BSR structure of a boolean block mask: (row_ptr int32 [nb+1], col_idx int32 [nnzb])."""
    bm = np.asarray(bm, dtype=bool)
    counts = bm.sum(axis=1)
    row_ptr = np.zeros(bm.shape[0] + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum(counts)
    col_idx = np.nonzero(bm)[1].astype(np.int32)
    return row_ptr, np.ascontiguousarray(col_idx)


_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def make_spmm(n_brows: int, n_bcols: int, n_cols: int, p: float, dtype: str = "bf16", seed: int = 0):
    """Inputs of Y = A X for a random BSR matrix A: (block mask, blocks, X) as CPU tensors.

    Block (m, k) is stored iid with probability ``p`` (one ``torch.rand`` draw
    of the ``[n_brows, n_bcols]`` grid, so block rows may be empty); the
    stored blocks ``[nnzb, 128, 128]`` in row-major BSR order and X
    ``[n_bcols * 128, n_cols]`` are iid N(0, 1), drawn in that order from one
    seeded generator and rounded to ``dtype``.
    """
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand(n_brows, n_bcols, generator=g, dtype=torch.float64) < p).numpy()
    nnzb = int(bm.sum())
    blocks = torch.randn(nnzb, BLOCK, BLOCK, generator=g, dtype=torch.float32).to(_TORCH_DTYPES[dtype])
    X = torch.randn(n_bcols * BLOCK, n_cols, generator=g, dtype=torch.float32).to(_TORCH_DTYPES[dtype])
    return np.ascontiguousarray(bm), blocks.contiguous(), X.contiguous()


def make_qkvdo(batch: int, heads: int, seq: int, head_dim: int, dtype: str = "f32",
               std: float = 1.0, seed: int = 0):
    """Q, K, V, dO as CPU tensors [B, H, S, D] of ``dtype`` (``"f32"``, ``"bf16"`` or ``"f16"``).

    Values are iid N(0, std^2) drawn in the order Q, K, V, dO from one seeded
    generator and rounded to ``dtype`` (round to nearest even for bf16 and f16).
    """
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(4):
        t = torch.randn(batch, heads, seq, head_dim, generator=g, dtype=torch.float32)
        if std != 1.0:
            t = t * std
        out.append(t.to(_TORCH_DTYPES[dtype]).contiguous())
    return tuple(out)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One measured workload: shape, mask recipe, operand dtype and input spread."""

    name: str
    batch: int
    heads: int
    seq: int
    head_dim: int
    mask: str
    radius: int = 1
    p: float = 0.0
    dtype: str = "bf16"
    std: float = 1.0

    @property
    def nb(self) -> int:
        return self.seq // BLOCK

    @property
    def scale(self) -> float:
        return 1.0 / float(self.head_dim) ** 0.5

    def block_mask(self) -> np.ndarray:
        return block_mask(self.mask, self.nb, radius=self.radius, p=self.p, seed=1)

    def inputs(self, seed: int = 0):
        return make_qkvdo(self.batch, self.heads, self.seq, self.head_dim, self.dtype, self.std, seed)


WORKLOADS = {
    # 4x4 block grid, band of radius 1, fp32 operands
    "tiny": Workload("tiny", 1, 1, 512, 64, "local", radius=1, dtype="f32"),
    # 16x16 grid, dilated band: |m-n| <= 4 and m-n even
    "dilated_s2048": Workload("dilated_s2048", 2, 8, 2048, 128, "dilated", radius=4, dtype="bf16"),
    # 64x64 grid, band of radius 2 plus global block row 0 and column 0 (436 stored blocks)
    "global_s8192": Workload("global_s8192", 1, 16, 8192, 128, "global", radius=2, dtype="bf16"),
    "global_s8192_f32": Workload("global_s8192_f32", 1, 16, 8192, 128, "global", radius=2, dtype="f32"),
    "global_s8192_f16": Workload("global_s8192_f16", 1, 16, 8192, 128, "global", radius=2, dtype="f16"),
    # head_dim 256 and 512 on a band of radius 3, inputs N(0, 0.5^2)
    "local_s8192_d256": Workload("local_s8192_d256", 1, 8, 8192, 256, "local", radius=3, dtype="bf16", std=0.5),
    "local_s8192_d512": Workload("local_s8192_d512", 1, 8, 8192, 512, "local", radius=3, dtype="bf16", std=0.5),
}
for _p in (0.01, 0.05, 0.13, 0.27, 0.5):
    WORKLOADS[f"random_p{_p}"] = Workload(f"random_p{_p}", 1, 16, 8192, 128, "random", p=_p, dtype="bf16")


def make_screened(n: int, n_cols: int, dtype: str = "bf16", seed: int = 0):
    """Inputs of the screened SpMM as CPU tensors: (A [n, n], diag [n] fp32, B [n, n_cols]).

    A and B are iid N(0, 1) drawn in that order from one seeded generator and
    rounded to ``dtype``; the bounds decay exponentially along the diagonal,
    diag_i = exp(-i / (n / 8)) + 1e-12, so a threshold keeps a band (the
    pages' screened-SpMM benchmark recipe).
    """
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(n, n, generator=g, dtype=torch.float32).to(_TORCH_DTYPES[dtype])
    B = torch.randn(n, n_cols, generator=g, dtype=torch.float32).to(_TORCH_DTYPES[dtype])
    pos = torch.arange(n, dtype=torch.float32)
    diag = torch.exp(-pos / (n / 8)) + 1e-12
    return A.contiguous(), diag.contiguous(), B.contiguous()
