"""CPU fp64 oracle for block-sparse times dense (BSR SpMM).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` may import this module; the library never calls it and it never
calls the library.  Inputs are numpy arrays already rounded to the operand
precision by the caller; everything is computed in float64 with plain numpy,
a matrix product being the only library step.

What it computes (the plain definition; "trnsparse 0.7.0 -> 0.9.0" diff,
CHANGELOG [0.8.0]: bsr_spmm_static multiplies the BSR matrix by a dense one,
walking only the stored blocks and addressing the dense operand by block
column): for a BSR matrix A of 128 x 128 blocks (``row_ptr``, ``col_idx`` and
the stored blocks in that order) and a dense X,

    Y[m*128 + i, c] = sum over stored j of block row m, k = col_idx[j],
                      sum_t blocks[j][i][t] * X[k*128 + t, c],

i.e. Y = A_dense X with A_dense zero outside the stored blocks.  A block row
with no stored block gives zero rows of Y.

Pinned by ``tests/test_oracle_spmm.py`` against element sums written out from
the formula above, identity blocks (Y = X), empty rows and linearity.
"""

from __future__ import annotations

import numpy as np

B = 128


def bsr_to_dense(blocks: np.ndarray, row_ptr: np.ndarray, col_idx: np.ndarray, n_brows: int,
                 n_bcols: int) -> np.ndarray:
    """The dense matrix of a BSR matrix (float64): stored blocks placed, zeros elsewhere."""
    A = np.zeros((n_brows * B, n_bcols * B), dtype=np.float64)
    for m in range(n_brows):
        for j in range(int(row_ptr[m]), int(row_ptr[m + 1])):
            k = int(col_idx[j])
            A[m * B:(m + 1) * B, k * B:(k + 1) * B] = blocks[j]
    return A


def spmm(blocks: np.ndarray, row_ptr: np.ndarray, col_idx: np.ndarray, n_brows: int, n_bcols: int,
         X: np.ndarray) -> np.ndarray:
    """Y = A X in float64."""
    return bsr_to_dense(blocks, row_ptr, col_idx, n_brows, n_bcols) @ np.asarray(X, dtype=np.float64)
