"""CPU fp64 oracle for the fused screened SpMM.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` may import this module; the library never calls it and it never
calls the library.  Inputs are numpy arrays (A and B already rounded to the
operand precision by the caller).

What it computes (the plain definition; "trnsparse 0.7.0 -> 0.9.0" diff,
docs: screened_spmm(A, diag, B, threshold) fuses the Schwarz pair bound,
the threshold mask and the matmul; mask semantics
``mask[i, j] = sqrt(|diag[i]|) * sqrt(|diag[j]|) > sqrt(threshold)``):

    C = (A o M) B,   M[i, j] = (q_i q_j > t),  q = sqrt(|diag|),  t = sqrt(threshold).

The mask is an integer decision made by floating point, so it is taken in
the kernel's precision (fp32: square roots, product and comparison), and the
masked product is then formed in float64 with a matrix product as the only
library step.

Pinned by ``tests/test_oracle_screened.py`` against per-element sums and
per-pair mask decisions written out from the formula, and the threshold-0
(plain product) and large-threshold (zero) special cases.
"""

from __future__ import annotations

import numpy as np


def schwarz_mask(diag: np.ndarray, threshold: float) -> np.ndarray:
    """Boolean [n, n] mask in fp32: sqrt|diag_i| * sqrt|diag_j| > sqrt(threshold)."""
    q = np.sqrt(np.abs(np.asarray(diag, dtype=np.float32)))
    t = np.sqrt(np.float32(threshold))
    return (q[:, None] * q[None, :]) > t


def screened_spmm(A: np.ndarray, diag: np.ndarray, B: np.ndarray, threshold: float) -> np.ndarray:
    """C = (A o M) B in float64."""
    M = schwarz_mask(diag, threshold)
    return (np.asarray(A, dtype=np.float64) * M) @ np.asarray(B, dtype=np.float64)
