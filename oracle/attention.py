"""CPU fp64 oracle for block-sparse attention over a BSR block mask.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.  The
library never calls it, and it never calls the library: it shares no code,
table or helper with the CUDA path.  Inputs come in as numpy arrays (already
rounded to the operand precision by the caller) and everything is computed in
float64 with plain numpy, a matrix product being the only library step.

What it computes (the plain definition; the method reaches the same result up
to rounding order):

* Block-sparse attention is dense softmax attention in which every score
  outside a stored block is removed: the pages verify the kernels against
  dense scaled-dot-product attention with the element mask built by repeating
  the block mask 128 x 128 ("trnsparse 0.7.0 -> 0.9.0" diff,
  ``benchmarks/bench_native_trn2.py``, ``section_attn``; "trnsparse 0.4.1 ->
  0.6.0" diff, CHANGELOG [0.4.2], tests/test_attention.py parity against a
  dense reference).
* Forward statistics: ``row_max`` is the maximum of the scaled scores of the
  row and ``row_denom`` the sum of ``exp(s - row_max)`` over its stored
  scores, both returned in fp32 by the kernels ("trnsparse 0.4.1 -> 0.6.0"
  diff, CHANGELOG [0.5.1], "Stats saving in forward" and ``return_stats``;
  "trnsparse 0.7.0 -> 0.9.0" diff, CHANGELOG [0.9.0], fp32 statistics for
  bf16 Q).  Natural-log units are the reading taken here.
* Backward: the analytic gradient of the softmax attention with the Flash
  Attention delta identity D_i = dO_i . O_i ("trnsparse 0.4.1 -> 0.6.0"
  diff, CHANGELOG [0.5.0]); the block walks of CHANGELOG [0.5.1]
  (``dQ_m += dS @ K_ki * scale`` row-first, ``dK_ki += dS.T @ Q_m * scale``
  and ``dV_ki += P.T @ dO_m`` column-first over a BSC view) are written out
  in ``attn_bwd_blockwalk``.

Readings where the pages are silent: a block row with no stored block yields
O = 0, row_max = -inf, row_denom = 0, and contributes nothing to any gradient.

Every function here is pinned by ``tests/test_oracle.py`` against something
other than itself (torch's fp64 scaled_dot_product_attention and its autograd,
brute-force loops, central finite differences, closed forms and exact
invariants).  No function is parity-unpinned.
"""

from __future__ import annotations

import numpy as np


def element_mask(block_mask: np.ndarray, block: int) -> np.ndarray:
    """Element mask [S, S]: M[i, j] is True iff block (i // block, j // block) is stored."""
    bm = np.asarray(block_mask, dtype=bool)
    return np.repeat(np.repeat(bm, block, axis=0), block, axis=1)


def block_mask_from_bsr(row_ptr, col_idx, n_bcols: int) -> np.ndarray:
    """Boolean block mask from BSR lists (block-row pointers, block-column indices)."""
    row_ptr = np.asarray(row_ptr)
    col_idx = np.asarray(col_idx)
    nb = len(row_ptr) - 1
    bm = np.zeros((nb, n_bcols), dtype=bool)
    for m in range(nb):
        for j in range(int(row_ptr[m]), int(row_ptr[m + 1])):
            bm[m, int(col_idx[j])] = True
    return bm


def bsc_from_block_mask(block_mask: np.ndarray):
    """Column-first (BSC) view of a block mask: (col_ptr [nbc+1], row_idx [nnzb]), rows ascending.

    The column-first traversal of the dK/dV walk ("trnsparse 0.4.1 -> 0.6.0"
    diff, CHANGELOG [0.5.1], ``_attn_bwd_dkdv_kernel``: "BSC view built on
    host").
    """
    bm = np.asarray(block_mask, dtype=bool)
    nbr, nbc = bm.shape
    col_ptr = [0]
    row_idx = []
    for n in range(nbc):
        for m in range(nbr):
            if bm[m, n]:
                row_idx.append(m)
        col_ptr.append(len(row_idx))
    return np.array(col_ptr, dtype=np.int64), np.array(row_idx, dtype=np.int64)


def _softmax_rows(S: np.ndarray):
    """Row max, row denominator and probabilities of a score matrix with -inf for removed entries."""
    m = S.max(axis=1)
    nonempty = np.isfinite(m)
    shift = np.where(nonempty, m, 0.0)
    E = np.exp(S - shift[:, None])  # exp(-inf) = 0 outside the stored blocks
    l = E.sum(axis=1)
    P = np.zeros_like(S)
    P[nonempty] = E[nonempty] / l[nonempty, None]
    return m, l, P


def _head_probs(q, k, block_mask, scale, block):
    S = scale * (q @ k.T)
    S = np.where(element_mask(block_mask, block), S, -np.inf)
    return _softmax_rows(S)


def attn_fwd(Q, K, V, block_mask, scale: float, block: int = 128):
    """Forward block-sparse attention in fp64.

    Q, K, V: [B, H, S, D] (any float dtype; upcast to float64).  block_mask:
    boolean [S/block, S/block], shared by every (batch, head).
    Returns O [B, H, S, D], row_max [B, H, S], row_denom [B, H, S] (float64).
    """
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    B, H, S, D = Q.shape
    O = np.zeros((B, H, S, D))
    row_max = np.empty((B, H, S))
    row_denom = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            m, l, P = _head_probs(Q[b, h], K[b, h], block_mask, scale, block)
            O[b, h] = P @ V[b, h]
            row_max[b, h] = m
            row_denom[b, h] = l
    return O, row_max, row_denom


def attn_bwd(Q, K, V, dO, block_mask, scale: float, block: int = 128):
    """Analytic backward of ``attn_fwd`` in fp64: (dQ, dK, dV), each [B, H, S, D].

    With P the row softmax over stored scores and O = P V:
      dV = P^T dO;  dP = dO V^T;  D_i = sum_d dO_id O_id;
      dS = P * (dP - D);  dQ = scale dS K;  dK = scale dS^T Q.
    """
    Q, K, V, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, dO))
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    B, H = Q.shape[:2]
    for b in range(B):
        for h in range(H):
            q, k, v, do = Q[b, h], K[b, h], V[b, h], dO[b, h]
            _, _, P = _head_probs(q, k, block_mask, scale, block)
            o = P @ v
            dV[b, h] = P.T @ do
            dP = do @ v.T
            delta = (do * o).sum(axis=1)
            dS = P * (dP - delta[:, None])
            dQ[b, h] = scale * (dS @ k)
            dK[b, h] = scale * (dS.T @ q)
    return dQ, dK, dV


def attn_bwd_blockwalk(Q, K, V, dO, row_ptr, col_idx, scale: float, block: int = 128):
    """The same backward, walking only stored blocks as the kernels do.

    dQ is accumulated block-row by block-row over the BSR lists; dK and dV
    column by column over the BSC view that this function builds from the BSR
    lists itself.  Statistics come from the forward definition, and P for a
    block (m, n) is exp(scale q k^T - row_max) / row_denom on that block only.
    """
    Q, K, V, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, dO))
    B, H, S, D = Q.shape
    nb = S // block
    bm = block_mask_from_bsr(row_ptr, col_idx, nb)
    col_ptr, row_idx = bsc_from_block_mask(bm)
    O, row_max, row_denom = attn_fwd(Q, K, V, bm, scale, block)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)

    def blk(x, i):
        return x[i * block:(i + 1) * block]

    for b in range(B):
        for h in range(H):
            q, k, v, do, o = Q[b, h], K[b, h], V[b, h], dO[b, h], O[b, h]
            delta = (do * o).sum(axis=1)

            def probs(m, n):
                s = scale * (blk(q, m) @ blk(k, n).T)
                return np.exp(s - blk(row_max[b, h], m)[:, None]) / blk(row_denom[b, h], m)[:, None]

            def dscore(m, n, p):
                dp = blk(do, m) @ blk(v, n).T
                return p * (dp - blk(delta, m)[:, None])

            for m in range(nb):  # row-first: dQ
                acc = np.zeros((block, D))
                for j in range(int(row_ptr[m]), int(row_ptr[m + 1])):
                    n = int(col_idx[j])
                    ds = dscore(m, n, probs(m, n))
                    acc += scale * (ds @ blk(k, n))
                dQ[b, h, m * block:(m + 1) * block] = acc
            for n in range(nb):  # column-first: dK, dV
                acc_k = np.zeros((block, D))
                acc_v = np.zeros((block, D))
                for t in range(int(col_ptr[n]), int(col_ptr[n + 1])):
                    m = int(row_idx[t])
                    p = probs(m, n)
                    ds = dscore(m, n, p)
                    acc_v += p.T @ blk(do, m)
                    acc_k += scale * (ds.T @ blk(q, m))
                dK[b, h, n * block:(n + 1) * block] = acc_k
                dV[b, h, n * block:(n + 1) * block] = acc_v
    return dQ, dK, dV


def attn_fwd_bwd_head(q, k, v, do, block_mask, scale: float, block: int = 128):
    """Forward and backward of one (batch, head) slice [S, D]: (o, row_max, row_denom, dq, dk, dv)."""
    args = [np.asarray(t, dtype=np.float64)[None, None] for t in (q, k, v, do)]
    o, rm, rd = attn_fwd(args[0], args[1], args[2], block_mask, scale, block)
    dq, dk, dv = attn_bwd(*args, block_mask, scale, block)
    return o[0, 0], rm[0, 0], rd[0, 0], dq[0, 0], dk[0, 0], dv[0, 0]
