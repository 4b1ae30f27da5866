"""Pins of the BSR SpMM oracle (oracle/spmm.py) against things other than itself."""

import numpy as np
import pytest

import oracle
from block_sparse_attention_bsr_gb300 import inputs

B = 128


def _case(n_brows, n_bcols, n_cols, p, seed):
    bm, blocks, X = inputs.make_spmm(n_brows, n_bcols, n_cols, p, "bf16", seed)
    rp, ci = inputs.bsr_from_block_mask(bm)
    return bm, rp, ci, blocks.double().numpy(), X.double().numpy()


@pytest.mark.parametrize("seed", [0, 1])
def test_elements_match_the_defining_sum(seed):
    # Y[m*128 + i, c] written out term by term over the row's stored blocks,
    # for sampled (row, column) entries -- no dense matrix involved
    bm, rp, ci, blocks, X = _case(3, 4, 64, 0.5, seed)
    Y = oracle.spmm(blocks, rp, ci, 3, 4, X)
    rng = np.random.default_rng(seed)
    for _ in range(40):
        row, c = int(rng.integers(3 * B)), int(rng.integers(64))
        m, i = divmod(row, B)
        want = 0.0
        for j in range(rp[m], rp[m + 1]):
            k = ci[j]
            for t in range(B):
                want += blocks[j][i][t] * X[k * B + t, c]
        assert abs(Y[row, c] - want) <= 1e-12 * max(1.0, abs(want))


def test_identity_blocks_give_x():
    n = 3
    blocks = np.stack([np.eye(B) for _ in range(n)])
    rp = np.arange(n + 1, dtype=np.int32)
    ci = np.arange(n, dtype=np.int32)
    X = np.random.default_rng(5).standard_normal((n * B, 192))
    assert np.array_equal(oracle.spmm(blocks, rp, ci, n, n, X), X)


def test_empty_block_row_is_zero():
    bm = np.array([[True, False], [False, False], [True, True]])
    rp, ci = inputs.bsr_from_block_mask(bm)
    blocks = np.random.default_rng(1).standard_normal((3, B, B))
    X = np.random.default_rng(2).standard_normal((2 * B, 64))
    Y = oracle.spmm(blocks, rp, ci, 3, 2, X)
    assert np.all(Y[B:2 * B] == 0)
    assert np.abs(Y[:B]).max() > 0 and np.abs(Y[2 * B:]).max() > 0


def test_linear_in_the_blocks():
    bm, rp, ci, b1, X = _case(2, 3, 64, 0.7, 3)
    b2 = np.random.default_rng(4).standard_normal(b1.shape)
    y1 = oracle.spmm(b1, rp, ci, 2, 3, X)
    y2 = oracle.spmm(b2, rp, ci, 2, 3, X)
    y12 = oracle.spmm(b1 + 2.0 * b2, rp, ci, 2, 3, X)
    assert np.allclose(y12, y1 + 2.0 * y2, rtol=0, atol=1e-10)


def test_block_placement_follows_col_idx():
    # one stored block in row 1 at column 2: only X's rows 256..383 matter
    bm = np.zeros((2, 3), bool)
    bm[1, 2] = True
    rp, ci = inputs.bsr_from_block_mask(bm)
    blk = np.random.default_rng(6).standard_normal((1, B, B))
    X = np.zeros((3 * B, 64))
    X[2 * B:] = np.random.default_rng(7).standard_normal((B, 64))
    Y = oracle.spmm(blk, rp, ci, 2, 3, X)
    assert np.all(Y[:B] == 0)
    assert np.allclose(Y[B:], blk[0] @ X[2 * B:], rtol=0, atol=1e-12)
    X[2 * B:] = 0
    assert np.all(oracle.spmm(blk, rp, ci, 2, 3, X) == 0)
