"""Pins for the CPU fp64 oracle (no GPU).

Each test checks the oracle against something other than itself: torch's
fp64 scaled_dot_product_attention and its autograd (a separate library
routine, the dense masked reference the pages verify against), brute-force
per-element loops, central finite differences, closed forms and exact
invariants of the softmax.  A dropped term, a wrong sign, a swapped index or a
transposed operand in the oracle fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_bsr_gb300 import inputs


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _torch_sdpa(Q, K, V, elem_mask, scale):
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=torch.tensor(elem_mask), scale=scale)
    return q, k, v, o


MASKS = [("local", 1), ("dilated", 2), ("global", 1), ("full", 0), ("diag", 0)]


@pytest.mark.parametrize("kind,radius", MASKS)
def test_matches_torch_sdpa_with_element_mask(kind, radius):
    # The pages' own check: dense SDPA with the block mask repeated to elements.
    block, nb, D = 32, 6, 16
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=radius)
    Q, K, V, dO = (_rand((2, 2, S, D), s) for s in range(4))
    scale = 1.0 / math.sqrt(D)
    O, rm, rd = oracle.attn_fwd(Q, K, V, bm, scale, block)
    em = oracle.element_mask(bm, block)
    q, k, v, o = _torch_sdpa(Q, K, V, em, scale)
    np.testing.assert_allclose(O, o.detach().numpy(), atol=1e-12, rtol=0)
    o.backward(torch.tensor(dO))
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, dO, bm, scale, block)
    np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-11, rtol=0)
    # log-sum-exp of the stored scores from the statistics equals torch's logsumexp
    Sm = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    Sm = np.where(em, Sm, -np.inf)
    lse = torch.logsumexp(torch.tensor(Sm), dim=-1).numpy()
    np.testing.assert_allclose(rm + np.log(rd), lse, atol=1e-12, rtol=0)
    np.testing.assert_allclose(rm, Sm.max(axis=-1), atol=1e-12, rtol=0)


def test_full_mask_equals_unmasked_dense_attention():
    block, nb, D = 64, 4, 32
    S = block * nb
    Q, K, V = (_rand((1, 3, S, D), s) for s in (10, 11, 12))
    O, _, _ = oracle.attn_fwd(Q, K, V, np.ones((nb, nb), bool), 0.2, block)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.tensor(x) for x in (Q, K, V)), scale=0.2).numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12, rtol=0)


def _brute_force(q, k, v, bm, block, scale):
    S, D = len(q), len(q[0])
    out, rmax, rden = [], [], []
    for i in range(S):
        scores = []
        for j in range(S):
            if bm[i // block][j // block]:
                s = 0.0
                for d in range(D):
                    s += q[i][d] * k[j][d]
                scores.append((j, scale * s))
        mx = max(s for _, s in scores)
        den = sum(math.exp(s - mx) for _, s in scores)
        row = [0.0] * D
        for j, s in scores:
            w = math.exp(s - mx) / den
            for d in range(D):
                row[d] += w * v[j][d]
        out.append(row)
        rmax.append(mx)
        rden.append(den)
    return out, rmax, rden


@pytest.mark.parametrize("kind", ["local", "dilated", "global"])
def test_brute_force_4x4_blocks(kind):
    # 4 x 4 block grid, per-element loops with no matrix helper.
    block, nb, D = 8, 4, 5
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=1)
    Q, K, V = (_rand((1, 1, S, D), s) for s in (20, 21, 22))
    scale = 0.37
    O, rm, rd = oracle.attn_fwd(Q, K, V, bm, scale, block)
    bo, bmx, bden = _brute_force(Q[0, 0].tolist(), K[0, 0].tolist(), V[0, 0].tolist(), bm.tolist(), block, scale)
    np.testing.assert_allclose(O[0, 0], np.array(bo), atol=1e-12, rtol=0)
    np.testing.assert_allclose(rm[0, 0], np.array(bmx), atol=1e-12, rtol=0)
    np.testing.assert_allclose(rd[0, 0], np.array(bden), rtol=1e-12, atol=0)


def test_brute_force_rows_at_block_128():
    # The real block size on a 4 x 4 grid (S = 512), a few rows by loops.
    block, nb, D = 128, 4, 8
    S = block * nb
    bm = inputs.block_mask("local", nb, radius=1)
    Q, K, V = (_rand((1, 1, S, D), s) for s in (30, 31, 32))
    O, rm, rd = oracle.attn_fwd(Q, K, V, bm, 0.125, block)
    q, k, v = Q[0, 0].tolist(), K[0, 0].tolist(), V[0, 0].tolist()
    for i in (0, 127, 128, 300, 511):
        scores = [(j, 0.125 * sum(q[i][d] * k[j][d] for d in range(D)))
                  for j in range(S) if bm[i // block, j // block]]
        mx = max(s for _, s in scores)
        den = sum(math.exp(s - mx) for _, s in scores)
        row = [sum(math.exp(s - mx) / den * v[j][d] for j, s in scores) for d in range(D)]
        np.testing.assert_allclose(O[0, 0, i], row, atol=1e-12)
        assert abs(rm[0, 0, i] - mx) < 1e-12 and abs(rd[0, 0, i] / den - 1) < 1e-12


@pytest.mark.parametrize("kind", ["local", "dilated", "global"])
def test_softmax_weights_sum_to_one(kind):
    block, nb, D = 16, 8, 8
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=2)
    Q, K, V = (_rand((2, 1, S, D), s, 2.0) for s in (40, 41, 42))
    scale = 0.5
    _, rm, rd = oracle.attn_fwd(Q, K, V, bm, scale, block)
    em = oracle.element_mask(bm, block)
    for b in range(2):
        s = scale * Q[b, 0] @ K[b, 0].T
        w = np.where(em, np.exp(s - rm[b, 0][:, None]), 0.0) / rd[b, 0][:, None]
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(w[~em] == 0)


def _loss(Q, K, V, dO, bm, scale, block):
    O, _, _ = oracle.attn_fwd(Q, K, V, bm, scale, block)
    return float((O * dO).sum())


@pytest.mark.parametrize("kind", ["local", "dilated", "global"])
def test_gradients_match_central_differences(kind):
    block, nb, D = 4, 4, 3
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=1)
    Q, K, V, dO = (_rand((1, 1, S, D), s) for s in (50, 51, 52, 53))
    scale = 0.7
    grads = oracle.attn_bwd(Q, K, V, dO, bm, scale, block)
    h = 1e-6
    for which, g in enumerate(grads):
        args = [Q, K, V]
        for idx in np.ndindex(*Q.shape):
            xp = [a.copy() for a in args]
            xm = [a.copy() for a in args]
            xp[which][idx] += h
            xm[which][idx] -= h
            fd = (_loss(*xp, dO, bm, scale, block) - _loss(*xm, dO, bm, scale, block)) / (2 * h)
            assert abs(fd - g[idx]) < 1e-7, (which, idx, fd, g[idx])


@pytest.mark.parametrize("kind", ["local", "dilated"])
def test_gradcheck_seq256_head_dim32_sampled(kind):
    # The pages' gradcheck workload: fp64, seq 256, head_dim 32 (sampled entries).
    block, nb, D = 64, 4, 32
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=2)
    Q, K, V, dO = (_rand((1, 1, S, D), s) for s in (60, 61, 62, 63))
    scale = 1 / math.sqrt(D)
    grads = oracle.attn_bwd(Q, K, V, dO, bm, scale, block)
    rng = np.random.default_rng(7)
    h = 1e-5
    for which, g in enumerate(grads):
        for _ in range(12):
            idx = (0, 0, int(rng.integers(S)), int(rng.integers(D)))
            xp = [a.copy() for a in (Q, K, V)]
            xm = [a.copy() for a in (Q, K, V)]
            xp[which][idx] += h
            xm[which][idx] -= h
            fd = (_loss(*xp, dO, bm, scale, block) - _loss(*xm, dO, bm, scale, block)) / (2 * h)
            assert abs(fd - g[idx]) < 1e-6, (which, idx, fd, g[idx])


def test_closed_form_zero_queries():
    # Q = 0: scores all 0 -> uniform weights over stored keys; row_max 0, row_denom = #keys.
    block, nb, D = 8, 5, 4
    S = block * nb
    bm = inputs.block_mask("global", nb, radius=1)
    K, V = _rand((1, 1, S, D), 70), _rand((1, 1, S, D), 71)
    O, rm, rd = oracle.attn_fwd(np.zeros_like(K), K, V, bm, 0.3, block)
    for i in range(S):
        cols = [j for j in range(S) if bm[i // block, j // block]]
        np.testing.assert_allclose(O[0, 0, i], V[0, 0, cols].mean(axis=0), atol=1e-13)
        assert rm[0, 0, i] == 0.0
        assert rd[0, 0, i] == len(cols)


def test_closed_form_constant_values():
    block, nb, D = 8, 4, 6
    S = block * nb
    bm = inputs.block_mask("dilated", nb, radius=2)
    Q, K = _rand((1, 2, S, D), 72), _rand((1, 2, S, D), 73)
    c = _rand((D,), 74)
    V = np.broadcast_to(c, (1, 2, S, D)).copy()
    O, _, _ = oracle.attn_fwd(Q, K, V, bm, 0.9, block)
    np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), atol=1e-13)


def test_diagonal_mask_is_per_block_dense_attention():
    block, nb, D = 16, 4, 8
    S = block * nb
    Q, K, V = (_rand((1, 1, S, D), s) for s in (80, 81, 82))
    O, _, _ = oracle.attn_fwd(Q, K, V, np.eye(nb, dtype=bool), 0.25, block)
    for m in range(nb):
        sl = slice(m * block, (m + 1) * block)
        ref = torch.nn.functional.scaled_dot_product_attention(
            *(torch.tensor(x[0, 0, sl]) for x in (Q, K, V)), scale=0.25).numpy()
        np.testing.assert_allclose(O[0, 0, sl], ref, atol=1e-12)


@pytest.mark.parametrize("kind", ["local", "dilated", "global"])
def test_gradient_invariants(kind):
    block, nb, D = 16, 6, 8
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=2)
    Q, K, V, dO = (_rand((1, 2, S, D), s) for s in (90, 91, 92, 93))
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, dO, bm, 0.4, block)
    # sum_j dS_ij = 0 per row, hence the key gradients sum to zero
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
    # rows of P sum to one, hence sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dV.sum(axis=2), dO.sum(axis=2), atol=1e-12)
    # keys all equal: scores constant along each row, so dQ = 0
    Kc = np.broadcast_to(K[:, :, :1], K.shape).copy()
    dQc, _, _ = oracle.attn_bwd(Q, Kc, V, dO, bm, 0.4, block)
    np.testing.assert_allclose(dQc, 0.0, atol=1e-12)


@pytest.mark.parametrize("kind", ["local", "dilated", "global", "random"])
def test_block_walk_equals_dense_backward(kind):
    block, nb, D = 16, 7, 8
    S = block * nb
    bm = inputs.block_mask(kind, nb, radius=2, p=0.3)
    row_ptr, col_idx = inputs.bsr_from_block_mask(bm)
    Q, K, V, dO = (_rand((1, 2, S, D), s) for s in (100, 101, 102, 103))
    ref = oracle.attn_bwd(Q, K, V, dO, bm, 0.3, block)
    got = oracle.attn_bwd_blockwalk(Q, K, V, dO, row_ptr, col_idx, 0.3, block)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, atol=1e-12)


def test_empty_block_row_reading():
    # A block row with no stored block: O = 0, row_max = -inf, row_denom = 0,
    # dQ = 0 there, and the other rows' results equal those with that row removed.
    block, nb, D = 8, 4, 4
    S = block * nb
    bm = inputs.block_mask("local", nb, radius=1)
    bm[2, :] = False
    Q, K, V, dO = (_rand((1, 1, S, D), s) for s in (110, 111, 112, 113))
    O, rm, rd = oracle.attn_fwd(Q, K, V, bm, 0.5, block)
    sl = slice(2 * block, 3 * block)
    assert np.all(O[0, 0, sl] == 0) and np.all(rm[0, 0, sl] == -np.inf) and np.all(rd[0, 0, sl] == 0)
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, dO, bm, 0.5, block)
    assert np.all(dQ[0, 0, sl] == 0)
    dO2 = dO.copy()
    dO2[0, 0, sl] = 0.0  # the empty rows' upstream gradient has no path to K, V
    _, dK2, dV2 = oracle.attn_bwd(Q, K, V, dO2, bm, 0.5, block)
    np.testing.assert_allclose(dK, dK2, atol=1e-14)
    np.testing.assert_allclose(dV, dV2, atol=1e-14)
    keep = np.r_[0:2 * block, 3 * block:S]
    em = oracle.element_mask(bm, block)[np.ix_(keep, np.arange(S))]
    q, k, v, o = _torch_sdpa(Q[:, :, keep], K, V, em, 0.5)
    np.testing.assert_allclose(O[:, :, keep], o.detach().numpy(), atol=1e-12)


def test_bsc_view_of_block_mask():
    bm = inputs.block_mask("random", 9, p=0.35)
    col_ptr, row_idx = oracle.bsc_from_block_mask(bm)
    assert col_ptr[-1] == bm.sum()
    for n in range(9):
        rows = row_idx[col_ptr[n]:col_ptr[n + 1]]
        assert list(rows) == [m for m in range(9) if bm[m, n]]
