"""The oracle's pins catch plausible mistakes in the oracle (no GPU).

Each case plants one mistake in a copy of ``oracle/attention.py`` (and, at
the end, of ``oracle/spmm.py`` and ``oracle/screened.py``) -- a
dropped term, a wrong sign, a swapped axis or index, a transposed operand, a
mask left out -- loads the copy as a module of its own, and runs the pins
below on it: torch's fp64 scaled_dot_product_attention and its autograd with
the element mask, brute-force per-element loops, central finite
differences, the empty-row reading and a brute-force column listing.  Every
mutant must fail at least one of them, and the unmodified source must pass
all of them.  The mistakes are planted in the oracle, on the CPU; the library
is not involved.
"""

import math
import os
import types

import numpy as np
import pytest
import torch

from block_sparse_attention_bsr_gb300 import inputs

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
SRC = open(os.path.join(ORACLE_DIR, "attention.py")).read()


def _load(src: str) -> types.ModuleType:
    mod = types.ModuleType("oracle_attention_variant")
    exec(compile(src, "oracle_attention_variant", "exec"), mod.__dict__)
    return mod


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def pin_torch_sdpa(mod):
    block, nb, D = 8, 4, 5
    S = block * nb
    bm = inputs.block_mask("global", nb, radius=1)
    bm[2, 0] = False  # a row whose stored columns are not symmetric
    Q, K, V, dO = (_rand((1, 2, S, D), s) for s in range(4))
    scale = 1.0 / math.sqrt(D)
    O, rm, rd = mod.attn_fwd(Q, K, V, bm, scale, block)
    em = np.repeat(np.repeat(bm, block, 0), block, 1)
    q, k, v = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=torch.tensor(em), scale=scale)
    o.backward(torch.tensor(dO))
    np.testing.assert_allclose(O, o.detach().numpy(), atol=1e-12, rtol=0)
    sm = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    sm = np.where(em, sm, -np.inf)
    np.testing.assert_allclose(rm, sm.max(axis=-1), atol=1e-12, rtol=0)
    np.testing.assert_allclose(rm + np.log(rd), torch.logsumexp(torch.tensor(sm), -1).numpy(), atol=1e-12, rtol=0)
    for got, ref in zip(mod.attn_bwd(Q, K, V, dO, bm, scale, block), (q.grad, k.grad, v.grad)):
        np.testing.assert_allclose(got, ref.numpy(), atol=1e-11, rtol=0)
    rp = np.concatenate([[0], np.cumsum(bm.sum(1))])
    ci = np.nonzero(bm)[1]
    for got, ref in zip(mod.attn_bwd_blockwalk(Q, K, V, dO, rp, ci, scale, block), (q.grad, k.grad, v.grad)):
        np.testing.assert_allclose(got, ref.numpy(), atol=1e-11, rtol=0)


def pin_brute_force(mod):
    block, nb, D = 2, 4, 3
    S = block * nb
    bm = inputs.block_mask("dilated", nb, radius=2)
    Q, K, V = (_rand((1, 1, S, D), s) for s in (10, 11, 12))
    scale = 0.9
    O, rm, rd = mod.attn_fwd(Q, K, V, bm, scale, block)
    for i in range(S):
        cols = [j for j in range(S) if bm[i // block, j // block]]
        s = [scale * sum(Q[0, 0, i, d] * K[0, 0, j, d] for d in range(D)) for j in cols]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        den = sum(w)
        assert abs(rm[0, 0, i] - mx) < 1e-12 and abs(rd[0, 0, i] - den) < 1e-12
        for d in range(D):
            ref = sum(wj * V[0, 0, j, d] for wj, j in zip(w, cols)) / den
            assert abs(O[0, 0, i, d] - ref) < 1e-12


def pin_central_differences(mod):
    block, nb, D = 2, 3, 2
    S = block * nb
    bm = inputs.block_mask("local", nb, radius=1)
    bm[0, 1] = False
    Q, K, V, dO = (_rand((1, 1, S, D), s) for s in (20, 21, 22, 23))
    scale = 0.8
    grads = mod.attn_bwd(Q, K, V, dO, bm, scale, block)
    h = 1e-6

    def loss(q, k, v):
        return float((mod.attn_fwd(q, k, v, bm, scale, block)[0] * dO).sum())

    for which, g in enumerate(grads):
        for idx in np.ndindex(*Q.shape):
            xp = [Q.copy(), K.copy(), V.copy()]
            xm = [Q.copy(), K.copy(), V.copy()]
            xp[which][idx] += h
            xm[which][idx] -= h
            fd = (loss(*xp) - loss(*xm)) / (2 * h)
            assert abs(fd - g[idx]) < 1e-7


def pin_empty_row(mod):
    block, nb, D = 2, 3, 2
    bm = np.zeros((nb, nb), bool)
    bm[0, 0] = bm[2, 1] = True  # block row 1 and block column 2 store nothing
    Q, K, V, dO = (_rand((1, 1, block * nb, D), s) for s in (30, 31, 32, 33))
    O, rm, rd = mod.attn_fwd(Q, K, V, bm, 0.5, block)
    assert np.all(O[0, 0, 2:4] == 0) and np.all(np.isneginf(rm[0, 0, 2:4])) and np.all(rd[0, 0, 2:4] == 0)
    dQ, dK, dV = mod.attn_bwd(Q, K, V, dO, bm, 0.5, block)
    assert np.all(dQ[0, 0, 2:4] == 0) and np.all(dK[0, 0, 4:6] == 0) and np.all(dV[0, 0, 4:6] == 0)


def pin_bsc(mod):
    bm = np.random.default_rng(40).random((5, 7)) < 0.4
    col_ptr, row_idx = mod.bsc_from_block_mask(bm)
    for n in range(7):
        assert list(row_idx[col_ptr[n]:col_ptr[n + 1]]) == [m for m in range(5) if bm[m, n]]
    rp = np.concatenate([[0], np.cumsum(bm.sum(1))])
    assert np.array_equal(mod.block_mask_from_bsr(rp, np.nonzero(bm)[1], 7), bm)


PINS = [pin_torch_sdpa, pin_brute_force, pin_central_differences, pin_empty_row, pin_bsc]


def _failing_pins(mod):
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # an assertion, or a mutant that no longer runs
            failed.append(pin.__name__)
    return failed


# (what the mistake is, the text it replaces, the replacement)
MUTANTS = [
    ("scale dropped from the scores", "S = scale * (q @ k.T)", "S = (q @ k.T)"),
    ("scores transposed", "S = scale * (q @ k.T)", "S = scale * (k @ q.T)"),
    ("mask not applied", "S = np.where(element_mask(block_mask, block), S, -np.inf)", "S = S"),
    ("mask transposed", "S = np.where(element_mask(block_mask, block), S, -np.inf)",
     "S = np.where(element_mask(block_mask.T, block), S, -np.inf)"),
    ("row sum over the wrong axis", "l = E.sum(axis=1)", "l = E.sum(axis=0)"),
    ("max shift left out of the sum", "E = np.exp(S - shift[:, None])", "E = np.exp(S)"),
    ("output from P transposed", "O[b, h] = P @ V[b, h]", "O[b, h] = P.T @ V[b, h]"),
    ("row_denom of another row", "row_denom[b, h] = l", "row_denom[b, h] = np.roll(l, 1)"),
    ("dV without the transpose", "dV[b, h] = P.T @ do", "dV[b, h] = P @ do"),
    ("dP from transposed operands", "dP = do @ v.T", "dP = v @ do.T"),
    ("delta with the wrong sign", "dS = P * (dP - delta[:, None])", "dS = P * (dP + delta[:, None])"),
    ("delta term dropped", "dS = P * (dP - delta[:, None])", "dS = P * dP"),
    ("delta over the wrong axis", "delta = (do * o).sum(axis=1)\n            dS",
     "delta = (do * o).sum(axis=0)\n            dS"),
    ("dQ without the scale", "dQ[b, h] = scale * (dS @ k)", "dQ[b, h] = dS @ k"),
    ("dK without the transpose", "dK[b, h] = scale * (dS.T @ q)", "dK[b, h] = scale * (dS @ q)"),
    ("block walk: probabilities without row_denom",
     "return np.exp(s - blk(row_max[b, h], m)[:, None]) / blk(row_denom[b, h], m)[:, None]",
     "return np.exp(s - blk(row_max[b, h], m)[:, None])"),
    ("block walk: dK block from the wrong query block", "acc_k += scale * (ds.T @ blk(q, m))",
     "acc_k += scale * (ds.T @ blk(q, n))"),
    ("block walk: dV from dS", "acc_v += p.T @ blk(do, m)", "acc_v += ds.T @ blk(do, m)"),
    ("block walk: dQ over the wrong key block", "acc += scale * (ds @ blk(k, n))", "acc += scale * (ds @ blk(k, m))"),
    ("BSC view: rows in descending order", "for m in range(nbr):", "for m in reversed(range(nbr)):"),
    ("BSR decode: columns off by one", "bm[m, int(col_idx[j])] = True", "bm[m, (int(col_idx[j]) + 1) % n_bcols] = True"),
]


def test_unmodified_oracle_passes_every_pin():
    assert _failing_pins(_load(SRC)) == []


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # some mutants divide by zero
@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_each_planted_mistake_fails_a_pin(what, old, new):
    assert SRC.count(old) == 1, f"the mutation site for '{what}' must occur exactly once"
    failed = _failing_pins(_load(SRC.replace(old, new)))
    assert failed, f"no pin caught: {what}"


# ---------------------------------------------------------------- SpMM --
SPMM_SRC = open(os.path.join(ORACLE_DIR, "spmm.py")).read()
BLK = 128


def pin_spmm_defining_sum(mod):
    bm = np.array([[True, False, True], [False, True, True]])
    rp = np.concatenate([[0], np.cumsum(bm.sum(1))])
    ci = np.nonzero(bm)[1]
    rng = np.random.default_rng(50)
    blocks = rng.standard_normal((len(ci), BLK, BLK))
    X = rng.standard_normal((3 * BLK, 8))
    Y = mod.spmm(blocks, rp, ci, 2, 3, X)
    for row, c in ((5, 1), (130, 7), (255, 0), (77, 4)):
        m, i = divmod(row, BLK)
        want = sum(blocks[j][i][t] * X[ci[j] * BLK + t, c] for j in range(rp[m], rp[m + 1]) for t in range(BLK))
        assert abs(Y[row, c] - want) <= 1e-10 * max(1.0, abs(want))


def pin_spmm_placement(mod):
    bm = np.zeros((2, 3), bool)
    bm[1, 2] = True
    blk = np.random.default_rng(51).standard_normal((1, BLK, BLK))
    X = np.random.default_rng(52).standard_normal((3 * BLK, 4))
    Y = mod.spmm(blk, np.array([0, 0, 1]), np.array([2]), 2, 3, X)
    assert np.all(Y[:BLK] == 0)
    assert np.allclose(Y[BLK:], blk[0] @ X[2 * BLK:], rtol=0, atol=1e-12)


SPMM_MUTANTS = [
    ("block placed at (column, row)", "A[m * B:(m + 1) * B, k * B:(k + 1) * B] = blocks[j]",
     "A[k * B:(k + 1) * B, m * B:(m + 1) * B] = blocks[j]"),
    ("block stored transposed", "A[m * B:(m + 1) * B, k * B:(k + 1) * B] = blocks[j]",
     "A[m * B:(m + 1) * B, k * B:(k + 1) * B] = blocks[j].T"),
    ("blocks taken from the wrong list entry", "] = blocks[j]", "] = blocks[j - 1]"),
    ("X transposed in the product", "@ np.asarray(X, dtype=np.float64)", "@ np.asarray(X, dtype=np.float64)[::-1]"),
]


def _spmm_failing(src):
    mod = types.ModuleType("oracle_spmm_variant")
    exec(compile(src, "oracle_spmm_variant", "exec"), mod.__dict__)
    failed = []
    for pin in (pin_spmm_defining_sum, pin_spmm_placement):
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_unmodified_spmm_oracle_passes_its_pins():
    assert _spmm_failing(SPMM_SRC) == []


@pytest.mark.parametrize("what,old,new", SPMM_MUTANTS, ids=[m[0] for m in SPMM_MUTANTS])
def test_each_planted_spmm_mistake_fails_a_pin(what, old, new):
    assert SPMM_SRC.count(old) == 1, f"the mutation site for '{what}' must occur exactly once"
    assert _spmm_failing(SPMM_SRC.replace(old, new)), f"no pin caught: {what}"


# ------------------------------------------------------ screened SpMM --
SCREEN_SRC = open(os.path.join(ORACLE_DIR, "screened.py")).read()


def pin_screen_pairs(mod):
    diag = np.random.default_rng(60).standard_normal(96).astype(np.float32) * 0.3
    thr = 1e-2
    M = mod.schwarz_mask(diag, thr)
    t = np.float32(math.sqrt(np.float32(thr)))
    for i in range(0, 96, 7):
        for j in range(0, 96, 5):
            qi = np.float32(math.sqrt(abs(float(diag[i]))))
            qj = np.float32(math.sqrt(abs(float(diag[j]))))
            assert bool(M[i, j]) == bool(np.float32(qi * qj) > t)


def pin_screen_defining_sum(mod):
    rng = np.random.default_rng(61)
    A, Bm = rng.standard_normal((48, 48)), rng.standard_normal((48, 6))
    diag = rng.standard_normal(48).astype(np.float32)
    thr = 0.05
    C = mod.screened_spmm(A, diag, Bm, thr)
    q = [math.sqrt(abs(float(x))) for x in diag]
    for i in range(0, 48, 5):
        for c in range(6):
            want = sum(A[i, j] * Bm[j, c] for j in range(48) if np.float32(q[i]) * np.float32(q[j]) > np.float32(
                math.sqrt(np.float32(thr))))
            assert abs(C[i, c] - want) <= 1e-10 * max(1.0, abs(want))


SCREEN_MUTANTS = [
    ("absolute value left out", "q = np.sqrt(np.abs(np.asarray(diag, dtype=np.float32)))",
     "q = np.sqrt(np.asarray(diag, dtype=np.float32))"),
    ("threshold not square-rooted", "t = np.sqrt(np.float32(threshold))", "t = np.float32(threshold)"),
    ("one-sided bound", "(q[:, None] * q[None, :]) > t", "(q[:, None] * q[:, None]) > t"),
    ("mask inverted", "(q[:, None] * q[None, :]) > t", "(q[:, None] * q[None, :]) <= t"),
    ("mask applied to B instead of A", "(np.asarray(A, dtype=np.float64) * M) @ np.asarray(B, dtype=np.float64)",
     "np.asarray(A, dtype=np.float64) @ (M[:, :B.shape[1]] * np.asarray(B, dtype=np.float64))"),
]


def _screen_failing(src):
    mod = types.ModuleType("oracle_screened_variant")
    exec(compile(src, "oracle_screened_variant", "exec"), mod.__dict__)
    failed = []
    for pin in (pin_screen_pairs, pin_screen_defining_sum):
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_unmodified_screened_oracle_passes_its_pins():
    assert _screen_failing(SCREEN_SRC) == []


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # the square root of a negative bound
@pytest.mark.parametrize("what,old,new", SCREEN_MUTANTS, ids=[m[0] for m in SCREEN_MUTANTS])
def test_each_planted_screened_mistake_fails_a_pin(what, old, new):
    assert SCREEN_SRC.count(old) == 1, f"the mutation site for '{what}' must occur exactly once"
    assert _screen_failing(SCREEN_SRC.replace(old, new)), f"no pin caught: {what}"
