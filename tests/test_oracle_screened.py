"""Pins of the screened-SpMM oracle (oracle/screened.py) against things other than itself."""

import math

import numpy as np

import oracle
from block_sparse_attention_bsr_gb300 import inputs


def _case(n=256, w=64, seed=0):
    A, diag, B = inputs.make_screened(n, w, "bf16", seed)
    return A.double().numpy(), diag.numpy(), B.double().numpy()


def test_mask_pairs_follow_the_bound():
    # each sampled pair decided from scalar float32 arithmetic
    _, diag, _ = _case(512)
    thr = 1e-2
    M = oracle.schwarz_mask(diag, thr)
    rng = np.random.default_rng(0)
    t = np.float32(math.sqrt(np.float32(thr)))
    for _ in range(500):
        i, j = int(rng.integers(512)), int(rng.integers(512))
        qi = np.float32(math.sqrt(abs(float(np.float32(diag[i])))))
        qj = np.float32(math.sqrt(abs(float(np.float32(diag[j])))))
        assert bool(M[i, j]) == bool(np.float32(qi * qj) > t)
    assert np.array_equal(M, M.T)


def test_elements_match_the_defining_sum():
    A, diag, B = _case(256, 64, 1)
    thr = 3e-2
    C = oracle.screened_spmm(A, diag, B, thr)
    M = oracle.schwarz_mask(diag, thr)
    rng = np.random.default_rng(1)
    for _ in range(30):
        i, c = int(rng.integers(256)), int(rng.integers(64))
        want = sum(A[i, j] * B[j, c] for j in range(256) if M[i, j])
        assert abs(C[i, c] - want) <= 1e-10 * max(1.0, abs(want))


def test_threshold_zero_is_the_plain_product():
    A, diag, B = _case(256, 64, 2)  # diag > 0 everywhere
    assert np.allclose(oracle.screened_spmm(A, diag, B, 0.0), A @ B, rtol=0, atol=1e-9)


def test_large_threshold_gives_zero():
    A, diag, B = _case(256, 64, 3)  # bounds <= 1
    assert np.all(oracle.screened_spmm(A, diag, B, 4.0) == 0)
