"""Host-side input generators: masks against closed-form counts, BSR encoding, seeding."""

import os

import numpy as np
import pytest

from block_sparse_attention_bsr_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mask_counts.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, nb, r, nnzb, mx, mn = line.split()
            rows.append((k, int(nb), int(r), int(nnzb), int(mx), int(mn)))
    return rows


@pytest.mark.parametrize("kind,nb,radius,nnzb,mx,mn", _golden_rows())
def test_mask_counts_match_closed_forms(kind, nb, radius, nnzb, mx, mn):
    bm = inputs.block_mask(kind, nb, radius=radius)
    counts = bm.sum(axis=1)
    assert bm.sum() == nnzb and counts.max() == mx and counts.min() == mn
    if kind == "local" or kind == "dilated":
        assert (bm == bm.T).all()


def test_random_mask_density_and_diagonal():
    for p in (0.01, 0.05, 0.13, 0.27, 0.5):
        bm = inputs.block_mask("random", 64, p=p, seed=1)
        assert bm[np.arange(64), np.arange(64)].all()
        off = bm.sum() - 64
        exp = p * 64 * 63
        assert abs(off - exp) < 5 * np.sqrt(exp * (1 - p)) + 1
        assert (inputs.block_mask("random", 64, p=p, seed=1) == bm).all()


def test_bsr_encoding_row_major():
    bm = inputs.block_mask("random", 11, p=0.3)
    row_ptr, col_idx = inputs.bsr_from_block_mask(bm)
    assert row_ptr.dtype == np.int32 and col_idx.dtype == np.int32
    assert row_ptr[0] == 0 and row_ptr[-1] == bm.sum()
    for m in range(11):
        cols = col_idx[row_ptr[m]:row_ptr[m + 1]]
        assert list(cols) == list(np.nonzero(bm[m])[0])


def test_seeded_inputs_reproducible_and_rounded():
    a = inputs.make_qkvdo(1, 2, 256, 64, "bf16", 0.5, seed=3)
    b = inputs.make_qkvdo(1, 2, 256, 64, "bf16", 0.5, seed=3)
    for x, y in zip(a, b):
        assert x.dtype == y.dtype and bool((x == y).all())
    f = inputs.make_qkvdo(1, 2, 256, 64, "f32", 0.5, seed=3)
    assert abs(float(f[0].std()) - 0.5) < 0.02
    assert bool((f[0].bfloat16() == a[0]).all())
