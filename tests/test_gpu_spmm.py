"""GPU parity of bsr_spmm (through the C ABI) against the fp64 oracle.

Tolerance, relative to the largest |Y|: the products of 16-bit operands are
exact in fp32 and the fp32 sums over at most a few thousand terms are far
below the final rounding of Y to the operand type (half a unit in the last
place: 2^-9 relative for bf16, 2^-12 for fp16), so 1e-2 (bf16) and 2e-3
(fp16) leave a margin of about five.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsr_gb300 as bsr
import oracle
from block_sparse_attention_bsr_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 2e-3}


def _run(n_brows, n_bcols, n_cols, p, dtype, seed=0):
    bm, blocks, X = inputs.make_spmm(n_brows, n_bcols, n_cols, p, dtype, seed)
    rp, ci = inputs.bsr_from_block_mask(bm)
    dev = torch.device("cuda")
    Y = torch.empty(n_brows * 128, n_cols, dtype=X.dtype, device=dev)
    bsr.bsr_spmm(blocks.to(dev), torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev), n_brows, n_bcols,
                 X.to(dev), Y)
    bsr.bsr_attn_check()
    got = Y.double().cpu().numpy()
    ref = oracle.spmm(blocks.double().numpy(), rp, ci, n_brows, n_bcols, X.double().numpy())
    return bm, got, ref


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(6, 5, 64, 0.4), (4, 8, 128, 0.5), (3, 3, 384, 1.0), (8, 8, 256, 0.1)])
def test_spmm_matches_oracle(shape, dtype):
    bm, got, ref = _run(*shape, dtype)
    err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= TOL[dtype], (shape, dtype, err)
    for m in np.nonzero(~bm.any(axis=1))[0]:  # empty block rows are zero
        assert np.all(got[m * 128:(m + 1) * 128] == 0)


def test_spmm_seq_8192_width_512():
    # the pages' shape (8192 x 8192 at block density ~13 %, times 8192 x 512),
    # checked on sampled block rows
    bm, blocks, X = inputs.make_spmm(64, 64, 512, 0.13, "bf16", 3)
    rp, ci = inputs.bsr_from_block_mask(bm)
    dev = torch.device("cuda")
    Y = torch.empty(64 * 128, 512, dtype=X.dtype, device=dev)
    bsr.bsr_spmm(blocks.to(dev), torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev), 64, 64, X.to(dev), Y)
    bsr.bsr_attn_check()
    got = Y.double().cpu().numpy()
    Xd = X.double().numpy()
    for m in (0, 17, 63):
        want = np.zeros((128, 512))
        for j in range(rp[m], rp[m + 1]):
            want += blocks[j].double().numpy() @ Xd[ci[j] * 128:(ci[j] + 1) * 128]
        err = np.abs(got[m * 128:(m + 1) * 128] - want).max() / max(np.abs(want).max(), 1e-30)
        assert err <= TOL["bf16"], (m, err)


def test_spmm_no_stored_block_gives_zeros():
    dev = torch.device("cuda")
    Y = torch.full((256, 64), 7.0, dtype=torch.bfloat16, device=dev)
    blocks = torch.empty(0, 128, 128, dtype=torch.bfloat16, device=dev)
    X = torch.randn(128, 64, device=dev).bfloat16()
    rp = torch.zeros(3, dtype=torch.int32, device=dev)
    ci = torch.zeros(1, dtype=torch.int32, device=dev)
    bsr.bsr_spmm(blocks, rp, ci, 2, 1, X, Y)
    torch.cuda.synchronize()
    assert bool((Y == 0).all())


@pytest.mark.parametrize("n_cols", [128, 256])
def test_spmm_heavy_row_beside_sparse_rows(n_cols):
    # block row 0 stores all 40 blocks, the others one to three; compared
    # whole against the oracle.
    nb = 40
    g = torch.Generator().manual_seed(5)
    bm = (torch.rand(nb, nb, generator=g) < 0.05).numpy()
    bm[np.arange(nb), np.arange(nb)] = True
    bm[0, :] = True
    nnzb = int(bm.sum())
    blocks = torch.randn(nnzb, 128, 128, generator=g).bfloat16()
    X = torch.randn(nb * 128, n_cols, generator=g).bfloat16()
    rp, ci = inputs.bsr_from_block_mask(bm)
    dev = torch.device("cuda")
    Y = torch.empty(nb * 128, n_cols, dtype=torch.bfloat16, device=dev)
    bsr.bsr_spmm(blocks.to(dev), torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev), nb, nb, X.to(dev), Y)
    bsr.bsr_attn_check()
    got = Y.double().cpu().numpy()
    ref = oracle.spmm(blocks.double().numpy(), rp, ci, nb, nb, X.double().numpy())
    err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= TOL["bf16"], err
