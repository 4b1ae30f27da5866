"""GPU parity of bsr_screened_spmm (through the C ABI) against the fp64 oracle.

The mask is decided in fp32 on both sides, so the comparison is of the
masked products only; tolerance relative to the largest |C| as for bsr_spmm
(1e-2 bf16, 2e-3 fp16: the final rounding of C dominates).
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsr_gb300 as bsr
import oracle
from block_sparse_attention_bsr_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 2e-3}


def _run(n, w, thr, dtype, seed=0):
    A, diag, B = inputs.make_screened(n, w, dtype, seed)
    dev = torch.device("cuda")
    C = torch.empty(n, w, dtype=A.dtype, device=dev)
    bsr.bsr_screened_spmm(A.to(dev), diag.to(dev), B.to(dev), thr, C)
    bsr.bsr_attn_check()
    got = C.double().cpu().numpy()
    ref = oracle.screened_spmm(A.double().numpy(), diag.numpy(), B.double().numpy(), thr)
    return got, ref


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("n,w,thr", [(1024, 128, 1e-2), (768, 64, 1e-1), (1024, 384, 1e-3), (512, 128, 0.5),
                                     (4096, 128, 1e-2), (4096, 256, 1e-3)])
def test_screened_matches_oracle(n, w, thr, dtype):
    got, ref = _run(n, w, thr, dtype)
    scale = max(np.abs(ref).max(), 1e-30)
    err = np.abs(got - ref).max() / scale
    assert err <= TOL[dtype], (n, w, thr, dtype, err)


def test_screened_threshold_zero_and_everything_screened():
    got, ref = _run(512, 64, 0.0, "bf16", 1)  # every pair kept: the plain product
    assert np.abs(got - ref).max() <= TOL["bf16"] * np.abs(ref).max()
    got, _ = _run(512, 64, 4.0, "bf16", 2)  # bounds <= 1: nothing kept, C = 0
    assert np.all(got == 0)
