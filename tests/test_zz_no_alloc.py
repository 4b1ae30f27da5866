"""The allocation-free backward entry point against the regular one (GPU).

bsr_attn_bwd_noalloc serves callers that cannot allocate device memory (the
device is owned by another allocator, or the hot path may not call the CUDA
allocator): it takes its scratch from static device memory instead.  Its
results must match bsr_attn_bwd's within the parity tolerance, on two calls
in a row (the second call reuses the static scratch the first one left
behind).  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsr_gb300 as bsr
from block_sparse_attention_bsr_gb300 import inputs

from parity import TOL

pytestmark = pytest.mark.gpu


def _max_err(a, b, dtype):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    if TOL[dtype]["out_abs"] is not None:
        return float(np.abs(a - b).max()), TOL[dtype]["out_abs"]
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)), TOL[dtype]["out_rel"]


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 128)])
def test_noalloc_backward_matches_regular_backward_twice(dtype, D):
    dev = torch.device("cuda")
    bm = inputs.block_mask("global", 6, radius=1)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, 6, dev)
    for call, seed in enumerate((11, 12)):
        Q, K, V, dO = (t.to(dev) for t in inputs.make_qkvdo(2, 3, 6 * 128, D, dtype, 1.0, seed))
        scale = 1.0 / np.sqrt(D)
        O = torch.empty_like(Q)
        rm = torch.empty(Q.shape[:3], device=dev, dtype=torch.float32)
        rd = torch.empty_like(rm)
        bsr.bsr_attn_fwd(Q, K, V, st.row_ptr, st.col_idx, st.n_brows, 128, scale, O, rm, rd)
        ref = [torch.empty_like(Q) for _ in range(3)]
        got = [torch.full_like(Q, float("nan")) for _ in range(3)]
        bsr.bsr_attn_bwd(Q, K, V, O, dO, rm, rd, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, scale, *ref)
        bsr.bsr_attn_bwd_noalloc(Q, K, V, O, dO, rm, rd, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, scale,
                                 *got)
        bsr.bsr_attn_check()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert not torch.isnan(g).any(), (call, name)
            err, tol = _max_err(g, r, dtype)
            assert err <= tol, (call, name, err, tol)


def test_noalloc_rejects_sizes_beyond_static_scratch():
    dev = torch.device("cuda")
    # batch * heads * seq = 2 * 4 * 131200 > 1,048,576 rows; rejected before any launch
    shape = (2, 4, 131200, 64)
    t = torch.empty(1, device=dev)
    desc = bsr.bsr_tensor(t.data_ptr(), bsr.BSR_F32, *shape)
    import ctypes

    lib = bsr.load_library()
    P = ctypes.c_void_p
    p = t.data_ptr()
    status = lib.bsr_attn_bwd_noalloc(*(ctypes.byref(desc) for _ in range(5)), P(p), P(p), P(p), P(p), P(p), P(p),
                                      0.125, *(ctypes.byref(desc) for _ in range(3)), None)
    assert status == 1
    assert "static scratch" in lib.bsr_last_error().decode()
