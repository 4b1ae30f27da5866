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

from parity import TOL, oracle_heads

pytestmark = pytest.mark.gpu


def _max_err(a, b, dtype):
    a = a.double().cpu().numpy() if hasattr(a, "cpu") else a
    b = b.double().cpu().numpy() if hasattr(b, "cpu") else b
    if TOL[dtype]["out_abs"] is not None:
        return float(np.abs(a - b).max()), TOL[dtype]["out_abs"]
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)), TOL[dtype]["out_rel"]


# (dtype, head_dim, block rows, batch, heads).  The 32-block-row case has
# block row 0 and block column 0 of 32 blocks, longer than the regular path's
# per-CTA share (max(8, stored blocks * heads / CTAs) = 8 blocks), so
# bsr_attn_bwd splits them into chunks merged by the last arriver while
# bsr_attn_bwd_noalloc walks them whole: the two paths differ there.
CASES = [("f32", 64, 6, 2, 3), ("bf16", 128, 6, 2, 3), ("bf16", 128, 32, 1, 2)]


@pytest.mark.parametrize("dtype,D,nb,B,H", CASES)
def test_noalloc_backward_matches_regular_backward_twice(dtype, D, nb, B, H):
    dev = torch.device("cuda")
    bm = inputs.block_mask("global", nb, radius=1)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, nb, dev)
    heads = [(b, h) for b in range(B) for h in range(H)]
    for call, seed in enumerate((11, 12)):
        hQ, hK, hV, hdO = inputs.make_qkvdo(B, H, nb * 128, D, dtype, 1.0, seed)
        Q, K, V, dO = (t.to(dev) for t in (hQ, hK, hV, hdO))
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
        orc = oracle_heads(hQ, hK, hV, hdO, bm, scale, heads)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert not torch.isnan(g).any(), (call, name)
            err, tol = _max_err(g, r, dtype)
            assert err <= tol, (call, name, "noalloc vs regular", err, tol)
            for label, t in (("noalloc", g), ("regular", r)):
                gh = np.stack([t[b, h].double().cpu().numpy() for b, h in heads])
                err, tol = _max_err(gh, orc[name], dtype)
                assert err <= tol, (call, name, label + " vs oracle", err, tol)


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
