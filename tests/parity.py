"""Helpers for the GPU-vs-oracle parity tests (the CUDA path is called through the C ABI)."""

from __future__ import annotations

import numpy as np
import torch

import block_sparse_attention_bsr_gb300 as bsr
import oracle

# Tolerances.  fp32 operands: max-abs 1e-4 on O / dQ / dK / dV and 1e-5
# relative on every element of the statistics.  bf16 operands: 2e-2
# relative-to-max on the outputs and gradients against the oracle run on the
# bf16-rounded inputs, 1e-4 relative on every element of the fp32 statistics.
# fp16 operands: the same with 5e-3 on the outputs and gradients -- P, dS and
# the outputs are rounded to 11 significant bits instead of 8 (relative step
# 2^-11 against 2^-8), so the bf16 bar scaled by the step ratio with a margin
# of about two.  The statistics are compared element by element:
# |got - ref| <= stat_rel * |ref| for row_denom (>= 1 on every non-empty row)
# and |got - ref| <= stat_rel * max(|ref|, 1) for row_max, whose value can
# sit near 0 where a relative bar alone would ask for more than fp32 gives.
TOL = {
    "f32": dict(out_abs=1e-4, out_rel=None, stat_rel=1e-5),
    "bf16": dict(out_abs=None, out_rel=2e-2, stat_rel=1e-4),
    "f16": dict(out_abs=None, out_rel=5e-3, stat_rel=1e-4),
}


def run_gpu(Q, K, V, dO, bm, scale, device="cuda", backward=True, two_pass=False, api="per-call"):
    """Runs forward (+ backward) through the C ABI on `device`; returns CPU float64 numpy arrays.

    ``api`` picks the entry points: "per-call" (bsr_attn_fwd / bsr_attn_bwd, which plan on every call) or
    "plan" (bsr_attn_fwd_plan / bsr_attn_bwd_plan on a plan built first, the calls the benchmark times).
    ``two_pass`` runs the statistics-first forward (bsr_attn_fwd_two_pass, per call)."""
    dev = torch.device(device)
    rp, ci = _bsr(bm)
    st = bsr.Structure(rp, ci, bm.shape[1], dev)
    q, k, v, do = (t.to(dev).contiguous() for t in (Q, K, V, dO))
    O = torch.empty_like(q)
    rm = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    rd = torch.empty_like(rm)
    plan = st.plan(q) if api == "plan" else None
    if plan is not None:
        bsr.bsr_attn_fwd_plan(plan, q, k, v, scale, O, rm, rd)
    else:
        bsr.bsr_attn_fwd(q, k, v, st.row_ptr, st.col_idx, st.n_brows, 128, scale, O, rm, rd, two_pass=two_pass)
    out = dict(O=O, row_max=rm, row_denom=rd)
    if backward:
        dQ, dK, dV = (torch.empty_like(q) for _ in range(3))
        if plan is not None:
            bsr.bsr_attn_bwd_plan(plan, q, k, v, O, do, rm, rd, scale, dQ, dK, dV)
        else:
            bsr.bsr_attn_bwd(q, k, v, O, do, rm, rd, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, scale,
                             dQ, dK, dV)
        out.update(dQ=dQ, dK=dK, dV=dV)
    bsr.bsr_attn_check()
    res = {n: t.double().cpu().numpy() for n, t in out.items()}
    if plan is not None:
        plan.close()
    return res


def kernels_run(Q, K, V, dO, bm, scale, device="cuda", api="per-call"):
    """Names of the library kernels one forward + backward launches (per-launch timing on)."""
    bsr.profile_collect()
    bsr.profile_enable(True)
    try:
        run_gpu(Q, K, V, dO, bm, scale, device=device, api=api)
    finally:
        bsr.profile_enable(False)
    return set(bsr.profile_collect())


def expected_plan_kernels(dtype: str, D: int, empty_lines: bool = False) -> set:
    """The kernels of a plan's creation (the planner, once) and of a forward + backward on it: the dK/dV walk
    (16-bit, head_dim 64 / 128) or the wide dK walk stores dS (fp32: as two bf16 pieces) and the dQ walk sums
    dS K over the stored tiles (dq_ds); in the wide kernels (head_dim 256 / 512, fp32) the dK walk also stores
    P^T and dV sums P^T dO over it (dv_ps); the zero-lines pass where lines are empty."""
    if dtype in ("bf16", "f16") and D <= 128:
        k = {"plan", "fwd_tc", "delta", "dkdv_tc", "dq_ds"}
    elif dtype in ("bf16", "f16"):  # the dK walk also stores P^T; dV streams it (dv_ps)
        k = {"plan", "fwd_wide", "delta", "dk_wide", "dq_ds", "dv_ps"}
    else:  # fp32: dS and P^T as two bf16 pieces each
        k = {"plan", "split3", "fwd_wide", "delta", "dk_wide", "dq_ds", "dv_ps"}
    return k | {"zero_lines"} if empty_lines else k


def expected_kernels(dtype: str, D: int) -> set:
    """The kernels that serve (dtype, head_dim) on the per-call entry points: the key-halves forward and the
    fused dK/dV backward for 16-bit operands with head_dim 64 / 128, the wide kernels otherwise (fp32 after its
    bf16 split); the outputs of empty lines are written by extra CTAs of the planner launches."""
    if dtype in ("bf16", "f16") and D <= 128:
        return {"plan", "fwd_tc", "delta_plan", "dq_tc", "dkdv_tc"}
    k = {"plan", "fwd_wide", "delta", "dq_wide", "dv_wide", "dk_wide"}
    return k | {"split3"} if dtype == "f32" else k


def _bsr(bm):
    from block_sparse_attention_bsr_gb300 import inputs

    return inputs.bsr_from_block_mask(bm)


def oracle_heads(Q, K, V, dO, bm, scale, heads, backward=True):
    """Oracle results for selected (batch, head) pairs: {name: [len(heads), S, ...]}."""
    res = {n: [] for n in ("O", "row_max", "row_denom", "dQ", "dK", "dV")}
    for b, h in heads:
        args = [t[b, h].double().numpy() for t in (Q, K, V, dO)]
        if backward:
            o, rm, rd, dq, dk, dv = oracle.attn_fwd_bwd_head(*args, bm, scale)
            res["dQ"].append(dq)
            res["dK"].append(dk)
            res["dV"].append(dv)
        else:
            o4, rm4, rd4 = oracle.attn_fwd(*(a[None, None] for a in args[:3]), bm, scale)
            o, rm, rd = o4[0, 0], rm4[0, 0], rd4[0, 0]
        res["O"].append(o)
        res["row_max"].append(rm)
        res["row_denom"].append(rd)
    return {n: np.stack(v) for n, v in res.items() if v}


def compare(got: dict, ref: dict, dtype: str, heads=None, what="", stat_rel=None) -> dict:
    """Asserts parity within TOL[dtype] (stat_rel overrides the statistics' bar); returns the measured errors."""
    tol = dict(TOL[dtype])
    if stat_rel is not None:
        tol["stat_rel"] = stat_rel
    errs = {}
    for name, r in ref.items():
        g = got[name]
        if heads is not None:
            g = np.stack([g[b, h] for b, h in heads])
        else:
            g = g.reshape(r.shape)
        if name in ("row_max", "row_denom"):
            fin = np.isfinite(r)
            assert np.array_equal(fin, np.isfinite(g)), f"{what} {name}: -inf pattern differs"
            if name == "row_denom":
                fin &= r != 0  # empty rows: exactly 0
            assert np.array_equal(g[~fin], r[~fin]), f"{what} {name}: empty-row values differ"
            if fin.any():
                floor = 1.0 if name == "row_max" else 0.0
                rel = np.abs(g[fin] - r[fin]) / np.maximum(np.abs(r[fin]), floor)
                err = float(rel.max())
            else:
                err = 0.0
            errs[name] = err
            assert err <= tol["stat_rel"], f"{what} {name}: elementwise relative error {err:.3e} > {tol['stat_rel']}"
            continue
        diff = np.abs(g - r)
        if tol["out_abs"] is not None:
            err = float(diff.max())
            errs[name] = err
            assert err <= tol["out_abs"], f"{what} {name}: max-abs error {err:.3e} > {tol['out_abs']}"
        else:
            err = float(diff.max() / max(np.abs(r).max(), 1e-30))
            errs[name] = err
            assert err <= tol["out_rel"], f"{what} {name}: rel-to-max error {err:.3e} > {tol['out_rel']}"
    return errs
