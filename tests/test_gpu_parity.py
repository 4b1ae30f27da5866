"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle.

Small workloads are compared element by element on every head; the seq-8192
workloads run in full on the GPU (the launch configuration the benchmark
times) and are compared on sampled heads, each recomputed whole by the
oracle.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_bsr_gb300 import inputs

from parity import compare, oracle_heads, run_gpu

pytestmark = pytest.mark.gpu


def _workload(name, heads=None, seed=0):
    wl = inputs.WORKLOADS[name]
    bm = wl.block_mask()
    Q, K, V, dO = wl.inputs(seed=seed)
    got = run_gpu(Q, K, V, dO, bm, wl.scale)
    if heads is None:
        heads = [(b, h) for b in range(wl.batch) for h in range(wl.heads)]
    ref = oracle_heads(Q, K, V, dO, bm, wl.scale, heads)
    return compare(got, ref, wl.dtype, heads=heads, what=name)


def test_tiny_fp32_all_heads():
    _workload("tiny")


def test_dilated_s2048_bf16_all_heads():
    _workload("dilated_s2048")


def _workload_as(name, dtype, heads=None, seed=0):
    # a workload's mask and shape with operands drawn in another dtype
    wl = inputs.WORKLOADS[name]
    bm = wl.block_mask()
    Q, K, V, dO = inputs.make_qkvdo(wl.batch, wl.heads, wl.seq, wl.head_dim, dtype, 1.0, seed)
    got = run_gpu(Q, K, V, dO, bm, wl.scale)
    if heads is None:
        heads = [(b, h) for b in range(wl.batch) for h in range(wl.heads)]
    ref = oracle_heads(Q, K, V, dO, bm, wl.scale, heads)
    return compare(got, ref, dtype, heads=heads, what=f"{name} {dtype}")


def test_dilated_s2048_f16_all_heads():
    _workload_as("dilated_s2048", "f16")


def test_global_s8192_f16_sampled_heads():
    _workload_as("global_s8192", "f16", heads=[(0, 0), (0, 15)])


@pytest.mark.parametrize("name", ["global_s8192", "global_s8192_f32"])
def test_global_s8192_sampled_heads(name):
    _workload(name, heads=[(0, 0), (0, 15)])


@pytest.mark.parametrize("name", ["local_s8192_d256", "local_s8192_d512"])
def test_local_s8192_large_head_dim_sampled_heads(name):
    _workload(name, heads=[(0, 0), (0, 7)])


@pytest.mark.parametrize("p", [0.01, 0.05, 0.13, 0.27, 0.5])
def test_random_density_sweep_sampled_head(p):
    _workload(f"random_p{p}", heads=[(0, 5)])


# ------------------------------------------------------------ edge cases --

def _edge(bm, dtype, D=64, B=1, H=2, std=1.0, seed=3):
    nb = bm.shape[0]
    Q, K, V, dO = inputs.make_qkvdo(B, H, nb * 128, D, dtype, std, seed)
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(Q, K, V, dO, bm, scale)
    ref = oracle_heads(Q, K, V, dO, bm, scale, [(b, h) for b in range(B) for h in range(H)])
    return got, compare(got, ref, dtype, heads=[(b, h) for b in range(B) for h in range(H)])


DTYPES = ["f32", "bf16", "f16"]


@pytest.mark.parametrize("dtype", DTYPES)
def test_empty_block_row_and_column(dtype):
    bm = inputs.block_mask("local", 5, radius=1)
    bm[2, :] = False  # block row 2 attends to nothing
    bm[:, 4] = False  # nobody attends to block column 4
    got, _ = _edge(bm, dtype)
    rows = slice(2 * 128, 3 * 128)
    assert np.all(got["O"][:, :, rows] == 0)
    assert np.all(got["row_max"][:, :, rows] == -np.inf) and np.all(got["row_denom"][:, :, rows] == 0)
    assert np.all(got["dQ"][:, :, rows] == 0)
    cols = slice(4 * 128, 5 * 128)
    assert np.all(got["dK"][:, :, cols] == 0) and np.all(got["dV"][:, :, cols] == 0)


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_stored_block(dtype):
    bm = np.zeros((3, 3), bool)
    bm[1, 2] = True
    _edge(bm, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_full_mask_ragged_grid(dtype):
    _edge(np.ones((5, 5), bool), dtype, D=128)


@pytest.mark.parametrize("dtype", DTYPES)
def test_heavy_row_beside_single_block_rows(dtype):
    bm = np.eye(9, dtype=bool)
    bm[0, :] = True
    bm[:, 3] = True
    _edge(bm, dtype, D=128, H=3)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_head_dims(dtype, D):
    bm = inputs.block_mask("random", 4, p=0.4, seed=D)
    _edge(bm, dtype, D=D, B=2, H=1, std=0.5)


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_block_sequence(dtype):
    _edge(np.ones((1, 1), bool), dtype, D=128, B=2, H=2)


def test_large_scores_stable():
    # Inputs with std 2: scores (std 4) reach about +-20, so the online
    # rescaling runs often.  fp32 score rounding grows with |score|, so the
    # max-abs bar is scaled by the value magnitude (std^2).
    bm = inputs.block_mask("global", 6, radius=1)
    std = 2.0
    Q, K, V, dO = inputs.make_qkvdo(1, 2, 6 * 128, 128, "f32", std, 4)
    scale = 1.0 / np.sqrt(128)
    got = run_gpu(Q, K, V, dO, bm, scale)
    ref = oracle_heads(Q, K, V, dO, bm, scale, [(0, 0), (0, 1)])
    for name in ("O", "dQ", "dK", "dV"):
        err = np.abs(got[name][0] - ref[name]).max()
        assert err <= 1e-4 * std ** 2, (name, err)
    compare({k: got[k] for k in ("row_max", "row_denom")}, {k: ref[k] for k in ("row_max", "row_denom")},
            "f32", heads=[(0, 0), (0, 1)])


def test_repeated_calls_identical():
    bm = inputs.block_mask("dilated", 6, radius=2)
    Q, K, V, dO = inputs.make_qkvdo(1, 4, 768, 128, "bf16", 1.0, 9)
    a = run_gpu(Q, K, V, dO, bm, 0.1)
    b = run_gpu(Q, K, V, dO, bm, 0.1)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_device_index_check_reports_error():
    # A column index outside the grid is skipped by the kernels' own bounds
    # check and reported through bsr_attn_check; nothing is read out of range.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    q = torch.randn(1, 1, 256, 64, device=dev)
    row_ptr = torch.tensor([0, 1, 2], dtype=torch.int32, device=dev)
    col_idx = torch.tensor([0, 7], dtype=torch.int32, device=dev)  # 7 is outside a 2-block grid
    O = torch.empty_like(q)
    rm = torch.empty(1, 1, 256, device=dev)
    rd = torch.empty_like(rm)
    bsr.bsr_attn_fwd(q, q, q, row_ptr, col_idx, 2, 128, 0.125, O, rm, rd)
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_check()
    assert e.value.status == 5
    bsr.bsr_attn_check()  # the status word was cleared


def test_backward_same_with_per_launch_timing():
    # With per-launch timing on, dQ and dK/dV run one after the other on the
    # caller's stream instead of side by side on two streams: same results.
    import block_sparse_attention_bsr_gb300 as bsr

    bm = inputs.block_mask("global", 16, radius=2)
    Q, K, V, dO = inputs.make_qkvdo(1, 4, 16 * 128, 128, "bf16", 1.0, 11)
    a = run_gpu(Q, K, V, dO, bm, 0.09)
    bsr.profile_enable(True)
    try:
        b = run_gpu(Q, K, V, dO, bm, 0.09)
    finally:
        bsr.profile_enable(False)
        bsr.profile_collect()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_misaligned_output_is_rejected():
    # Output views must be 16-byte aligned (vector stores in the epilogues):
    # a view one element in is refused on the host, nothing is launched.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    q = torch.randn(1, 1, 256, 64, device=dev, dtype=torch.bfloat16)
    row_ptr = torch.tensor([0, 1, 2], dtype=torch.int32, device=dev)
    col_idx = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    buf = torch.empty(1 * 1 * 256 * 64 + 1, device=dev, dtype=torch.bfloat16)
    O = buf[1:].view(1, 1, 256, 64)
    rm = torch.empty(1, 1, 256, device=dev)
    rd = torch.empty_like(rm)
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_fwd(q, q, q, row_ptr, col_idx, 2, 128, 0.125, O, rm, rd)
    assert e.value.status == 1 and "aligned" in str(e.value)


def test_autograd_wrapper_matches_direct_calls():
    # block_sparse_attention (torch autograd over the C ABI) gives the direct
    # calls' outputs and gradients bit for bit.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    bm = inputs.block_mask("local", 8, radius=2)
    Q, K, V, dO = inputs.make_qkvdo(1, 2, 8 * 128, 128, "bf16", 1.0, 21)
    direct = run_gpu(Q, K, V, dO, bm, 1.0 / np.sqrt(128))
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, bm.shape[1], dev)
    q, k, v = (t.to(dev).requires_grad_() for t in (Q, K, V))
    O, rm, rd = bsr.block_sparse_attention(q, k, v, st, return_stats=True)
    O.backward(dO.to(dev))
    got = dict(O=O.detach(), row_max=rm, row_denom=rd, dQ=q.grad, dK=k.grad, dV=v.grad)
    for name, t in got.items():
        assert np.array_equal(t.double().cpu().numpy(), direct[name]), name


# ------------------------------------------------ statistics-first forward --

FWD = ("O", "row_max", "row_denom")


def _two_pass(bm, dtype, D=128, B=1, H=2, seed=5, backward=False, heads=None):
    nb = bm.shape[0]
    Q, K, V, dO = inputs.make_qkvdo(B, H, nb * 128, D, dtype, 1.0, seed)
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(Q, K, V, dO, bm, scale, backward=backward, two_pass=True)
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    ref = oracle_heads(Q, K, V, dO, bm, scale, heads, backward=backward)
    names = FWD + (("dQ", "dK", "dV") if backward else ())
    compare({k: got[k] for k in names}, {k: ref[k] for k in names}, dtype, heads=heads, what="two-pass")
    return Q, K, V, dO, bm, scale, got


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_two_pass_forward_matches_oracle(dtype):
    # a heavy row (split into chunks on the full-size grid below) beside
    # single-block rows, and the statistics feeding the backward
    bm = np.eye(9, dtype=bool)
    bm[0, :] = True
    bm[:, 3] = True
    _two_pass(bm, dtype, H=3, backward=True)


def test_two_pass_forward_global_s8192_sampled_heads():
    # the full-size launch configuration: block row 0 (64 blocks) is split
    # across CTAs in both passes
    wl = inputs.WORKLOADS["global_s8192"]
    bm = wl.block_mask()
    Q, K, V, dO = wl.inputs(seed=0)
    got = run_gpu(Q, K, V, dO, bm, wl.scale, backward=False, two_pass=True)
    heads = [(0, 0), (0, 15)]
    ref = oracle_heads(Q, K, V, dO, bm, wl.scale, heads, backward=False)
    compare({k: got[k] for k in FWD}, {k: ref[k] for k in FWD}, "bf16", heads=heads, what="two-pass global_s8192")
    # same statistics as the online forward up to rounding, same output
    one = run_gpu(Q, K, V, dO, bm, wl.scale, backward=False)
    for k in ("row_max", "row_denom"):
        scale_ = np.abs(one[k][np.isfinite(one[k])]).max()
        assert np.nanmax(np.abs(got[k] - one[k])) <= 1e-5 * scale_, k
    assert np.abs(got["O"] - one["O"]).max() <= 2e-2 * np.abs(one["O"]).max()


def test_two_pass_forward_empty_block_row():
    bm = inputs.block_mask("local", 5, radius=1)
    bm[2, :] = False
    *_, got = _two_pass(bm, "bf16", D=64)
    rows = slice(2 * 128, 3 * 128)
    assert np.all(got["O"][:, :, rows] == 0)
    assert np.all(got["row_max"][:, :, rows] == -np.inf) and np.all(got["row_denom"][:, :, rows] == 0)


def test_two_pass_forward_refuses_fp32():
    import block_sparse_attention_bsr_gb300 as bsr

    bm = np.ones((2, 2), bool)
    Q, K, V, dO = inputs.make_qkvdo(1, 1, 256, 64, "f32", 1.0, 1)
    with pytest.raises(bsr.BsrError) as e:
        run_gpu(Q, K, V, dO, bm, 0.125, backward=False, two_pass=True)
    assert e.value.status == 2
