"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle.

Every workload runs in full on the GPU through both sets of entry points:
on a plan (the launch configuration the benchmark times) and per call.  The
global-mask and head_dim-256 / 512 workloads are compared element by element
on every (batch, head); the density sweep on four heads of sixteen, each
recomputed whole by the oracle.  Separate tests check which kernels served
each workload.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_bsr_gb300 import inputs

from parity import compare, expected_kernels, expected_plan_kernels, kernels_run, oracle_heads, run_gpu

pytestmark = pytest.mark.gpu


def _both_apis(Q, K, V, dO, bm, scale, dtype, heads, what):
    # the plan's entry points and the per-call ones against one oracle run
    got = {api: run_gpu(Q, K, V, dO, bm, scale, api=api) for api in ("plan", "per-call")}
    ref = oracle_heads(Q, K, V, dO, bm, scale, heads)
    return {api: compare(g, ref, dtype, heads=heads, what=f"{what} ({api})") for api, g in got.items()}


def _workload(name, heads=None, seed=0):
    wl = inputs.WORKLOADS[name]
    Q, K, V, dO = wl.inputs(seed=seed)
    if heads is None:
        heads = [(b, h) for b in range(wl.batch) for h in range(wl.heads)]
    return _both_apis(Q, K, V, dO, wl.block_mask(), wl.scale, wl.dtype, heads, name)


def test_tiny_fp32_all_heads():
    _workload("tiny")


def test_dilated_s2048_bf16_all_heads():
    _workload("dilated_s2048")


def _workload_as(name, dtype, heads=None, seed=0):
    # a workload's mask and shape with operands drawn in another dtype
    wl = inputs.WORKLOADS[name]
    Q, K, V, dO = inputs.make_qkvdo(wl.batch, wl.heads, wl.seq, wl.head_dim, dtype, 1.0, seed)
    if heads is None:
        heads = [(b, h) for b in range(wl.batch) for h in range(wl.heads)]
    return _both_apis(Q, K, V, dO, wl.block_mask(), wl.scale, dtype, heads, f"{name} {dtype}")


def test_dilated_s2048_f16_all_heads():
    _workload_as("dilated_s2048", "f16")


def test_global_s8192_f16_all_heads():
    _workload_as("global_s8192", "f16")


@pytest.mark.parametrize("name", ["global_s8192", "global_s8192_f32"])
def test_global_s8192_all_heads(name):
    _workload(name)


@pytest.mark.parametrize("name", ["local_s8192_d256", "local_s8192_d512"])
def test_local_s8192_large_head_dim_all_heads(name):
    _workload(name)


@pytest.mark.parametrize("p", [0.01, 0.05, 0.13, 0.27, 0.5])
def test_random_density_sweep_four_heads(p):
    _workload(f"random_p{p}", heads=[(0, 0), (0, 5), (0, 10), (0, 15)])


@pytest.mark.parametrize("name", sorted(inputs.WORKLOADS))
def test_workload_runs_on_its_tensor_core_kernels(name):
    # the kernels each workload launches, by name: no other code path serves it
    wl = inputs.WORKLOADS[name]
    Q, K, V, dO = wl.inputs(seed=0)
    bm = wl.block_mask()
    got = kernels_run(Q, K, V, dO, bm, wl.scale)
    assert got == expected_kernels(wl.dtype, wl.head_dim), (name, sorted(got))
    empty = bool((bm.sum(1) == 0).any() or (bm.sum(0) == 0).any())
    got = kernels_run(Q, K, V, dO, bm, wl.scale, api="plan")
    assert got == expected_plan_kernels(wl.dtype, wl.head_dim, empty), (name, "plan", sorted(got))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_every_dtype_and_head_dim_runs_on_tensor_core_kernels(dtype, D):
    bm = inputs.block_mask("local", 3, radius=1)
    Q, K, V, dO = inputs.make_qkvdo(1, 2, 3 * 128, D, dtype, 1.0, 1)
    got = kernels_run(Q, K, V, dO, bm, 1.0 / np.sqrt(D))
    assert got == expected_kernels(dtype, D), (dtype, D, sorted(got))
    got = kernels_run(Q, K, V, dO, bm, 1.0 / np.sqrt(D), api="plan")
    assert got == expected_plan_kernels(dtype, D), (dtype, D, "plan", sorted(got))


# ------------------------------------------------------------ edge cases --

def _edge(bm, dtype, D=64, B=1, H=2, std=1.0, seed=3):
    # both sets of entry points against the oracle; returns the plan's results
    nb = bm.shape[0]
    Q, K, V, dO = inputs.make_qkvdo(B, H, nb * 128, D, dtype, std, seed)
    scale = 1.0 / np.sqrt(D)
    heads = [(b, h) for b in range(B) for h in range(H)]
    ref = oracle_heads(Q, K, V, dO, bm, scale, heads)
    for api in ("per-call", "plan"):
        got = run_gpu(Q, K, V, dO, bm, scale, api=api)
        errs = compare(got, ref, dtype, heads=heads, what=api)
    return got, errs


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


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("bf16", 256), ("f32", 128)])
def test_mostly_empty_lines(dtype, D):
    # Only block rows 0-1 and block columns 0-3 hold blocks: 30 of 32 block
    # rows and 28 of 32 block columns are empty, in each of 16 heads.  The
    # work lists leave empty lines out (most persistent CTAs get no item at
    # all) and a separate pass writes their outputs.  Four heads are compared
    # with the oracle; every head's empty lines must come out as exact zeros
    # (-inf / 0 statistics).
    nb, B, H = 32, 2, 8
    bm = np.zeros((nb, nb), bool)
    bm[0:2, 0:4] = True
    Q, K, V, dO = inputs.make_qkvdo(B, H, nb * 128, D, dtype, 1.0, 5)
    scale = 1.0 / np.sqrt(D)
    heads = [(0, 0), (0, 5), (1, 2), (1, 7)]
    ref = oracle_heads(Q, K, V, dO, bm, scale, heads)
    for api in ("per-call", "plan"):
        got = run_gpu(Q, K, V, dO, bm, scale, api=api)
        compare(got, ref, dtype, heads=heads, what=f"mostly empty ({api})")
        rows, cols = slice(2 * 128, None), slice(4 * 128, None)
        assert np.all(got["O"][:, :, rows] == 0) and np.all(got["dQ"][:, :, rows] == 0)
        assert np.all(got["row_max"][:, :, rows] == -np.inf) and np.all(got["row_denom"][:, :, rows] == 0)
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
@pytest.mark.parametrize("D", [128, 256, 512])
def test_heavy_row_beside_single_block_rows(dtype, D):
    # Block row 0 and block column 3 hold all 20 blocks of their line, the
    # other lines one or two: the planner cuts the two long lines into chunks
    # of at most 8 blocks (three each), merged by the last chunk to finish.
    bm = np.eye(20, dtype=bool)
    bm[0, :] = True
    bm[:, 3] = True
    _edge(bm, dtype, D=D, H=3)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_head_dims(dtype, D):
    bm = inputs.block_mask("random", 4, p=0.4, seed=D)
    _edge(bm, dtype, D=D, B=2, H=1)


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_block_sequence(dtype):
    _edge(np.ones((1, 1), bool), dtype, D=128, B=2, H=2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_long_sequence_over_2048_block_rows(dtype):
    # 2100 block rows (seq 268800): the planner takes its paths for long line
    # lists (the backward's lists are built in a launch of their own above
    # 512 lines, and placed with atomics instead of the stable order above
    # 2048).  With the band |m - n| <= 1 the rows of block row m see only
    # key blocks m-1..m+1 and the keys of block column n only query blocks
    # n-1..n+1, so windows of five blocks around sampled n give the oracle's
    # exact values for O, the statistics and dQ of block row n and dK, dV of
    # block column n (the window's edge rows are complete for those).
    nb, D = 2100, 64
    bm = inputs.block_mask("local", nb, radius=1)
    Q, K, V, dO = inputs.make_qkvdo(1, 1, nb * 128, D, dtype, 1.0, 41)
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(Q, K, V, dO, bm, scale)
    for n in (0, 1, 700, 1049, 2098, 2099):
        lo, hi = max(n - 2, 0), min(n + 3, nb)
        sl = slice(lo * 128, hi * 128)
        sub = [t[:, :, sl] for t in (Q, K, V, dO)]
        ref = oracle_heads(*sub, bm[lo:hi, lo:hi], scale, [(0, 0)])
        rows = slice((n - lo) * 128, (n - lo + 1) * 128)
        piece = {k: got[k][:, :, n * 128:(n + 1) * 128] for k in ref}
        want = {k: r[:, rows] for k, r in ref.items()}
        compare(piece, want, dtype, heads=[(0, 0)], what=f"long sequence, block {n}")


def test_large_scores_stable():
    # Inputs with std 4: scores scale * q.k have std 16 and reach about +-70,
    # so the online rescaling runs often and the softmax is sharply peaked.
    # The max-abs bar of the N(0, 1) case, 1e-4, is scaled by how each output
    # grows with the input spread s: O = P V and dV = P^T dO grow like s;
    # dQ = scale dS K and dK = scale dS^T Q, with dS = P o (dO V^T - D), grow
    # like s^3.  The fp32 path keeps about 2^-23 relative error per product,
    # so these bars leave the same margin as at s = 1.
    bm = inputs.block_mask("global", 6, radius=1)
    std = 4.0
    Q, K, V, dO = inputs.make_qkvdo(1, 2, 6 * 128, 128, "f32", std, 4)
    scale = 1.0 / np.sqrt(128)
    got = run_gpu(Q, K, V, dO, bm, scale)
    ref = oracle_heads(Q, K, V, dO, bm, scale, [(0, 0), (0, 1)])
    bars = {"O": 1e-4 * std, "dV": 1e-4 * std, "dQ": 1e-4 * std ** 3, "dK": 1e-4 * std ** 3}
    for name, bar in bars.items():
        err = np.abs(got[name][0] - ref[name]).max()
        assert err <= bar, (name, err, bar)
    # The statistics: a score is an fp32 sum of 128 products whose sizes grow
    # like s^2, so its rounding error, which enters row_denom as a relative
    # error, grows like s^2 too (an exactly rounded fp32 dot product of these
    # terms has the same growth); the N(0, 1) bar 1e-5 is scaled by s^2.
    compare({k: got[k] for k in ("row_max", "row_denom")}, {k: ref[k] for k in ("row_max", "row_denom")},
            "f32", heads=[(0, 0), (0, 1)], stat_rel=1e-5 * std ** 2)


def test_repeated_calls_identical():
    bm = inputs.block_mask("dilated", 6, radius=2)
    Q, K, V, dO = inputs.make_qkvdo(1, 4, 768, 128, "bf16", 1.0, 9)
    a = run_gpu(Q, K, V, dO, bm, 0.1)
    b = run_gpu(Q, K, V, dO, bm, 0.1)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def _fwd_bwd_on_device(case):
    # one per-call forward + backward; the outputs stay on the device
    import block_sparse_attention_bsr_gb300 as bsr

    st, q, k, v, do, scale = case
    O = torch.empty_like(q)
    rm = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    rd = torch.empty_like(rm)
    bsr.bsr_attn_fwd(q, k, v, st.row_ptr, st.col_idx, st.n_brows, 128, scale, O, rm, rd)
    dQ, dK, dV = (torch.empty_like(q) for _ in range(3))
    bsr.bsr_attn_bwd(q, k, v, O, do, rm, rd, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, scale, dQ, dK, dV)
    return [O, rm, rd, dQ, dK, dV]


def test_kernel_sequence_soak():
    # The persistent kernels restart their work queues, rings and barriers on
    # every launch.  This runs the fp32 wide path (tiny), the bf16 and fp16
    # head_dim-128 kernels (dilated_s2048), the head_dim-256 wide kernels
    # and the global mask's split lines back to back, twelve times over.
    # Every repeat must reproduce the first results bit for bit: each output
    # tile has one writer, split lines merge in chunk order and nothing
    # accumulates by atomics, so the results do not depend on the schedule.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    cases = []
    for name, dtype in (("tiny", None), ("dilated_s2048", None), ("dilated_s2048", "f16")):
        wl = inputs.WORKLOADS[name]
        bm = wl.block_mask()
        if dtype is None:
            host = wl.inputs(seed=1)
        else:
            host = inputs.make_qkvdo(wl.batch, wl.heads, wl.seq, wl.head_dim, dtype, 1.0, 1)
        rp, ci = inputs.bsr_from_block_mask(bm)
        cases.append((bsr.Structure(rp, ci, bm.shape[0], dev), *(t.to(dev) for t in host), wl.scale))
    for kind, nb, D, heads in (("local", 6, 256, 2), ("global", 20, 128, 4)):
        bm = inputs.block_mask(kind, nb, radius=1)
        host = inputs.make_qkvdo(1, heads, nb * 128, D, "bf16", 1.0, 2)
        rp, ci = inputs.bsr_from_block_mask(bm)
        cases.append((bsr.Structure(rp, ci, nb, dev), *(t.to(dev) for t in host), 1.0 / np.sqrt(D)))
    first = [_fwd_bwd_on_device(c) for c in cases]
    bsr.bsr_attn_check()
    for _ in range(11):
        for c, ref in zip(cases, first):
            got = _fwd_bwd_on_device(c)
            bsr.bsr_attn_check()
            for name, a, b in zip(("O", "row_max", "row_denom", "dQ", "dK", "dV"), got, ref):
                assert torch.equal(a, b), name


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_device_index_check_reports_error(dtype):
    # A column index outside the grid is skipped by the kernels' own bounds
    # check and reported through bsr_attn_check.  The operands are views of
    # 1024-row buffers, so even a read of block column 7 would stay inside
    # the allocation.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    buf = torch.randn(1, 1, 1024, 64, device=dev).to(dtype)
    q = buf[:, :, :256]
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


def test_bounded_wait_gives_up_and_reports_timeout():
    # With the wait limit lowered to 100 ns the kernels' pipeline waits
    # expire: each CTA raises its abort flag, drains its copies and MMAs,
    # frees its tensor memory and returns, and bsr_attn_check reports
    # BSR_ERR_TIMEOUT.  Afterwards, with the default limit back, the same
    # calls give the oracle's results (the context is intact).
    import block_sparse_attention_bsr_gb300 as bsr

    bm = inputs.block_mask("global", 16, radius=2)
    Q, K, V, dO = inputs.make_qkvdo(1, 4, 16 * 128, 128, "bf16", 1.0, 13)
    scale = 1.0 / np.sqrt(128)
    timed_out = 0
    bsr.set_wait_limit(100)
    try:
        for _ in range(3):
            try:
                run_gpu(Q, K, V, dO, bm, scale)
            except bsr.BsrError as e:
                assert e.status == 4, str(e)
                timed_out += 1
    finally:
        bsr.set_wait_limit(0)
    assert timed_out > 0
    bsr.bsr_attn_check()  # nothing left over
    got = run_gpu(Q, K, V, dO, bm, scale)
    heads = [(0, h) for h in range(4)]
    compare(got, oracle_heads(Q, K, V, dO, bm, scale, heads), "bf16", heads=heads)


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


def _wrapper_inputs(dtype="bf16", D=128, api="plan"):
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    bm = inputs.block_mask("local", 8, radius=2)
    Q, K, V, dO = inputs.make_qkvdo(1, 2, 8 * 128, D, dtype, 1.0, 21)
    direct = run_gpu(Q, K, V, dO, bm, 1.0 / np.sqrt(D), api=api)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, bm.shape[1], dev)
    return Q, K, V, dO, st, direct, dev


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("bf16", 256)])
def test_autograd_wrapper_matches_direct_calls(dtype, D):
    # block_sparse_attention (the planned custom-op pair with its registered
    # autograd formula, on the structure's plan) gives the plan entry points'
    # outputs and gradients bit for bit; the per-call pair torch.ops.bsr.
    # bsr_attn / bsr_attn_bwd gives the per-call entry points' bit for bit.
    import block_sparse_attention_bsr_gb300 as bsr

    Q, K, V, dO, st, direct, dev = _wrapper_inputs(dtype, D)
    q, k, v = (t.to(dev).requires_grad_() for t in (Q, K, V))
    O, rm, rd = bsr.block_sparse_attention(q, k, v, st, return_stats=True)
    O.backward(dO.to(dev))
    got = dict(O=O.detach(), row_max=rm, row_denom=rd, dQ=q.grad, dK=k.grad, dV=v.grad)
    for name, t in got.items():
        assert np.array_equal(t.double().cpu().numpy(), direct[name]), name

    direct = run_gpu(Q, K, V, dO, inputs.block_mask("local", 8, radius=2), 1.0 / np.sqrt(D), api="per-call")
    ops = bsr.register_ops()
    q, k, v = (t.to(dev).requires_grad_() for t in (Q, K, V))
    O, rm, rd = ops.bsr_attn(q, k, v, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, 1.0 / float(np.sqrt(D)))
    O.backward(dO.to(dev))
    got = dict(O=O.detach(), row_max=rm, row_denom=rd, dQ=q.grad, dK=k.grad, dV=v.grad)
    for name, t in got.items():
        assert np.array_equal(t.double().cpu().numpy(), direct[name]), ("per-call ops", name)


def test_custom_op_pair_under_torch_compile_fullgraph():
    # torch.compile traces block_sparse_attention as torch.ops.bsr.bsr_attn
    # and its registered backward, single ops (fullgraph: no graph break);
    # the compiled forward and backward (aot_eager backend: no generated
    # kernels) match the per-call entry points bit for bit.
    import block_sparse_attention_bsr_gb300 as bsr

    Q, K, V, dO, st, direct, dev = _wrapper_inputs(api="per-call")

    def f(q, k, v):
        return bsr.block_sparse_attention(q, k, v, st, return_stats=True)

    cf = torch.compile(f, fullgraph=True, backend="aot_eager")
    q, k, v = (t.to(dev).requires_grad_() for t in (Q, K, V))
    O, rm, rd = cf(q, k, v)
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


# ------------------------------------------------------------ reusable plans --

@pytest.mark.parametrize("dtype,D,nb,H", [("bf16", 128, 20, 3), ("f16", 64, 9, 2), ("f32", 64, 6, 2),
                                          ("f32", 128, 20, 2), ("bf16", 256, 20, 2), ("bf16", 512, 4, 1)])
def test_plan_calls_match_unplanned_calls_repeatedly(dtype, D, nb, H):
    # Forward and backward on one plan, three times in a row (after each
    # launch the kernels put the plan's work-queue counter back to the grid
    # size and its other counters back to 0), give the same results every
    # time, and the per-call entry points' results bit for bit -- except dQ,
    # which the plan sums from the dS tiles of the dK/dV (or dK) walk (the
    # per-call walk recomputes dS), and the wide kernels' dV, summed from the
    # P^T tiles of the dK walk (for fp32 with the piece products in another
    # order): those are held to the oracle.  nb = 20 has block row 0 and column 0 long
    # enough to be split into chunks.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    bm = inputs.block_mask("global", nb, radius=1)
    Q, K, V, dO = inputs.make_qkvdo(1, H, nb * 128, D, dtype, 1.0, 17)
    scale = 1.0 / np.sqrt(D)
    ref = run_gpu(Q, K, V, dO, bm, scale)
    streamed = {"dQ"} | ({"dV"} if dtype == "f32" or D > 128 else set())
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, nb, dev)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    plan = st.plan(q)
    first = None
    for _ in range(3):
        O = torch.empty_like(q)
        rm = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
        rd = torch.empty_like(rm)
        dQ, dK, dV = (torch.full_like(q, float("nan")) for _ in range(3))
        bsr.bsr_attn_fwd_plan(plan, q, k, v, scale, O, rm, rd)
        bsr.bsr_attn_bwd_plan(plan, q, k, v, O, do, rm, rd, scale, dQ, dK, dV)
        bsr.bsr_attn_check()
        got = {n: t.double().cpu().numpy() for n, t in dict(O=O, row_max=rm, row_denom=rd, dQ=dQ, dK=dK,
                                                               dV=dV).items()}
        for name, t in got.items():
            if name not in streamed:
                assert np.array_equal(t, ref[name]), name
        if first is None:
            first = got
        for name, t in got.items():
            assert np.array_equal(t, first[name]), ("repeat", name)
    heads = [(0, h) for h in range(H)]
    ref_o = oracle_heads(Q, K, V, dO, bm, scale, heads)
    compare({n: first[n] for n in streamed}, {n: ref_o[n] for n in streamed}, dtype, heads=heads,
            what="plan, streamed walks")


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_plan_with_empty_lines(dtype, D):
    # A plan over a mask with empty block rows and columns: the planned calls
    # write the empty lines' outputs (they are not in the plan's work lists)
    # into NaN-filled outputs and match the per-call entry points bit for bit
    # (dQ, summed from the stored dS tiles on a plan: the empty rows exactly,
    # the rest against the oracle).
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    nb, H = 12, 3
    bm = np.zeros((nb, nb), bool)
    bm[0:3, 0:5] = True
    bm[7, 7] = True
    Q, K, V, dO = inputs.make_qkvdo(1, H, nb * 128, D, dtype, 1.0, 23)
    scale = 1.0 / np.sqrt(D)
    ref = run_gpu(Q, K, V, dO, bm, scale)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, nb, dev)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    plan = st.plan(q)
    for _ in range(2):
        O = torch.full_like(q, float("nan"))
        rm = torch.full(q.shape[:3], float("nan"), device=dev, dtype=torch.float32)
        rd = torch.full_like(rm, float("nan"))
        dQ, dK, dV = (torch.full_like(q, float("nan")) for _ in range(3))
        bsr.bsr_attn_fwd_plan(plan, q, k, v, scale, O, rm, rd)
        bsr.bsr_attn_bwd_plan(plan, q, k, v, O, do, rm, rd, scale, dQ, dK, dV)
        bsr.bsr_attn_check()
        got = dict(O=O, row_max=rm, row_denom=rd, dQ=dQ, dK=dK, dV=dV)
        for name, t in got.items():
            if name == "dQ" or (name == "dV" and dtype == "f32"):
                g = t.double().cpu().numpy()
                empty = np.repeat((bm.sum(1) if name == "dQ" else bm.sum(0)) == 0, 128)
                assert np.all(g[:, :, empty] == 0), f"{name} of empty lines"
                heads = [(0, h) for h in range(H)]
                compare({name: g}, {name: oracle_heads(Q, K, V, dO, bm, scale, heads)[name]}, dtype, heads=heads,
                        what=f"plan {name}")
                continue
            assert np.array_equal(t.double().cpu().numpy(), ref[name]), name


def test_plan_refuses_other_shapes():
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    bm = inputs.block_mask("local", 4, radius=1)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, 4, dev)
    q = torch.zeros(1, 2, 512, 64, device=dev, dtype=torch.bfloat16)
    plan = bsr.Plan(st, 1, 1, 64, torch.bfloat16)  # one head, operands have two
    O = torch.empty_like(q)
    rm = torch.empty(q.shape[:3], device=dev)
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_fwd_plan(plan, q, q, q, 0.125, O, rm, rm.clone())
    assert e.value.status == 1 and "plan" in str(e.value)
    plan.close()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_plan_refuses_a_bsc_view_of_other_blocks(dtype):
    # The plan maps every BSC entry to its BSR position (where the dK/dV or
    # dK walk stores that block's dS tile for the dQ walk); a row_idx naming
    # a block that the BSR lists do not store is refused at creation, on the
    # host, before any kernel reads the map.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    bm = inputs.block_mask("local", 6, radius=1)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, 6, dev)
    ri = st.host["row_idx"].copy()
    ri[0] = 5  # column 0 holds rows 0 and 1; block (5, 0) is not stored
    st.dev["row_idx"] = torch.from_numpy(ri).to(dev)
    with pytest.raises(bsr.BsrError) as e:
        bsr.Plan(st, 1, 1, 64, dtype)
    assert e.value.status == 1 and "BSC entry 0" in str(e.value)


@pytest.mark.parametrize("api", ["plan", "per-call"])
def test_step_captured_in_a_cuda_graph(api):
    # One forward + backward captured in a CUDA graph (stream capture through
    # torch.cuda.graph) and replayed on new inputs copied into the captured
    # buffers gives the eager calls' results bit for bit: the calls launch on
    # the caller's stream, fork and join their second stream with events,
    # and (per call) allocate their scratch stream-ordered, all of which
    # capture records.
    import block_sparse_attention_bsr_gb300 as bsr

    dev = torch.device("cuda")
    nb, H, D = 20, 3, 128
    bm = inputs.block_mask("global", nb, radius=1)
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, nb, dev)
    scale = 1.0 / np.sqrt(D)
    bufs = [t.to(dev) for t in inputs.make_qkvdo(1, H, nb * 128, D, "bf16", 1.0, 70)]
    q, k, v, do = bufs
    O = torch.empty_like(q)
    rm = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    rd = torch.empty_like(rm)
    dQ, dK, dV = (torch.empty_like(q) for _ in range(3))
    plan = st.plan(q) if api == "plan" else None

    def step():
        if plan is not None:
            bsr.bsr_attn_fwd_plan(plan, q, k, v, scale, O, rm, rd)
            bsr.bsr_attn_bwd_plan(plan, q, k, v, O, do, rm, rd, scale, dQ, dK, dV)
        else:
            bsr.bsr_attn_fwd(q, k, v, st.row_ptr, st.col_idx, st.n_brows, 128, scale, O, rm, rd)
            bsr.bsr_attn_bwd(q, k, v, O, do, rm, rd, st.row_ptr, st.col_idx, st.col_ptr, st.row_idx, scale,
                             dQ, dK, dV)

    step()  # first calls outside capture (kernel attributes, the second stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (71, 72):
        new = [t.to(dev) for t in inputs.make_qkvdo(1, H, nb * 128, D, "bf16", 1.0, seed)]
        for dst, src in zip(bufs, new):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        bsr.bsr_attn_check()
        replayed = [t.clone() for t in (O, rm, rd, dQ, dK, dV)]
        step()
        torch.cuda.synchronize()
        bsr.bsr_attn_check()
        for name, a, b in zip(("O", "row_max", "row_denom", "dQ", "dK", "dV"), replayed, (O, rm, rd, dQ, dK, dV)):
            assert torch.equal(a, b), (api, seed, name)
