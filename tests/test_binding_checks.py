"""The Python binding only marshals arguments: wrong shapes, dtypes or host
tensors are refused before anything reaches the library (no GPU needed)."""

import pytest

torch = pytest.importorskip("torch")

import block_sparse_attention_bsr_gb300 as bsr  # noqa: E402


def _spmm_args(**kw):
    a = dict(blocks=torch.zeros(2, 128, 128, dtype=torch.bfloat16), row_ptr=torch.zeros(3, dtype=torch.int32),
             col_idx=torch.zeros(2, dtype=torch.int32), n_brows=2, n_bcols=1,
             X=torch.zeros(128, 64, dtype=torch.bfloat16), Y=torch.zeros(256, 64, dtype=torch.bfloat16))
    a.update(kw)
    return a


def test_spmm_refuses_fp32_blocks():
    with pytest.raises(TypeError):
        bsr.bsr_spmm(**_spmm_args(blocks=torch.zeros(2, 128, 128)))


def test_spmm_refuses_host_tensors():
    with pytest.raises(ValueError):
        bsr.bsr_spmm(**_spmm_args())


def test_spmm_refuses_mixed_dtypes():
    with pytest.raises(ValueError):
        bsr.bsr_spmm(**_spmm_args(X=torch.zeros(128, 64, dtype=torch.float16)))


def test_screened_refuses_fp32_and_host_tensors():
    A = torch.zeros(256, 256)
    with pytest.raises(TypeError):
        bsr.bsr_screened_spmm(A, torch.ones(256), torch.zeros(256, 64), 1e-3, torch.zeros(256, 64))
    A = A.bfloat16()
    with pytest.raises(ValueError):
        bsr.bsr_screened_spmm(A, torch.ones(256), torch.zeros(256, 64, dtype=torch.bfloat16), 1e-3,
                              torch.zeros(256, 64, dtype=torch.bfloat16))


def test_forward_refuses_unsupported_dtype():
    q = torch.zeros(1, 1, 256, 64, dtype=torch.float64)
    with pytest.raises(TypeError):
        bsr.bsr_attn_fwd(q, q, q, None, None, 2, 128, 0.125, q, None, None)


def test_custom_op_pair_is_registered_with_fake_implementations():
    # torch.ops.bsr.bsr_attn / bsr_attn_bwd exist with their schemas, and
    # their fake implementations give the output shapes and dtypes graph
    # tracing needs (no kernel runs under FakeTensorMode).
    from torch._subclasses.fake_tensor import FakeTensorMode

    ops = bsr.register_ops()
    assert "float scale" in str(ops.bsr_attn.default._schema)
    assert "Tensor dO" in str(ops.bsr_attn_bwd.default._schema)
    with FakeTensorMode():
        q = torch.empty(2, 3, 256, 64, dtype=torch.bfloat16)
        i = torch.empty(3, dtype=torch.int32)
        O, rm, rd = ops.bsr_attn(q, q, q, i, i, i, i, 0.125)
        assert O.shape == q.shape and O.dtype == q.dtype
        assert rm.shape == (2, 3, 256) and rm.dtype == torch.float32 and rd.shape == rm.shape
        dq, dk, dv = ops.bsr_attn_bwd(q, q, q, O, O, rm, rd, i, i, i, i, 0.125)
        assert dq.shape == dk.shape == dv.shape == q.shape and dq.dtype == q.dtype
    # the planned pair (a plan handle instead of the structure tensors)
    assert "int plan" in str(ops.bsr_attn_planned.default._schema)
    assert "int plan" in str(ops.bsr_attn_planned_bwd.default._schema)
    with FakeTensorMode():
        q = torch.empty(2, 3, 256, 64, dtype=torch.float16)
        O, rm, rd = ops.bsr_attn_planned(q, q, q, 12345, 0.125)
        assert O.shape == q.shape and O.dtype == q.dtype and rm.shape == (2, 3, 256) and rd.dtype == torch.float32
        dq, dk, dv = ops.bsr_attn_planned_bwd(q, q, q, O, O, rm, rd, 12345, 0.125)
        assert dq.shape == dk.shape == dv.shape == q.shape and dv.dtype == q.dtype
