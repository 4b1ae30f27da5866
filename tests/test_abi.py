"""C-ABI library checks that need no GPU: exports, host structure helpers, argument errors."""

import ctypes
import os
import re

import numpy as np
import pytest

import block_sparse_attention_bsr_gb300 as bsr
import oracle
from block_sparse_attention_bsr_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bsr.LIB_PATH):
        from block_sparse_attention_bsr_gb300 import _build

        _build.build()
    return bsr.load_library()


def _declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(bsr_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"bsr_attn_fwd", "bsr_attn_bwd", "bsr_build_bsc", "bsr_validate"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(bsr.EXPORTS) == declared


@pytest.mark.parametrize("kind,p", [("local", 0), ("dilated", 0), ("global", 0), ("random", 0.2), ("random", 0.6),
                                    ("full", 0), ("diag", 0)])
def test_build_bsc_matches_oracle_transpose(lib, kind, p):
    bm = inputs.block_mask(kind, 23, radius=3, p=p)
    rp, ci = inputs.bsr_from_block_mask(bm)
    cp, ri = bsr.bsr_build_bsc(rp, ci, 23, 23)
    ocp, ori = oracle.bsc_from_block_mask(bm)
    assert np.array_equal(cp, ocp) and np.array_equal(ri, ori)


def test_build_bsc_empty_structure(lib):
    rp = np.zeros(5, np.int32)
    cp, ri = bsr.bsr_build_bsc(rp, np.zeros(0, np.int32), 4, 4)
    assert np.array_equal(cp, np.zeros(5)) and ri.size == 0


@pytest.mark.parametrize("rp,ci,msg", [
    ([1, 2], [0, 0], "row_ptr\\[0\\]"),
    ([0, 2, 1], [0, 1], "decreases"),
    ([0, 2], [1, 1], "ascending"),
    ([0, 2], [1, 0], "ascending"),
    ([0, 1], [4], "outside"),
    ([0, 1], [-1], "outside"),
])
def test_validate_rejects_malformed(lib, rp, ci, msg):
    nb = len(rp) - 1
    with pytest.raises(bsr.BsrError, match=msg) as e:
        bsr.bsr_validate(np.array(rp), np.array(ci), nb, 4)
    assert e.value.status == 1
    with pytest.raises(bsr.BsrError):
        bsr.bsr_build_bsc(np.array(rp), np.array(ci), nb, 4)


def _fake(dtype=0, b=1, h=1, s=256, d=64, ptr=0x1000):
    return bsr.bsr_tensor(ptr, dtype, b, h, s, d)


def _fwd(lib, Q=None, K=None, V=None, O=None, n_brows=2, block=128, scale=0.125, ptrs=(0x10, 0x20, 0x30, 0x40)):
    Q, K, V, O = (x if x is not None else _fake() for x in (Q, K, V, O))
    P = ctypes.c_void_p
    return lib.bsr_attn_fwd(ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V), P(ptrs[0]), P(ptrs[1]), n_brows,
                            block, scale, ctypes.byref(O), P(ptrs[2]), P(ptrs[3]), None)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(block=64), 2, "block"),
    (dict(Q=_fake(d=96)), 2, "head_dim"),
    (dict(Q=_fake(d=32)), 2, "head_dim"),
    (dict(K=_fake(dtype=1)), 2, "dtype"),
    (dict(V=_fake(dtype=7)), 2, "dtype"),
    (dict(Q=_fake(dtype=2), K=_fake(dtype=2), V=_fake(dtype=2)), 2, "dtype"),  # fp16 beside an fp32 O
    (dict(O=_fake(s=384)), 1, "shape"),
    (dict(Q=_fake(ptr=0)), 1, "null"),
    (dict(ptrs=(0, 0x20, 0x30, 0x40)), 1, "null"),
    (dict(ptrs=(0x10, 0x20, 0, 0x40)), 1, "null"),
    (dict(n_brows=3), 1, "n_brows"),
    (dict(Q=_fake(s=200), K=_fake(s=200), V=_fake(s=200), O=_fake(s=200)), 1, "multiple"),
    (dict(scale=float("nan")), 1, "scale"),
    (dict(O=_fake(ptr=0x1002)), 1, "aligned"),
    (dict(Q=_fake(ptr=0x1008)), 1, "aligned"),
])
def test_fwd_rejects_bad_arguments_on_host(lib, kw, status, msg):
    # Every case fails in the host checks, before any CUDA call.
    assert _fwd(lib, **kw) == status
    assert re.search(msg, lib.bsr_last_error().decode())


@pytest.mark.parametrize("kw", [dict(), dict(d=256)])
def test_two_pass_forward_refuses_unsupported_operands_on_host(lib, kw):
    # fp32 operands, or bf16 with head_dim 256: refused before any CUDA call
    dtype = 0 if not kw else 1
    Q, K, V, O = (_fake(dtype=dtype, **kw) for _ in range(4))
    P = ctypes.c_void_p
    st = lib.bsr_attn_fwd_two_pass(ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V), P(0x10), P(0x20), 2, 128,
                                   0.125, ctypes.byref(O), P(0x30), P(0x40), None)
    assert st == 2 and "two_pass" in lib.bsr_last_error().decode()


@pytest.mark.parametrize("kw,status,msg", [
    (dict(block=64), 2, "block"),
    (dict(dtype=0), 2, "dtype"),
    (dict(n_cols=96), 2, "multiple of 64"),
    (dict(n_cols=0), 1, "sizes"),
    (dict(X=0), 1, "null"),
    (dict(Y=0x1008), 1, "aligned"),
])
def test_spmm_rejects_bad_arguments_on_host(lib, kw, status, msg):
    a = dict(blocks=0x1000, dtype=1, row_ptr=0x10, col_idx=0x20, n_brows=2, n_bcols=2, nnzb=3, block=128,
             X=0x2000, n_cols=128, Y=0x3000)
    a.update(kw)
    P = ctypes.c_void_p
    st = lib.bsr_spmm(P(a["blocks"]), a["dtype"], P(a["row_ptr"]), P(a["col_idx"]), a["n_brows"], a["n_bcols"],
                      a["nnzb"], a["block"], P(a["X"]), a["n_cols"], P(a["Y"]), None)
    assert st == status
    assert re.search(msg, lib.bsr_last_error().decode())


@pytest.mark.parametrize("kw,status,msg", [
    (dict(dtype=0), 2, "dtype"),
    (dict(n=200), 2, "multiple of 128"),
    (dict(n_cols=96), 2, "multiple of 64"),
    (dict(threshold=-1.0), 1, "threshold"),
    (dict(threshold=float("nan")), 1, "threshold"),
    (dict(diag=0), 1, "null"),
    (dict(C=0x1008), 1, "aligned"),
])
def test_screened_spmm_rejects_bad_arguments_on_host(lib, kw, status, msg):
    a = dict(A=0x1000, diag=0x2000, B=0x3000, dtype=1, n=256, n_cols=128, threshold=1e-3, C=0x4000)
    a.update(kw)
    P = ctypes.c_void_p
    st = lib.bsr_screened_spmm(P(a["A"]), P(a["diag"]), P(a["B"]), a["dtype"], a["n"], a["n_cols"],
                               a["threshold"], P(a["C"]), None)
    assert st == status
    assert re.search(msg, lib.bsr_last_error().decode())


def test_bwd_rejects_bad_arguments_on_host(lib):
    t = [_fake() for _ in range(8)]
    t[4] = _fake(dtype=1)  # dO in bf16 beside fp32 operands
    P = ctypes.c_void_p
    st = lib.bsr_attn_bwd(*(ctypes.byref(x) for x in t[:5]), P(1), P(2), P(3), P(4), P(5), P(6), 0.125,
                          *(ctypes.byref(x) for x in t[5:]), None)
    assert st == 2 and "dO" in lib.bsr_last_error().decode()
    t[4] = _fake()
    st = lib.bsr_attn_bwd(*(ctypes.byref(x) for x in t[:5]), P(1), P(2), P(3), P(0), P(5), P(6), 0.125,
                          *(ctypes.byref(x) for x in t[5:]), None)
    assert st == 1


def test_autograd_wrapper_refuses_host_tensors():
    # The wrapper only marshals arguments: host tensors are refused before
    # anything reaches the library.
    torch = pytest.importorskip("torch")
    import block_sparse_attention_bsr_gb300 as bsr

    class _St:  # a structure stand-in: never dereferenced
        row_ptr = col_idx = col_ptr = row_idx = None
        n_brows = 2

    x = torch.zeros(1, 1, 256, 64)
    with pytest.raises(ValueError, match="CUDA"):
        bsr.block_sparse_attention(x, x, x, _St())
