"""Block-sparse attention over BSR-128 block masks on GB300 (sm_103a).

A thin ctypes binding over the C-ABI library ``libbsrattn.so`` (declared in
``include/bsr_attn.h``).  The functions below only marshal arguments: torch
tensors become bsr_tensor descriptors and device pointers, the current torch
stream becomes the ``stream`` argument, and a non-OK status raises
``BsrError``.  Every step of the computation runs in the library's CUDA
kernels; if the library is missing, calls fail loudly (there is no fallback).
"""

from __future__ import annotations

import ctypes
import os
import weakref

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbsrattn.so")

BSR_F32, BSR_BF16, BSR_F16 = 0, 1, 2
STATUS_NAMES = {0: "BSR_OK", 1: "BSR_ERR_INVALID_ARG", 2: "BSR_ERR_UNSUPPORTED", 3: "BSR_ERR_CUDA",
                4: "BSR_ERR_TIMEOUT", 5: "BSR_ERR_DEVICE_CHECK"}

# Every symbol include/bsr_attn.h declares.
EXPORTS = ("bsr_attn_fwd", "bsr_attn_fwd_two_pass", "bsr_spmm", "bsr_screened_spmm", "bsr_attn_bwd",
           "bsr_attn_bwd_noalloc", "bsr_plan_create", "bsr_plan_destroy", "bsr_plan_work_list", "bsr_attn_fwd_plan",
           "bsr_attn_bwd_plan",
           "bsr_build_bsc", "bsr_validate", "bsr_attn_check", "bsr_set_wait_limit", "bsr_last_error",
           "bsr_profile_enable", "bsr_profile_collect")


class BsrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class bsr_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("seq", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class bsr_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_float)]


_lib_handle = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libbsrattn.so and declares its prototypes (raises if it was not built)."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(block_sparse_attention_bsr_gb300/_build.py); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    P, I32, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    T = ctypes.POINTER(bsr_tensor)
    lib.bsr_attn_fwd.argtypes = [T, T, T, P, P, I32, I32, F32, T, P, P, P]
    lib.bsr_attn_fwd_two_pass.argtypes = [T, T, T, P, P, I32, I32, F32, T, P, P, P]
    lib.bsr_spmm.argtypes = [P, I32, P, P, I32, I32, I32, I32, P, I32, P, P]
    lib.bsr_screened_spmm.argtypes = [P, P, P, I32, I32, I32, F32, P, P]
    lib.bsr_attn_bwd.argtypes = [T, T, T, T, T, P, P, P, P, P, P, F32, T, T, T, P]
    lib.bsr_attn_bwd_noalloc.argtypes = [T, T, T, T, T, P, P, P, P, P, P, F32, T, T, T, P]
    lib.bsr_plan_create.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, P, ctypes.POINTER(ctypes.c_void_p)]
    lib.bsr_plan_destroy.argtypes = [P]
    lib.bsr_plan_work_list.argtypes = [P, I32, P, I32, P, P]
    lib.bsr_attn_fwd_plan.argtypes = [P, T, T, T, F32, T, P, P, P]
    lib.bsr_attn_bwd_plan.argtypes = [P, T, T, T, T, T, P, P, F32, T, T, T, P]
    lib.bsr_build_bsc.argtypes = [P, P, I32, I32, P, P]
    lib.bsr_validate.argtypes = [P, P, I32, I32]
    lib.bsr_attn_check.argtypes = [P]
    lib.bsr_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.bsr_last_error.argtypes = []
    lib.bsr_last_error.restype = ctypes.c_char_p
    lib.bsr_profile_enable.argtypes = [I32]
    lib.bsr_profile_enable.restype = None
    lib.bsr_profile_collect.argtypes = [ctypes.POINTER(bsr_kernel_time), I32]
    lib.bsr_profile_collect.restype = I32
    for name in ("bsr_attn_fwd", "bsr_attn_fwd_two_pass", "bsr_spmm", "bsr_screened_spmm", "bsr_attn_bwd",
                 "bsr_attn_bwd_noalloc", "bsr_plan_create", "bsr_plan_destroy", "bsr_attn_fwd_plan",
                 "bsr_attn_bwd_plan", "bsr_build_bsc", "bsr_validate", "bsr_attn_check", "bsr_set_wait_limit"):
        getattr(lib, name).restype = I32
    _lib_handle = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        msg = load_library().bsr_last_error().decode(errors="replace")
        raise BsrError(status, msg)


def _desc(t) -> bsr_tensor:
    import torch

    if t.dtype == torch.float32:
        dt = BSR_F32
    elif t.dtype == torch.bfloat16:
        dt = BSR_BF16
    elif t.dtype == torch.float16:
        dt = BSR_F16
    else:
        raise TypeError(f"unsupported dtype {t.dtype} (float32, bfloat16 or float16)")
    if t.dim() != 4 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError("dense operands must be contiguous CUDA tensors [batch, heads, seq, head_dim]")
    b, h, s, d = t.shape
    return bsr_tensor(t.data_ptr(), dt, b, h, s, d)


def _dev_ptr(t, dtype_name: str) -> int:
    if not t.is_cuda or not t.is_contiguous() or str(t.dtype) != dtype_name:
        raise ValueError(f"expected a contiguous CUDA {dtype_name} tensor, got {t.dtype} on {t.device}")
    return t.data_ptr()


def _stream(stream, like) -> int:
    import torch

    if stream is None:
        return torch.cuda.current_stream(like.device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def bsr_attn_fwd(Q, K, V, row_ptr, col_idx, n_brows: int, block: int, scale: float, O, row_max, row_denom,
                 stream=None, two_pass: bool = False) -> None:
    """Forward block-sparse attention: writes O, row_max, row_denom (see include/bsr_attn.h).

    ``two_pass`` selects the statistics-first variant (bsr_attn_fwd_two_pass)."""
    lib = load_library()
    q, k, v, o = (_desc(t) for t in (Q, K, V, O))
    fn = lib.bsr_attn_fwd_two_pass if two_pass else lib.bsr_attn_fwd
    _check(fn(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                            _dev_ptr(row_ptr, "torch.int32"), _dev_ptr(col_idx, "torch.int32"),
                            int(n_brows), int(block), float(scale), ctypes.byref(o),
                            _dev_ptr(row_max, "torch.float32"), _dev_ptr(row_denom, "torch.float32"),
                            _stream(stream, Q)))


def bsr_spmm(blocks, row_ptr, col_idx, n_brows: int, n_bcols: int, X, Y, stream=None) -> None:
    """Y = A X for the BSR matrix A of 128 x 128 blocks and a dense X (see include/bsr_attn.h).

    blocks: [nnzb, 128, 128] bf16 / fp16 CUDA tensor (the stored blocks in BSR
    order); X: [n_bcols * 128, n_cols] and Y: [n_brows * 128, n_cols] of the
    same dtype; row_ptr / col_idx int32 CUDA tensors.
    """
    import torch

    codes = {torch.bfloat16: BSR_BF16, torch.float16: BSR_F16}
    if blocks.dtype not in codes:
        raise TypeError(f"unsupported dtype {blocks.dtype} (bfloat16 or float16)")
    for name, t in (("blocks", blocks), ("X", X), ("Y", Y)):
        if t.dtype != blocks.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor of dtype {blocks.dtype}")
    if blocks.dim() != 3 or tuple(blocks.shape[1:]) != (128, 128) or X.dim() != 2 or Y.dim() != 2:
        raise ValueError("blocks must be [nnzb, 128, 128], X and Y two-dimensional")
    if X.shape[0] != n_bcols * 128 or Y.shape[0] != n_brows * 128 or X.shape[1] != Y.shape[1]:
        raise ValueError("X must be [n_bcols * 128, n_cols] and Y [n_brows * 128, n_cols]")
    lib = load_library()
    _check(lib.bsr_spmm(blocks.data_ptr(), codes[blocks.dtype], _dev_ptr(row_ptr, "torch.int32"),
                        _dev_ptr(col_idx, "torch.int32"), int(n_brows), int(n_bcols), int(blocks.shape[0]), 128,
                        X.data_ptr(), int(X.shape[1]), Y.data_ptr(), _stream(stream, X)))


def bsr_screened_spmm(A, diag, B, threshold: float, C, stream=None) -> None:
    """C = (A o M) B with M[i, j] = sqrt|diag_i| sqrt|diag_j| > sqrt(threshold) (see include/bsr_attn.h).

    A: [n, n], B and C: [n, n_cols] bf16 / fp16 CUDA tensors; diag: fp32 CUDA tensor [n].
    """
    import torch

    codes = {torch.bfloat16: BSR_BF16, torch.float16: BSR_F16}
    if A.dtype not in codes:
        raise TypeError(f"unsupported dtype {A.dtype} (bfloat16 or float16)")
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dtype != A.dtype or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous two-dimensional CUDA tensor of dtype {A.dtype}")
    n = A.shape[0]
    if A.shape[1] != n or B.shape[0] != n or tuple(C.shape) != tuple(B.shape) or tuple(diag.shape) != (n,):
        raise ValueError("A must be [n, n], B and C [n, n_cols], diag [n]")
    lib = load_library()
    _check(lib.bsr_screened_spmm(A.data_ptr(), _dev_ptr(diag, "torch.float32"), B.data_ptr(), codes[A.dtype], int(n),
                                 int(B.shape[1]), float(threshold), C.data_ptr(), _stream(stream, A)))


def bsr_attn_bwd(Q, K, V, O, dO, row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx, scale: float,
                 dQ, dK, dV, stream=None) -> None:
    """Backward block-sparse attention: writes dQ, dK, dV (see include/bsr_attn.h)."""
    lib = load_library()
    q, k, v, o, do, dq, dk, dv = (_desc(t) for t in (Q, K, V, O, dO, dQ, dK, dV))
    i32 = "torch.int32"
    _check(lib.bsr_attn_bwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(o), ctypes.byref(do),
                            _dev_ptr(row_max, "torch.float32"), _dev_ptr(row_denom, "torch.float32"),
                            _dev_ptr(row_ptr, i32), _dev_ptr(col_idx, i32), _dev_ptr(col_ptr, i32),
                            _dev_ptr(row_idx, i32), float(scale),
                            ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), _stream(stream, Q)))


def bsr_attn_bwd_noalloc(Q, K, V, O, dO, row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx, scale: float,
                         dQ, dK, dV, stream=None) -> None:
    """Backward pass that allocates no device memory (static scratch; see include/bsr_attn.h).

    For callers that cannot allocate: another allocator owns the device
    memory, or the hot path must not call the CUDA allocator.  Limited to
    batch * heads * seq <= 1,048,576 (9 MiB of static device memory);
    calls that overlap on the GPU race.
    """
    lib = load_library()
    q, k, v, o, do, dq, dk, dv = (_desc(t) for t in (Q, K, V, O, dO, dQ, dK, dV))
    i32 = "torch.int32"
    _check(lib.bsr_attn_bwd_noalloc(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(o),
                                    ctypes.byref(do), _dev_ptr(row_max, "torch.float32"),
                                    _dev_ptr(row_denom, "torch.float32"), _dev_ptr(row_ptr, i32),
                                    _dev_ptr(col_idx, i32), _dev_ptr(col_ptr, i32), _dev_ptr(row_idx, i32),
                                    float(scale), ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                    _stream(stream, Q)))


# Live plans by handle (weak: a plan lives as long as its owner holds it);
# the planned custom ops carry only the handle.
_PLANS = weakref.WeakValueDictionary()


def _plan_of(handle: int) -> "Plan":
    p = _PLANS.get(int(handle))
    if p is None:
        raise ValueError(f"no live plan with handle {handle:#x}")
    return p


class Plan:
    """A reusable plan (bsr_plan_create): the work lists and scratch of one block mask for operands of
    shape [batch, heads, n_brows * 128, head_dim] and one dtype.  Freed with bsr_plan_destroy when
    the object is collected (or by close())."""

    _CODES = None

    def __init__(self, structure: "Structure", batch: int, heads: int, head_dim: int, dtype, stream=None):
        import torch

        codes = {torch.float32: BSR_F32, torch.bfloat16: BSR_BF16, torch.float16: BSR_F16}
        if dtype not in codes:
            raise TypeError(f"unsupported dtype {dtype} (float32, bfloat16 or float16)")
        lib = load_library()
        h = ctypes.c_void_p()
        s = torch.cuda.current_stream(structure.row_ptr.device).cuda_stream if stream is None else _stream(stream, None)
        _check(lib.bsr_plan_create(structure.row_ptr.data_ptr(), structure.col_idx.data_ptr(),
                                   structure.col_ptr.data_ptr(), structure.row_idx.data_ptr(), structure.n_brows,
                                   int(batch), int(heads), int(head_dim), codes[dtype], s, ctypes.byref(h)))
        self.handle = h.value
        self.key = (int(batch), int(heads), int(head_dim), dtype)
        _PLANS[self.handle] = self

    def work_list(self, which: int = 0, stream=None):
        """One of the plan's work lists (bsr_plan_work_list): an int32 array [items, 4] of
        (line, first, n, slot) in the order the kernels draw them, and a dict with the item count, the
        persistent CTAs G, the heads the planner counts and the number of distinct item lengths."""
        import numpy as np
        import torch

        lib = load_library()
        info = np.zeros(4, dtype=np.int32)
        cap = 1 << 16
        items = np.zeros((cap, 4), dtype=np.int32)
        s = torch.cuda.current_stream().cuda_stream if stream is None else _stream(stream, None)
        _check(lib.bsr_plan_work_list(self.handle, int(which), items.ctypes.data, cap, info.ctypes.data, s))
        n = int(info[0])
        return items[:n].copy(), {"items": n, "G": int(info[1]), "heads": int(info[2]), "buckets": int(info[3])}

    def close(self) -> None:
        if getattr(self, "handle", None):
            if _PLANS.get(self.handle) is self:
                del _PLANS[self.handle]
            load_library().bsr_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown
            pass


def bsr_attn_fwd_plan(plan: Plan, Q, K, V, scale: float, O, row_max, row_denom, stream=None) -> None:
    """Forward pass on a reusable plan (bsr_attn_fwd_plan in include/bsr_attn.h)."""
    lib = load_library()
    q, k, v, o = (_desc(t) for t in (Q, K, V, O))
    _check(lib.bsr_attn_fwd_plan(plan.handle, ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), float(scale),
                                 ctypes.byref(o), _dev_ptr(row_max, "torch.float32"),
                                 _dev_ptr(row_denom, "torch.float32"), _stream(stream, Q)))


def bsr_attn_bwd_plan(plan: Plan, Q, K, V, O, dO, row_max, row_denom, scale: float, dQ, dK, dV,
                      stream=None) -> None:
    """Backward pass on a reusable plan (bsr_attn_bwd_plan in include/bsr_attn.h)."""
    lib = load_library()
    q, k, v, o, do, dq, dk, dv = (_desc(t) for t in (Q, K, V, O, dO, dQ, dK, dV))
    _check(lib.bsr_attn_bwd_plan(plan.handle, ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(o),
                                 ctypes.byref(do), _dev_ptr(row_max, "torch.float32"),
                                 _dev_ptr(row_denom, "torch.float32"), float(scale), ctypes.byref(dq),
                                 ctypes.byref(dk), ctypes.byref(dv), _stream(stream, Q)))


def _host_i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def bsr_validate(row_ptr_h, col_idx_h, n_brows: int, n_bcols: int) -> None:
    """Checks host BSR lists; raises BsrError with the library's message if they are malformed."""
    rp, ci = _host_i32(row_ptr_h), _host_i32(col_idx_h)
    if len(rp) != n_brows + 1:
        raise BsrError(1, f"row_ptr has {len(rp)} entries, expected n_brows + 1 = {n_brows + 1}")
    _check(load_library().bsr_validate(rp.ctypes.data, ci.ctypes.data if ci.size else None, n_brows, n_bcols))


def bsr_build_bsc(row_ptr_h, col_idx_h, n_brows: int, n_bcols: int):
    """Host BSC transpose: returns (col_ptr int32 [n_bcols+1], row_idx int32 [nnzb])."""
    rp, ci = _host_i32(row_ptr_h), _host_i32(col_idx_h)
    if len(rp) != n_brows + 1:
        raise BsrError(1, f"row_ptr has {len(rp)} entries, expected n_brows + 1 = {n_brows + 1}")
    nnzb = int(rp[-1]) if len(rp) else 0
    col_ptr = np.zeros(n_bcols + 1, dtype=np.int32)
    row_idx = np.zeros(max(nnzb, 1), dtype=np.int32)
    _check(load_library().bsr_build_bsc(rp.ctypes.data, ci.ctypes.data if ci.size else None, n_brows, n_bcols,
                                        col_ptr.ctypes.data, row_idx.ctypes.data))
    return col_ptr, row_idx[:nnzb]


def bsr_attn_check(stream=None) -> None:
    """Synchronises the stream and raises if a kernel reported a timeout or a failed index check."""
    import torch

    s = torch.cuda.current_stream().cuda_stream if stream is None else _stream(stream, None)
    _check(load_library().bsr_attn_check(s))


def set_wait_limit(ns: int = 0) -> None:
    """Limit of the kernels' bounded device-side waits in ns (0: the default 2 s); see include/bsr_attn.h."""
    _check(load_library().bsr_set_wait_limit(int(ns)))


def profile_enable(on: bool = True) -> None:
    load_library().bsr_profile_enable(1 if on else 0)


def profile_collect() -> dict:
    """{kernel name: (launches, total ms)} since the last collect (events on the launching stream)."""
    buf = (bsr_kernel_time * 64)()
    n = load_library().bsr_profile_collect(buf, 64)
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n)}


class Structure:
    """Device copies of one BSR block mask and its BSC transpose (built by bsr_build_bsc)."""

    def __init__(self, row_ptr_h, col_idx_h, n_bcols: int, device):
        import torch

        rp, ci = _host_i32(row_ptr_h), _host_i32(col_idx_h)
        self.n_brows = len(rp) - 1
        self.n_bcols = n_bcols
        bsr_validate(rp, ci, self.n_brows, n_bcols)
        cp, ri = bsr_build_bsc(rp, ci, self.n_brows, n_bcols)
        self.host = dict(row_ptr=rp, col_idx=ci, col_ptr=cp, row_idx=ri)
        # an empty index array still gets one element so its device pointer is valid
        self.dev = {k: torch.from_numpy(v if v.size else np.zeros(1, np.int32)).to(device)
                    for k, v in self.host.items()}
        self.nnzb = int(rp[-1])
        self._plans = {}

    def plan(self, Q) -> "Plan":
        """The reusable plan of this mask for operands shaped and typed like Q (built on first use)."""
        b, h, s, d = Q.shape
        if s != self.n_brows * 128:
            raise ValueError(f"seq {s} does not match the mask's {self.n_brows} block rows")
        key = (b, h, d, Q.dtype)
        if key not in self._plans:
            self._plans[key] = Plan(self, b, h, d, Q.dtype)
        return self._plans[key]

    @property
    def row_ptr(self):
        return self.dev["row_ptr"]

    @property
    def col_idx(self):
        return self.dev["col_idx"]

    @property
    def col_ptr(self):
        return self.dev["col_ptr"]

    @property
    def row_idx(self):
        return self.dev["row_idx"]


_OPS = None


def register_ops():
    """Registers the custom-op pair torch.ops.bsr.bsr_attn / torch.ops.bsr.bsr_attn_bwd (once) and returns
    the torch.ops.bsr namespace.

    bsr_attn(Q, K, V, row_ptr, col_idx, col_ptr, row_idx, scale) -> (O, row_max, row_denom) runs
    bsr_attn_fwd; bsr_attn_bwd(Q, K, V, O, dO, row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx,
    scale) -> (dQ, dK, dV) runs bsr_attn_bwd.  The forward carries the BSC lists (col_ptr, row_idx) only so
    that its registered autograd formula can hand them to the backward op.  Both have fake (meta)
    implementations, so graph tracing (torch.compile, torch.export) sees each as one opaque op; the pages
    register their kernels the same way, as a custom-op pair with register_autograd ("trnsparse 0.7.0 ->
    0.9.0" diff, CHANGELOG [0.8.0]).
    """
    global _OPS
    if _OPS is not None:
        return _OPS
    import torch

    # explicit schemas: this module's annotations are strings (postponed evaluation)
    @torch.library.custom_op("bsr::bsr_attn", mutates_args=(),
                             schema="(Tensor Q, Tensor K, Tensor V, Tensor row_ptr, Tensor col_idx, Tensor col_ptr, "
                                    "Tensor row_idx, float scale) -> (Tensor, Tensor, Tensor)")
    def _fwd(Q, K, V, row_ptr, col_idx, col_ptr, row_idx, scale):
        O = torch.empty_like(Q)
        rm = torch.empty(Q.shape[:3], device=Q.device, dtype=torch.float32)
        rd = torch.empty_like(rm)
        bsr_attn_fwd(Q, K, V, row_ptr, col_idx, Q.shape[2] // 128, 128, scale, O, rm, rd)
        return O, rm, rd

    @_fwd.register_fake
    def _fwd_fake(Q, K, V, row_ptr, col_idx, col_ptr, row_idx, scale):
        rm = Q.new_empty(Q.shape[:3], dtype=torch.float32)
        return torch.empty_like(Q), rm, torch.empty_like(rm)

    @torch.library.custom_op("bsr::bsr_attn_bwd", mutates_args=(),
                             schema="(Tensor Q, Tensor K, Tensor V, Tensor O, Tensor dO, Tensor row_max, "
                                    "Tensor row_denom, Tensor row_ptr, Tensor col_idx, Tensor col_ptr, "
                                    "Tensor row_idx, float scale) -> (Tensor, Tensor, Tensor)")
    def _bwd(Q, K, V, O, dO, row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx, scale):
        dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))
        bsr_attn_bwd(Q, K, V, O, dO.contiguous(), row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx, scale,
                     dQ, dK, dV)
        return dQ, dK, dV

    @_bwd.register_fake
    def _bwd_fake(Q, K, V, O, dO, row_max, row_denom, row_ptr, col_idx, col_ptr, row_idx, scale):
        return torch.empty_like(Q), torch.empty_like(Q), torch.empty_like(Q)

    def _setup_context(ctx, inputs, output):
        Q, K, V, row_ptr, col_idx, col_ptr, row_idx, scale = inputs
        O, rm, rd = output
        ctx.save_for_backward(Q, K, V, O, rm, rd, row_ptr, col_idx, col_ptr, row_idx)
        ctx.scale = scale
        ctx.mark_non_differentiable(rm, rd)

    def _backward(ctx, dO, _drm, _drd):
        Q, K, V, O, rm, rd, row_ptr, col_idx, col_ptr, row_idx = ctx.saved_tensors
        dQ, dK, dV = torch.ops.bsr.bsr_attn_bwd(Q, K, V, O, dO.contiguous(), rm, rd, row_ptr, col_idx, col_ptr,
                                                row_idx, ctx.scale)
        return dQ, dK, dV, None, None, None, None, None

    _fwd.register_autograd(_backward, setup_context=_setup_context)

    # The same pair on a reusable plan (bsr_attn_fwd_plan / bsr_attn_bwd_plan),
    # the plan passed as its handle: block_sparse_attention runs these with the
    # plan its Structure keeps for the operands' shape.  The autograd context
    # holds the plan itself, so it outlives the forward until the backward ran.
    @torch.library.custom_op("bsr::bsr_attn_planned", mutates_args=(),
                             schema="(Tensor Q, Tensor K, Tensor V, int plan, float scale) -> (Tensor, Tensor, Tensor)")
    def _pfwd(Q, K, V, plan, scale):
        O = torch.empty_like(Q)
        rm = torch.empty(Q.shape[:3], device=Q.device, dtype=torch.float32)
        rd = torch.empty_like(rm)
        bsr_attn_fwd_plan(_plan_of(plan), Q, K, V, scale, O, rm, rd)
        return O, rm, rd

    @_pfwd.register_fake
    def _pfwd_fake(Q, K, V, plan, scale):
        rm = Q.new_empty(Q.shape[:3], dtype=torch.float32)
        return torch.empty_like(Q), rm, torch.empty_like(rm)

    @torch.library.custom_op("bsr::bsr_attn_planned_bwd", mutates_args=(),
                             schema="(Tensor Q, Tensor K, Tensor V, Tensor O, Tensor dO, Tensor row_max, "
                                    "Tensor row_denom, int plan, float scale) -> (Tensor, Tensor, Tensor)")
    def _pbwd(Q, K, V, O, dO, row_max, row_denom, plan, scale):
        dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))
        bsr_attn_bwd_plan(_plan_of(plan), Q, K, V, O, dO.contiguous(), row_max, row_denom, scale, dQ, dK, dV)
        return dQ, dK, dV

    @_pbwd.register_fake
    def _pbwd_fake(Q, K, V, O, dO, row_max, row_denom, plan, scale):
        return torch.empty_like(Q), torch.empty_like(Q), torch.empty_like(Q)

    def _psetup_context(ctx, inputs, output):
        Q, K, V, plan, scale = inputs
        O, rm, rd = output
        ctx.save_for_backward(Q, K, V, O, rm, rd)
        ctx.plan = plan
        ctx.plan_obj = _PLANS.get(plan)
        ctx.scale = scale
        ctx.mark_non_differentiable(rm, rd)

    def _pbackward(ctx, dO, _drm, _drd):
        Q, K, V, O, rm, rd = ctx.saved_tensors
        dQ, dK, dV = torch.ops.bsr.bsr_attn_planned_bwd(Q, K, V, O, dO.contiguous(), rm, rd, ctx.plan, ctx.scale)
        return dQ, dK, dV, None, None

    _pfwd.register_autograd(_pbackward, setup_context=_psetup_context)
    _OPS = torch.ops.bsr
    return _OPS


def block_sparse_attention(Q, K, V, structure: "Structure", scale=None, return_stats: bool = False):
    """softmax(scale * Q K^T over the stored 128 x 128 blocks) V, differentiable in Q, K and V.

    Q, K, V: contiguous CUDA tensors [batch, heads, seq, head_dim] (bf16, fp16 or
    fp32, 16-byte aligned); `structure`: a Structure of the block mask on the same
    device; scale defaults to 1 / sqrt(head_dim).  Runs the custom op
    torch.ops.bsr.bsr_attn_planned (bsr_attn_fwd_plan on the current stream, on
    the plan the structure keeps for Q's shape and dtype, built on first use)
    with its registered backward torch.ops.bsr.bsr_attn_planned_bwd
    (bsr_attn_bwd_plan).  While torch.compile traces it, it runs the per-call
    pair torch.ops.bsr.bsr_attn / bsr_attn_bwd instead (building a plan is a
    host-side library call the tracer cannot take into a graph).  With
    return_stats the fp32 row_max / row_denom statistics come back as well
    (they carry no gradient).
    """
    import torch

    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if not getattr(t, "is_cuda", False):
            raise ValueError(f"{name} must be a CUDA tensor")
    if scale is None:
        scale = 1.0 / float(Q.shape[-1]) ** 0.5
    ops = register_ops()
    if torch.compiler.is_compiling():
        O, rm, rd = ops.bsr_attn(Q, K, V, structure.row_ptr, structure.col_idx, structure.col_ptr,
                                 structure.row_idx, float(scale))
    else:
        O, rm, rd = ops.bsr_attn_planned(Q, K, V, structure.plan(Q).handle, float(scale))
    return (O, rm, rd) if return_stats else O
