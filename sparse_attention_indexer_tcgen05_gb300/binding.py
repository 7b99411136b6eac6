"""Thin PyTorch binding of libcsa_indexer.so (ctypes).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.  PyTorch supplies
device memory (outputs and workspace) and the current stream.  The functions keep the C ABI's names:

    csa_indexer_fwd(params, q_idx, w, k_idx)                        -> (ids, selscore)
    csa_teacher(params, q, kv, kv_c, sink, ids)                     -> teacher
    csa_teacher_from_lse(params, q, kv_c, lse_nc, ids)              -> teacher
    csa_indexer_bwd(params, q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore[, teacher])
                                                                    -> (loss, dq_idx, dw, dk_idx)
    csa_scores_debug(params, q_idx, w, k_idx, row_begin, row_count) -> scores

and ``CSAIndexerLoss`` wraps the step as an autograd function (forward returns ids and the loss; backward
returns the stored indexer gradients scaled by the incoming gradient).

Importing this module loads the library and raises ImportError if it has not been built: there is no
fallback implementation.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa_indexer.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -m sparse_attention_indexer_tcgen05_gb300.build` (or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

SBHD, BSHD, THD = 0, 1, 2
F32, BF16 = 0, 1
LAYOUTS = {"sbhd": SBHD, "bshd": BSHD, "thd": THD}
DTYPES = {"f32": F32, "bf16": BF16, torch.float32: F32, torch.bfloat16: BF16}
TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}

STATUS = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARG", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_ALIGNMENT",
          4: "CSA_ERR_WORKSPACE", 5: "CSA_ERR_CUDA", 6: "CSA_ERR_TIMEOUT"}


# csa_teacher_mode: the full-CSA teacher, or the compressed-only one the issue reports (A/B control)
TEACHER_MODES = {"full": 0, "compressed_only": 1}


class csa_params(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int32), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("seqlen", ctypes.c_int32), ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_q_unpadded", ctypes.c_void_p),
        ("max_seqlen_q", ctypes.c_int32), ("key_rows", ctypes.c_int32), ("compress_ratio", ctypes.c_int32),
        ("window", ctypes.c_int32), ("topk", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float), ("sparse_loss", ctypes.c_int32), ("reduction", ctypes.c_int32),
        ("loss_coeff", ctypes.c_float), ("teacher_mode", ctypes.c_int32),
        ("require_tensor_cores", ctypes.c_int32),
    ]


_P = ctypes.POINTER(csa_params)
_vp, _sz, _i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
for _name, _args, _res in [
    ("csa_topk_width", [_P], ctypes.c_int32),
    ("csa_key_width", [_P], ctypes.c_int32),
    ("csa_teacher_width", [_P], ctypes.c_int32),
    ("csa_rows", [_P], ctypes.c_int64),
    ("csa_compressed_rows", [_P], ctypes.c_int64),
    ("csa_workspace_size", [_P], ctypes.c_size_t),
    ("csa_indexer_fwd", [_P, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    ("csa_teacher", [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    ("csa_teacher_from_lse", [_P, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    ("csa_indexer_bwd", [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                         _vp],
     ctypes.c_int),
    ("csa_scores_debug", [_P, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _sz, _vp], ctypes.c_int),
    ("csa_indexer_bwd_noalloc", [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
     ctypes.c_int),
    ("csa_check_device_status", [_vp], ctypes.c_int),
    ("csa_selftest_bounded_wait", [_vp], ctypes.c_int),
    ("csa_last_timeout_site", [], ctypes.c_int32),
    ("csa_last_path", [], ctypes.c_char_p),
    ("csa_last_cuda_error", [], ctypes.c_char_p),
    ("csa_kernel_launches", [], ctypes.c_uint64),
    ("csa_status_string", [ctypes.c_int], ctypes.c_char_p),
]:
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = ("csa_topk_width", "csa_key_width", "csa_teacher_width", "csa_rows", "csa_compressed_rows",
            "csa_workspace_size", "csa_indexer_fwd", "csa_teacher", "csa_teacher_from_lse", "csa_indexer_bwd",
            "csa_scores_debug",
            "csa_indexer_bwd_noalloc",
            "csa_check_device_status", "csa_selftest_bounded_wait", "csa_last_timeout_site", "csa_last_path",
            "csa_last_cuda_error",
            "csa_kernel_launches",
            "csa_status_string")


class CSAError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = _lib.csa_status_string(status).decode()
        if status == 5:  # CSA_ERR_CUDA
            msg += " (" + _lib.csa_last_cuda_error().decode() + ")"
        if status == 6:  # CSA_ERR_TIMEOUT
            msg += f" (kernel {_lib.csa_last_timeout_site() // 100}, wait site {_lib.csa_last_timeout_site() % 100})"
        super().__init__(f"{call}: {msg}")


def _check(status: int, call: str):
    if status != 0:
        raise CSAError(status, call)


class Params:
    """Geometry and flags of one step (the C struct csa_params plus references to its cu_seqlens tensors).

    For THD, ``cu_seqlens_q`` / ``cu_seqlens_q_unpadded`` are int32 CUDA tensors, ``batch`` is the number of
    segments, ``seqlen`` the physical rows, ``max_seqlen_q`` the longest unpadded segment (host int) and
    ``key_rows`` the rows of k_idx / kv_c.
    """

    def __init__(self, layout, dtype, batch, seqlen, compress_ratio, window, topk, heads, head_dim, idx_heads,
                 idx_dim, softmax_scale, sparse_loss=True, reduction="mean", loss_coeff=1.0, cu_seqlens_q=None,
                 cu_seqlens_q_unpadded=None, max_seqlen_q=0, key_rows=0, teacher_mode="full",
                 require_tensor_cores=False):
        self.cu = cu_seqlens_q
        self.cur = cu_seqlens_q_unpadded
        for t in (self.cu, self.cur):
            if t is not None and (t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous()):
                raise ValueError("cu_seqlens tensors must be contiguous int32 CUDA tensors")
        lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
        if lay == THD and self.cu is not None:
            batch = self.cu.numel() - 1
        self.c = csa_params(lay, DTYPES[dtype] if not isinstance(dtype, int) else dtype, int(batch), int(seqlen),
                            self.cu.data_ptr() if self.cu is not None else None,
                            self.cur.data_ptr() if self.cur is not None else None, int(max_seqlen_q), int(key_rows),
                            int(compress_ratio), int(window), int(topk), int(heads), int(head_dim), int(idx_heads),
                            int(idx_dim), float(softmax_scale), 1 if sparse_loss else 0,
                            0 if reduction in ("mean", 0) else 1, float(loss_coeff),
                            TEACHER_MODES[teacher_mode] if isinstance(teacher_mode, str) else int(teacher_mode),
                            1 if require_tensor_cores else 0)

    @property
    def ref(self):
        return ctypes.byref(self.c)

    @property
    def K(self) -> int:
        return _lib.csa_topk_width(self.ref)

    @property
    def key_width(self) -> int:
        return _lib.csa_key_width(self.ref)

    @property
    def teacher_width(self) -> int:
        return _lib.csa_teacher_width(self.ref)

    @property
    def rows(self) -> int:
        return _lib.csa_rows(self.ref)

    @property
    def compressed_rows(self) -> int:
        return _lib.csa_compressed_rows(self.ref)

    @property
    def workspace_bytes(self) -> int:
        return _lib.csa_workspace_size(self.ref)

    @property
    def value_dtype(self) -> torch.dtype:
        return TORCH_DTYPE[self.c.dtype]


def csa_topk_width(p: Params) -> int:
    return p.K


def csa_workspace_size(p: Params) -> int:
    return p.workspace_bytes


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_tensor(t, name, dtype, device, numel=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def _workspace(p: Params, device, workspace):
    n = p.workspace_bytes
    if workspace is None:
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=device)
    return workspace, workspace.numel()


@contextlib.contextmanager
def _nvtx(name):
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


def csa_indexer_fwd(p: Params, q_idx, w, k_idx, workspace=None, ids=None, selscore=None):
    """Steps 1-2: scores + top-k.  Returns (ids [rows, K] int32, selscore [rows, K] fp32)."""
    dev = q_idx.device
    rows, K, HI, DI = p.rows, p.K, p.c.idx_heads, p.c.idx_dim
    _check_tensor(q_idx, "q_idx", p.value_dtype, dev, rows * HI * DI)
    _check_tensor(w, "w", torch.float32, dev, rows * HI)
    _check_tensor(k_idx, "k_idx", p.value_dtype, dev, p.compressed_rows * DI)
    if ids is None:
        ids = torch.empty((rows, K), dtype=torch.int32, device=dev)
    if selscore is None:
        selscore = torch.empty((rows, K), dtype=torch.float32, device=dev)
    ws, nws = _workspace(p, dev, workspace)
    with _nvtx("csa_indexer_fwd"):
        st = _lib.csa_indexer_fwd(p.ref, _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(ids), _ptr(selscore), _ptr(ws), nws,
                                  _stream(dev))
    _check(st, "csa_indexer_fwd")
    return ids, selscore


def csa_teacher(p: Params, q, kv, kv_c, sink, ids, workspace=None, out=None):
    """Step 3: full-CSA teacher for the given ids.  Returns teacher [rows, teacher_width] fp32."""
    dev = q.device
    rows, H, D = p.rows, p.c.heads, p.c.head_dim
    _check_tensor(q, "q", p.value_dtype, dev, rows * H * D)
    _check_tensor(kv, "kv", p.value_dtype, dev, rows * D)
    _check_tensor(kv_c, "kv_c", p.value_dtype, dev, p.compressed_rows * D)
    _check_tensor(sink, "sink", torch.float32, dev, H)
    _check_tensor(ids, "ids", torch.int32, dev, rows * p.K)
    if out is None:
        out = torch.empty((rows, p.teacher_width), dtype=torch.float32, device=dev)
    ws, nws = _workspace(p, dev, workspace)
    with _nvtx("csa_teacher"):
        st = _lib.csa_teacher(p.ref, _ptr(q), _ptr(kv), _ptr(kv_c), _ptr(sink), _ptr(ids), _ptr(out), _ptr(ws), nws,
                              _stream(dev))
    _check(st, "csa_teacher")
    return out


def csa_teacher_from_lse(p: Params, q, kv_c, lse_nc, ids, workspace=None, out=None):
    """Step 3 from a given non-compressed log-sum-exp lse_nc [rows, heads] fp32 (natural log of exp(sink) plus
    the window's exponentials, per row and head).  Returns teacher [rows, teacher_width] fp32."""
    dev = q.device
    rows, H, D = p.rows, p.c.heads, p.c.head_dim
    _check_tensor(q, "q", p.value_dtype, dev, rows * H * D)
    _check_tensor(kv_c, "kv_c", p.value_dtype, dev, p.compressed_rows * D)
    _check_tensor(lse_nc, "lse_nc", torch.float32, dev, rows * H)
    _check_tensor(ids, "ids", torch.int32, dev, rows * p.K)
    if out is None:
        out = torch.empty((rows, p.teacher_width), dtype=torch.float32, device=dev)
    ws, nws = _workspace(p, dev, workspace)
    with _nvtx("csa_teacher_from_lse"):
        st = _lib.csa_teacher_from_lse(p.ref, _ptr(q), _ptr(kv_c), _ptr(lse_nc), _ptr(ids), _ptr(out), _ptr(ws), nws,
                                       _stream(dev))
    _check(st, "csa_teacher_from_lse")
    return out


def csa_indexer_bwd(p: Params, q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore, teacher=None, workspace=None,
                    out=None, row_loss=None):
    """Steps 3-5: teacher (unless given), KL and indexer gradients.
    Returns (loss [] fp32, dq_idx like q_idx, dw like w, dk_idx like k_idx).  If row_loss (a [rows] fp32 tensor)
    is given, it receives the unscaled per-row KL."""
    dev = q_idx.device
    rows, K, HI, DI = p.rows, p.K, p.c.idx_heads, p.c.idx_dim
    _check_tensor(q_idx, "q_idx", p.value_dtype, dev, rows * HI * DI)
    _check_tensor(w, "w", torch.float32, dev, rows * HI)
    _check_tensor(k_idx, "k_idx", p.value_dtype, dev, p.compressed_rows * DI)
    _check_tensor(ids, "ids", torch.int32, dev, rows * K)
    _check_tensor(selscore, "selscore", torch.float32, dev, rows * K)
    if teacher is None:
        H, D = p.c.heads, p.c.head_dim
        _check_tensor(q, "q", p.value_dtype, dev, rows * H * D)
        _check_tensor(kv, "kv", p.value_dtype, dev, rows * D)
        _check_tensor(kv_c, "kv_c", p.value_dtype, dev, p.compressed_rows * D)
        _check_tensor(sink, "sink", torch.float32, dev, H)
    else:
        _check_tensor(teacher, "teacher", torch.float32, dev, rows * p.teacher_width)
    if out is None:
        out = (torch.empty((), dtype=torch.float32, device=dev), torch.empty_like(q_idx), torch.empty_like(w),
               torch.empty_like(k_idx))
    loss, dq, dw, dk = out
    if row_loss is not None:
        _check_tensor(row_loss, "row_loss", torch.float32, dev, rows)
    ws, nws = _workspace(p, dev, workspace)
    with _nvtx("csa_indexer_bwd"):
        st = _lib.csa_indexer_bwd(p.ref, _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(q), _ptr(kv), _ptr(kv_c), _ptr(sink),
                                  _ptr(ids), _ptr(selscore), _ptr(teacher), _ptr(loss), _ptr(row_loss), _ptr(dq),
                                  _ptr(dw), _ptr(dk), _ptr(ws), nws, _stream(dev))
    _check(st, "csa_indexer_bwd")
    return loss, dq, dw, dk


NOALLOC_SCRATCH_BYTES = 64 << 20


def csa_indexer_bwd_noalloc(p: Params, q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore, teacher=None, out=None,
                            row_loss=None):
    """csa_indexer_bwd without a workspace, for callers that cannot allocate device memory: the library uses
    its own fixed 64 MiB device scratch (shared by every call on a device; serialise overlapping calls).
    Returns (loss, dq_idx, dw, dk_idx); raises CSAError (CSA_ERR_WORKSPACE) if the problem needs more scratch."""
    dev = q_idx.device
    rows = p.rows
    if out is None:
        out = (torch.empty((), dtype=torch.float32, device=dev), torch.empty_like(q_idx), torch.empty_like(w),
               torch.empty_like(k_idx))
    loss, dq, dw, dk = out
    with _nvtx("csa_indexer_bwd_noalloc"):
        st = _lib.csa_indexer_bwd_noalloc(p.ref, _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(q), _ptr(kv), _ptr(kv_c),
                                          _ptr(sink), _ptr(ids), _ptr(selscore), _ptr(teacher), _ptr(loss),
                                          _ptr(row_loss), _ptr(dq), _ptr(dw), _ptr(dk), _stream(dev))
    _check(st, "csa_indexer_bwd_noalloc")
    return loss, dq, dw, dk


def csa_scores_debug(p: Params, q_idx, w, k_idx, row_begin=0, row_count=None, workspace=None):
    """Test aid: the fp32 scores the forward selects from, [row_count, key_width] (-inf where not visible)."""
    dev = q_idx.device
    if row_count is None:
        row_count = p.rows - row_begin
    out = torch.empty((row_count, p.key_width), dtype=torch.float32, device=dev)
    ws, nws = _workspace(p, dev, workspace)
    st = _lib.csa_scores_debug(p.ref, _ptr(q_idx), _ptr(w), _ptr(k_idx), int(row_begin), int(row_count), _ptr(out),
                               _ptr(ws), nws, _stream(dev))
    _check(st, "csa_scores_debug")
    return out


def csa_check_device_status(device=None):
    st = _lib.csa_check_device_status(_stream(device) if torch.cuda.is_available() else None)
    _check(st, "csa_check_device_status")


def csa_last_path() -> str:
    return _lib.csa_last_path().decode()


def csa_last_timeout_site() -> int:
    """100 x kernel + wait site of the last timeout csa_check_device_status reported (0 before any)."""
    return int(_lib.csa_last_timeout_site())


def csa_last_cuda_error() -> str:
    return _lib.csa_last_cuda_error().decode()


def csa_kernel_launches() -> int:
    return int(_lib.csa_kernel_launches())


class CSAIndexerLoss(torch.autograd.Function):
    """ids, loss = CSAIndexerLoss.apply(q_idx, w, k_idx, q, kv, kv_c, sink, params).

    The forward runs the whole step (scores + top-k, teacher, KL, gradients) and keeps only the three
    indexer gradients for the backward, so no score graph is ever retained.  Gradients flow to q_idx,
    w and k_idx only; q, kv, kv_c and sink receive none (they are the detached teacher side)."""

    @staticmethod
    def forward(ctx, q_idx, w, k_idx, q, kv, kv_c, sink, params):
        ids, sel = csa_indexer_fwd(params, q_idx.contiguous(), w.contiguous(), k_idx.contiguous())
        loss, dq, dw, dk = csa_indexer_bwd(params, q_idx.contiguous(), w.contiguous(), k_idx.contiguous(),
                                           q.contiguous(), kv.contiguous(), kv_c.contiguous(), sink.contiguous(),
                                           ids, sel)
        ctx.save_for_backward(dq, dw, dk)
        ctx.mark_non_differentiable(ids)
        return ids, loss

    @staticmethod
    def backward(ctx, _gid, gloss):
        dq, dw, dk = ctx.saved_tensors
        return (dq * gloss.to(dq.dtype), dw * gloss, dk * gloss.to(dk.dtype), None, None, None, None, None)


def csa_indexer_loss(q_idx, w, k_idx, q, kv, kv_c, sink, params: Params):
    return CSAIndexerLoss.apply(q_idx, w, k_idx, q, kv, kv_c, sink, params)
