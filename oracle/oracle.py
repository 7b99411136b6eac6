"""Python front of the float64 oracle (``csa_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's CPU
baseline leg, never by the library.  It marshals numpy arrays into the C oracle and back;
every step of the method is computed in the C file.

The oracle takes the same tensor layouts as the library (SBHD, BSHD, THD) as float64 copies of
the exact input values, and its own parameter block (it shares nothing with the CUDA side).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

LAYOUTS = {"sbhd": 0, "bshd": 1, "thd": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (float64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int), ("batch", ctypes.c_int), ("seqlen", ctypes.c_int),
        ("cu_q", ctypes.c_void_p), ("cu_q_real", ctypes.c_void_p), ("max_seqlen", ctypes.c_int),
        ("ratio", ctypes.c_int), ("window", ctypes.c_int), ("topk", ctypes.c_int),
        ("heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("idx_heads", ctypes.c_int),
        ("idx_dim", ctypes.c_int), ("scale", ctypes.c_double), ("sparse", ctypes.c_int),
        ("reduction", ctypes.c_int), ("coeff", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Params)
            vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.orc_key_width.argtypes = [P]
            lib.orc_topk_width.argtypes = [P]
            lib.orc_rows.argtypes = [P]
            lib.orc_teacher_width.argtypes = [P]
            lib.orc_scores.argtypes = [P, vp, vp, vp, vp, i32, i32, vp]
            lib.orc_topk.argtypes = [P, vp, vp, i32, vp]
            lib.orc_teacher.argtypes = [P, vp, vp, vp, vp, vp, vp, i32, i32, vp]
            lib.orc_noncompressed_lse.argtypes = [P, vp, vp, vp, vp, i32, i32, vp]
            lib.orc_teacher_lse.argtypes = [P, vp, vp, vp, vp, vp, i32, i32, vp]
            lib.orc_attention.argtypes = [P, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp]
            lib.orc_kl_row.argtypes = [vp, vp, i32, vp, vp]
            lib.orc_kl_row.restype = dbl
            lib.orc_loss_factor.argtypes = [P]
            lib.orc_loss_factor.restype = dbl
            lib.orc_loss_grads.argtypes = [P, vp, vp, vp, vp, vp, vp, i32, i32, ctypes.c_long, vp, vp, vp, vp]
            lib.orc_loss_grads.restype = dbl
            lib.orc_num_threads.restype = i32
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Problem:
    """One step's geometry and flags, in the oracle's own terms.

    layout: "sbhd" | "bshd" | "thd"; for THD, batch is the number of segments and seqlen the
    number of physical rows, and cu_seqlens_q / cu_seqlens_q_unpadded give the segments.
    """

    def __init__(self, layout, batch, seqlen, ratio, window, topk, heads, head_dim, idx_heads, idx_dim,
                 scale, sparse=True, reduction="mean", coeff=1.0, cu_seqlens_q=None,
                 cu_seqlens_q_unpadded=None, max_seqlen_q=0):
        self.layout = layout
        self.cu = None if cu_seqlens_q is None else np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        self.cur = None if cu_seqlens_q_unpadded is None else np.ascontiguousarray(cu_seqlens_q_unpadded,
                                                                                   dtype=np.int32)
        if layout == "thd":
            batch = len(self.cu) - 1
            seqlen = int(self.cu[-1])
        self.p = _Params(LAYOUTS[layout], int(batch), int(seqlen), _ptr(self.cu), _ptr(self.cur),
                         int(max_seqlen_q), int(ratio), int(window), int(topk), int(heads), int(head_dim),
                         int(idx_heads), int(idx_dim), float(scale), 1 if sparse else 0,
                         0 if reduction == "mean" else 1, float(coeff))
        self.lib = _load()

    @classmethod
    def from_inputs(cls, inp, **over):
        c = inp.cfg
        kw = dict(layout=c.layout, batch=c.batch, seqlen=c.seqlen, ratio=c.ratio, window=c.window,
                  topk=c.topk, heads=c.heads, head_dim=c.head_dim, idx_heads=c.idx_heads, idx_dim=c.idx_dim,
                  scale=c.scale, sparse=c.sparse, reduction=c.reduction, coeff=c.coeff,
                  cu_seqlens_q=inp.cu_seqlens_q, cu_seqlens_q_unpadded=inp.cu_seqlens_q_unpadded,
                  max_seqlen_q=inp.max_seqlen_q)
        kw.update(over)
        return cls(**kw)

    # geometry -----------------------------------------------------------
    @property
    def key_width(self) -> int:
        return self.lib.orc_key_width(ctypes.byref(self.p))

    @property
    def K(self) -> int:
        return self.lib.orc_topk_width(ctypes.byref(self.p))

    @property
    def rows(self) -> int:
        return self.lib.orc_rows(ctypes.byref(self.p))

    @property
    def teacher_width(self) -> int:
        return self.lib.orc_teacher_width(ctypes.byref(self.p))

    @property
    def loss_factor(self) -> float:
        return self.lib.orc_loss_factor(ctypes.byref(self.p))

    def _rows(self, rows):
        if rows is None:
            rows = np.arange(self.rows, dtype=np.int32)
        return np.ascontiguousarray(rows, dtype=np.int32)

    # steps --------------------------------------------------------------
    def scores(self, q_idx, w, k_idx, rows=None, compact=False) -> np.ndarray:
        """Dense float64 indexer scores [len(rows), key_width]; -inf where not visible.
        compact=True: q_idx and w hold only the listed rows, in list order."""
        rows = self._rows(rows)
        qi, ww, ki = _f64(q_idx), _f64(w), _f64(k_idx)
        out = np.empty((len(rows), self.key_width), np.float64)
        self.lib.orc_scores(ctypes.byref(self.p), _ptr(qi), _ptr(ww), _ptr(ki), _ptr(rows), len(rows), int(compact),
                            _ptr(out))
        return out

    def topk(self, scores, rows=None) -> np.ndarray:
        """Top-k ids [len(rows), K] (ascending ids, -1 pads) from given dense scores."""
        rows = self._rows(rows)
        sc = _f64(scores)
        assert sc.shape == (len(rows), self.key_width)
        ids = np.empty((len(rows), self.K), np.int32)
        self.lib.orc_topk(ctypes.byref(self.p), _ptr(sc), _ptr(rows), len(rows), _ptr(ids))
        return ids

    def teacher(self, q, kv, kv_c, sink, ids, rows=None, compact=False) -> np.ndarray:
        """Full-CSA teacher [len(rows), teacher_width] for the given ids of those rows.
        compact=True: q holds only the listed rows, in list order."""
        rows = self._rows(rows)
        qq, kvv, kc, sk = _f64(q), _f64(kv), _f64(kv_c), _f64(sink)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        assert ids.shape == (len(rows), self.K)
        out = np.empty((len(rows), self.teacher_width), np.float64)
        self.lib.orc_teacher(ctypes.byref(self.p), _ptr(qq), _ptr(kvv), _ptr(kc), _ptr(sk), _ptr(ids), _ptr(rows),
                             len(rows), int(compact), _ptr(out))
        return out

    def noncompressed_lse(self, q, kv, sink, rows=None, compact=False) -> np.ndarray:
        """u [len(rows), heads]: log(exp(a_h) + sum over the window of exp(sigma q.kv)) per row and head."""
        rows = self._rows(rows)
        qq, kvv, sk = _f64(q), _f64(kv), _f64(sink)
        out = np.empty((len(rows), self.p.heads), np.float64)
        self.lib.orc_noncompressed_lse(ctypes.byref(self.p), _ptr(qq), _ptr(kvv), _ptr(sk), _ptr(rows), len(rows),
                                       int(compact), _ptr(out))
        return out

    def teacher_from_lse(self, q, kv_c, lse, ids, rows=None, compact=False) -> np.ndarray:
        """The teacher [len(rows), teacher_width] from a given non-compressed log-sum-exp lse [len(rows), heads]."""
        rows = self._rows(rows)
        qq, kc, ls = _f64(q), _f64(kv_c), _f64(lse)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        assert ids.shape == (len(rows), self.K) and ls.shape == (len(rows), self.p.heads)
        out = np.empty((len(rows), self.teacher_width), np.float64)
        self.lib.orc_teacher_lse(ctypes.byref(self.p), _ptr(qq), _ptr(kc), _ptr(ls), _ptr(ids), _ptr(rows),
                                 len(rows), int(compact), _ptr(out))
        return out

    def attention(self, q, kv, kv_c, sink, ids, rows=None, compact=False):
        """The CSA sparse attention forward of the listed rows: (O [len(rows), heads, head_dim], lse [len(rows),
        heads]) over the sink, the window rows and the selected compressed rows (keys and values alike)."""
        rows = self._rows(rows)
        qq, kvv, kc, sk = _f64(q), _f64(kv), _f64(kv_c), _f64(sink)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        assert ids.shape == (len(rows), self.K)
        out = np.empty((len(rows), self.p.heads, self.p.head_dim), np.float64)
        lse = np.empty((len(rows), self.p.heads), np.float64)
        self.lib.orc_attention(ctypes.byref(self.p), _ptr(qq), _ptr(kvv), _ptr(kc), _ptr(sk), _ptr(ids), _ptr(rows),
                               len(rows), int(compact), _ptr(out), _ptr(lse))
        return out, lse

    def loss_grads(self, q_idx, w, k_idx, ids, teacher, rows=None, want_dk=True, compact=False):
        """(loss, loss_rows, dq[rows,HI,DI], dw[rows,HI], dk[key rows, DI] or None) for the listed rows.
        compact=True: q_idx and w hold only the listed rows, in list order."""
        rows = self._rows(rows)
        qi, ww, ki = _f64(q_idx), _f64(w), _f64(k_idx)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        te = _f64(teacher)
        HI, DI = self.p.idx_heads, self.p.idx_dim
        n_key_rows = ki.size // DI
        lr = np.empty(len(rows), np.float64)
        dq = np.empty((len(rows), HI, DI), np.float64)
        dw = np.empty((len(rows), HI), np.float64)
        dk = np.zeros((n_key_rows, DI), np.float64) if want_dk else None
        loss = self.lib.orc_loss_grads(ctypes.byref(self.p), _ptr(qi), _ptr(ww), _ptr(ki), _ptr(ids), _ptr(te),
                                       _ptr(rows), len(rows), int(compact), n_key_rows, _ptr(lr), _ptr(dq), _ptr(dw),
                                       _ptr(dk))
        return loss, lr, dq, dw, dk

    def step(self, inp, rows=None, want_dk=True):
        """Whole step on the listed rows (all rows by default): scores, ids, teacher, loss and gradients,
        all from the oracle's own float64 selection.  With a row list, only those rows of the row-dependent
        inputs are widened to float64 (compact mode)."""
        if rows is None:
            rows = self._rows(None)
            qi, ww, qq = inp.q_idx.values, inp.w.values, inp.q.values
            compact = False
        else:
            rows = self._rows(rows)
            qi, ww, qq = inp.q_idx.rows_f32(rows), inp.w.rows_f32(rows), inp.q.rows_f32(rows)
            compact = True
        sc = self.scores(qi, ww, inp.k_idx.values, rows, compact=compact)
        ids = self.topk(sc, rows)
        te = self.teacher(qq, inp.kv.values, inp.kv_c.values, inp.sink.values, ids, rows, compact=compact)
        loss, lr, dq, dw, dk = self.loss_grads(qi, ww, inp.k_idx.values, ids, te, rows, want_dk=want_dk,
                                               compact=compact)
        return dict(scores=sc, ids=ids, teacher=te, loss=loss, loss_rows=lr, dq=dq, dw=dw, dk=dk, rows=rows)


def kl_row(t, I, want_grad=True):
    """KL(t || softmax(I)) of one row and its derivative w.r.t. I (the oracle's step 4)."""
    lib = _load()
    t = _f64(t)
    I = _f64(I)
    g = np.empty_like(I) if want_grad else None
    p = np.empty_like(I)
    L = lib.orc_kl_row(_ptr(t), _ptr(I), len(I), _ptr(g), _ptr(p))
    return L, g, p


def num_threads() -> int:
    return _load().orc_num_threads()
