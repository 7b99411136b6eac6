"""Seeded synthetic inputs for the CSA Lightning-Indexer training step.

This module only draws random numbers and lays them out in the tensor layouts the
library accepts (SBHD, BSHD, THD).  It holds none of the method's arithmetic: no
score, mask, top-k, softmax or gradient is computed here.  Both the float64 oracle's
tests and the GPU path's tests and benchmark take their inputs from it, so the two
sides read the same bytes.

Recipe (one stream per tensor, so every tensor is reproducible on its own):
  * generator: numpy PCG64 seeded with SeedSequence([config_seed, tensor_id]);
  * q, kv, kv_c, q_idx, k_idx ~ N(0, 1) / sqrt(own last dim) (q, kv, kv_c optionally ~ N(0, qk_std^2),
    used with qk_std = 1 for a teacher-sensitivity input whose attention logits are of order one);
  * w ~ U(0, 1) (the indexer weights as passed, i.e. with the indexer softmax
    scale already folded in);
  * sink ~ N(sink_mean, sink_std^2), one logit per main-attention head (sink_mean = 0 except for the
    teacher-sensitivity input);
  * bf16 tensors are rounded from float32 on the host with round-to-nearest-even;
  * THD document lengths ~ U{lo..hi} drawn while the running total fits; the rest
    of the token budget is padding absorbed into the last segment.

Workloads are the five shapes the pages' bug report and PR discuss (tiny fp32
check, BSHD bf16, packed THD bf16, 64k long context, dense-loss sweep).
"""
from __future__ import annotations

import dataclasses
import math
import os
from typing import Optional

import numpy as np

TENSOR_IDS = {
    "q_idx": 1, "w": 2, "k_idx": 3, "q": 4, "kv": 5, "kv_c": 6, "sink": 7,
    "doclens": 8, "variant": 9,
}

_BLOCK = 1 << 22  # elements per independently seeded block (parallel, thread-count independent)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    layout: str            # "bshd" | "sbhd" | "thd"
    dtype: str             # "f32" | "bf16"
    batch: int             # BSHD/SBHD: sequences. THD: ignored (derived)
    seqlen: int            # BSHD/SBHD: per-sequence length. THD: total physical tokens
    ratio: int
    heads: int
    head_dim: int
    idx_heads: int
    idx_dim: int
    topk: int
    window: int
    sink_std: float = 1.0
    sparse: bool = True
    reduction: str = "mean"   # "mean" over physical rows | "sum"
    coeff: float = 1.0
    seed: int = 0
    doc_len: tuple = (512, 4096)  # THD only: inclusive range of document lengths
    softmax_scale: Optional[float] = None  # default 1/sqrt(head_dim)
    qk_std: Optional[float] = None  # std of q, kv and kv_c (default 1/sqrt(head_dim)); 1.0 gives logits of order one
    sink_mean: float = 0.0

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.head_dim)

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# The five workloads (shapes, sizes and value distributions of the pages' cases).
CONFIGS = {
    "tiny_fp32": Config("tiny_fp32", "bshd", "f32", 1, 256, 4, 8, 64, 4, 32, 16, 32, seed=0,
                        softmax_scale=1.0 / 8.0),
    "bshd_bf16": Config("bshd_bf16", "bshd", "bf16", 2, 4096, 4, 64, 192, 64, 128, 512, 128, seed=1),
    "thd_bf16": Config("thd_bf16", "thd", "bf16", 0, 16384, 4, 64, 192, 64, 128, 512, 128, seed=2),
    "long_bf16": Config("long_bf16", "bshd", "bf16", 1, 65536, 4, 128, 512, 64, 128, 2048, 128,
                        sink_std=2.0, seed=3),
    "dense_bf16": Config("dense_bf16", "bshd", "bf16", 1, 32768, 128, 128, 512, 64, 128, 256, 512,
                         sparse=False, seed=4),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even); returns the uint16 bit patterns."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, tensor: str, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, TENSOR_IDS[tensor], extra])))


def _blocks(n: int, fill):
    """Run fill(block_index, start, stop) over fixed blocks of _BLOCK elements, on a thread pool."""
    nb = (n + _BLOCK - 1) // _BLOCK
    if nb <= 1:
        for i in range(nb):
            fill(i, 0, n)
        return
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(max_workers=min(nb, os.cpu_count() or 4)) as ex:
        list(ex.map(lambda i: fill(i, i * _BLOCK, min(n, (i + 1) * _BLOCK)), range(nb)))


def _normal_into(seed: int, tensor: str, n: int, std: float, dtype: str):
    """N(0, std^2) draws, one seeded stream per block: float32 values, or bf16 bit patterns."""
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(i, a, b):
        x = _rng(seed, tensor, 1 + i).standard_normal(b - a, dtype=np.float32) * np.float32(std)
        out[a:b] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    _blocks(n, fill)
    return out


class Tensor:
    """One input tensor: bf16 bit patterns (bf16 tensors) or float32 values (fp32 tensors).

    ``values`` gives the exact float32 values (computed on demand for bf16); ``rows_f32(idx)`` gives the values
    of selected rows of the flattened leading dims without widening the whole tensor.
    """

    def __init__(self, values: Optional[np.ndarray] = None, bits: Optional[np.ndarray] = None, lead: int = 1):
        assert (values is None) != (bits is None) or values is not None
        self._values = values
        self.bits = bits
        self.lead = lead  # number of leading dims that index rows

    @property
    def values(self) -> np.ndarray:
        if self._values is None:
            self._values = bf16_bits_to_f32(self.bits).reshape(self.bits.shape)
        return self._values

    @property
    def shape(self):
        return (self.bits if self.bits is not None else self._values).shape

    def rows_f32(self, idx) -> np.ndarray:
        src = self.bits if self.bits is not None else self._values
        flat = src.reshape((-1,) + src.shape[self.lead:])
        sel = flat[np.asarray(idx)]
        return bf16_bits_to_f32(sel).reshape(sel.shape) if self.bits is not None else np.array(sel, np.float32)


def _make(values: np.ndarray, dtype: str, lead: int = 1) -> Tensor:
    if dtype == "bf16":
        return Tensor(bits=f32_to_bf16_bits(values).reshape(values.shape), lead=lead)
    return Tensor(np.ascontiguousarray(values, dtype=np.float32), lead=lead)


def thd_doc_lengths(cfg: Config):
    """Seeded document lengths for a packed THD batch.

    Returns (cu_seqlens_q, cu_seqlens_q_unpadded, max_seqlen_q = longest unpadded segment): lengths ~ U{lo..hi} are drawn
    while the running total fits in cfg.seqlen; the remaining tokens are padding absorbed into
    the last segment (physical offsets), and the unpadded offsets stop at the real total.
    """
    lo, hi = cfg.doc_len
    rng = _rng(cfg.seed, "doclens")
    lens = []
    total = 0
    while True:
        L = int(rng.integers(lo, hi + 1))
        if total + L > cfg.seqlen:
            break
        lens.append(L)
        total += L
    if not lens:  # budget below the smallest length: one short document
        lens = [cfg.seqlen]
        total = cfg.seqlen
    real = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    phys = real.copy()
    phys[-1] = cfg.seqlen
    max_len = int(np.max(np.diff(real)))  # longest unpadded segment: padding rows see no keys
    return phys, real, max_len


@dataclasses.dataclass
class Inputs:
    cfg: Config
    q_idx: Tensor
    w: Tensor
    k_idx: Tensor
    q: Tensor
    kv: Tensor
    kv_c: Tensor
    sink: Tensor
    cu_seqlens_q: Optional[np.ndarray] = None
    cu_seqlens_q_unpadded: Optional[np.ndarray] = None
    max_seqlen_q: int = 0

    @property
    def rows(self) -> int:
        c = self.cfg
        return c.seqlen if c.layout == "thd" else c.batch * c.seqlen


def _lead_shapes(cfg: Config, n_c_rows: int):
    """Leading dims of (query-like tensors, compressed tensors) for the layout."""
    if cfg.layout == "bshd":
        return (cfg.batch, cfg.seqlen), (cfg.batch, cfg.seqlen // cfg.ratio)
    if cfg.layout == "sbhd":
        return (cfg.seqlen, cfg.batch), (cfg.seqlen // cfg.ratio, cfg.batch)
    return (cfg.seqlen,), (n_c_rows,)


def generate(cfg: Config, skip=()) -> Inputs:
    """Draw every input of one step for `cfg`.  Names listed in `skip` are left as 0-size arrays
    (used by callers that need only the indexer-side tensors)."""
    cu = cur = None
    max_len = 0
    n_c_rows = 0
    if cfg.layout == "thd":
        cu, cur, max_len = thd_doc_lengths(cfg)
        # compressed rows are laid out per segment by physical length // ratio; since only the
        # last segment carries padding, the unpadded packing cumsum(real // ratio) is a prefix
        n_c_rows = int(sum((cu[i + 1] - cu[i]) // cfg.ratio for i in range(len(cu) - 1)))
    # All draws are made in the canonical (BSHD/THD) order; SBHD is a transpose of the same draw,
    # so a BSHD and an SBHD input of one config hold the same logical values.
    canon = cfg if cfg.layout != "sbhd" else cfg.replace(layout="bshd")
    cq, cc = _lead_shapes(canon, n_c_rows)
    nlead = 2 if canon.layout != "thd" else 1

    def normal_tensor(name, shape, std):
        if name in skip:
            return Tensor(np.zeros((0,), np.float32))
        n = int(np.prod(shape))
        arr = _normal_into(cfg.seed, name, n, std, cfg.dtype).reshape(shape)
        return Tensor(bits=arr, lead=nlead) if cfg.dtype == "bf16" else Tensor(arr, lead=nlead)

    q_idx = normal_tensor("q_idx", cq + (cfg.idx_heads, cfg.idx_dim), 1.0 / math.sqrt(cfg.idx_dim))
    k_idx = normal_tensor("k_idx", cc + (cfg.idx_dim,), 1.0 / math.sqrt(cfg.idx_dim))
    main_std = cfg.qk_std if cfg.qk_std is not None else 1.0 / math.sqrt(cfg.head_dim)
    q = normal_tensor("q", cq + (cfg.heads, cfg.head_dim), main_std)
    kv = normal_tensor("kv", cq + (cfg.head_dim,), main_std)
    kv_c = normal_tensor("kv_c", cc + (cfg.head_dim,), main_std)
    if "w" in skip:
        w = Tensor(np.zeros((0,), np.float32))
    else:
        n = int(np.prod(cq)) * cfg.idx_heads
        wv = np.empty(n, np.float32)

        def fill(i, a, b):
            wv[a:b] = _rng(cfg.seed, "w", 1 + i).random(b - a, dtype=np.float32)

        _blocks(n, fill)
        w = Tensor(wv.reshape(cq + (cfg.idx_heads,)), lead=nlead)
    sink = Tensor(_rng(cfg.seed, "sink").standard_normal(cfg.heads, dtype=np.float32) * np.float32(cfg.sink_std)
                  + np.float32(cfg.sink_mean))

    inp = Inputs(cfg, q_idx, w, k_idx, q, kv, kv_c, sink, cu, cur, max_len)
    if cfg.layout == "sbhd":
        inp = to_sbhd(inp)
    return inp


def _swap01(t: Tensor) -> Tensor:
    if len(t.shape) < 2:
        return t
    if t.bits is not None:
        return Tensor(bits=np.ascontiguousarray(np.swapaxes(t.bits, 0, 1)), lead=t.lead)
    return Tensor(np.ascontiguousarray(np.swapaxes(t.values, 0, 1)), lead=t.lead)


def to_sbhd(inp: Inputs) -> Inputs:
    """Re-lay a BSHD input as SBHD (same values, sequence-major)."""
    c = inp.cfg.replace(layout="sbhd")
    return Inputs(c, _swap01(inp.q_idx), _swap01(inp.w), _swap01(inp.k_idx), _swap01(inp.q),
                  _swap01(inp.kv), _swap01(inp.kv_c), inp.sink)


def to_thd(inp: Inputs) -> Inputs:
    """Re-lay a BSHD input as a packed THD batch of equal-length, unpadded segments."""
    c = inp.cfg
    assert c.layout == "bshd"
    B, S = c.batch, c.seqlen

    def flat(t: Tensor) -> Tensor:
        if t.bits is not None:
            return Tensor(bits=np.ascontiguousarray(t.bits.reshape((-1,) + t.bits.shape[2:])), lead=1)
        return Tensor(np.ascontiguousarray(t.values.reshape((-1,) + t.values.shape[2:])), lead=1)

    cu = (np.arange(B + 1) * S).astype(np.int32)
    c2 = c.replace(layout="thd", seqlen=B * S, batch=0)
    return Inputs(c2, flat(inp.q_idx), flat(inp.w), flat(inp.k_idx), flat(inp.q), flat(inp.kv),
                  flat(inp.kv_c), inp.sink, cu, cu.copy(), S)


def dense_variant(inp: Inputs, v: int) -> Inputs:
    """Teacher-sensitivity variant v of the dense-loss sweep.

    Variants 0..3 move every original-KV (window) value by +3 or -3: kv += 3 * e_v with e_v a seeded
    +-1 vector over the head dimension (the same for every row).  Variants 4..7 add +3 / -3 to the sink
    of one seeded head.  Only window values or one head's sink change; indexer inputs and compressed KV
    do not.
    """
    c = inp.cfg
    rng = _rng(c.seed, "variant", v)
    kv, sink = inp.kv, inp.sink
    if v < 4:
        e = np.where(rng.random(c.head_dim) < 0.5, -3.0, 3.0).astype(np.float32)
        kv = _make((inp.kv.values + e).astype(np.float32), c.dtype, lead=inp.kv.lead)
    else:
        h = int(rng.integers(0, c.heads))
        s = inp.sink.values.copy()
        s[h] += np.float32(3.0 if v % 2 == 0 else -3.0)
        sink = Tensor(s)
    return dataclasses.replace(inp, kv=kv, sink=sink)


def tiny(name="tiny", layout="bshd", dtype="f32", batch=1, seqlen=64, ratio=4, heads=2, head_dim=16,
         idx_heads=2, idx_dim=8, topk=8, window=8, **kw) -> Config:
    """Helper for small test shapes."""
    return Config(name, layout, dtype, batch, seqlen, ratio, heads, head_dim, idx_heads, idx_dim, topk,
                  window, **kw)
