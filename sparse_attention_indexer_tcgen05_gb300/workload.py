"""Moves seeded synthetic inputs (``synth``) onto a CUDA device and builds the matching ``Params``.

Host<->device plumbing only; no step of the method is computed here.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import synth
from .binding import Params


def tensor_to_torch(t: synth.Tensor, dtype: str, device, pin: bool = False) -> torch.Tensor:
    """Exact bytes of a synth tensor as a torch tensor (bf16 from its bit patterns, else fp32)."""
    if t.bits is not None and dtype == "bf16":
        host = torch.from_numpy(np.ascontiguousarray(t.bits).view(np.int16)).view(torch.bfloat16)
    else:
        host = torch.from_numpy(np.ascontiguousarray(t.values, dtype=np.float32))
    if device is None or device == "cpu":
        return host.pin_memory() if pin else host
    return host.to(device, non_blocking=False)


@dataclasses.dataclass
class DeviceInputs:
    params: Params
    q_idx: torch.Tensor
    w: torch.Tensor
    k_idx: torch.Tensor
    q: torch.Tensor
    kv: torch.Tensor
    kv_c: torch.Tensor
    sink: torch.Tensor
    cu: torch.Tensor = None
    cur: torch.Tensor = None

    @property
    def indexer(self):
        return self.q_idx, self.w, self.k_idx

    @property
    def teacher_side(self):
        return self.q, self.kv, self.kv_c, self.sink

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.q_idx, self.w, self.k_idx, self.q, self.kv,
                                                          self.kv_c, self.sink))


def params_for(inp: synth.Inputs, cu=None, cur=None, **over) -> Params:
    c = inp.cfg
    kw = dict(layout=c.layout, dtype=c.dtype, batch=c.batch if c.layout != "thd" else len(inp.cu_seqlens_q) - 1,
              seqlen=c.seqlen, compress_ratio=c.ratio, window=c.window, topk=c.topk, heads=c.heads,
              head_dim=c.head_dim, idx_heads=c.idx_heads, idx_dim=c.idx_dim, softmax_scale=c.scale,
              sparse_loss=c.sparse, reduction=c.reduction, loss_coeff=c.coeff, cu_seqlens_q=cu,
              cu_seqlens_q_unpadded=cur, max_seqlen_q=inp.max_seqlen_q,
              key_rows=inp.k_idx.values.shape[0] if c.layout == "thd" else 0)
    kw.update(over)
    return Params(**kw)


def to_device(inp: synth.Inputs, device="cuda:0", **over) -> DeviceInputs:
    c = inp.cfg
    cu = cur = None
    if c.layout == "thd":
        cu = torch.from_numpy(np.ascontiguousarray(inp.cu_seqlens_q, dtype=np.int32)).to(device)
        cur = torch.from_numpy(np.ascontiguousarray(inp.cu_seqlens_q_unpadded, dtype=np.int32)).to(device)
    p = params_for(inp, cu, cur, **over)
    conv = lambda t: tensor_to_torch(t, c.dtype, device)
    f32 = lambda t: tensor_to_torch(t, "f32", device)
    return DeviceInputs(p, conv(inp.q_idx), f32(inp.w), conv(inp.k_idx), conv(inp.q), conv(inp.kv), conv(inp.kv_c),
                        f32(inp.sink), cu, cur)
