"""bench.py's host-side pieces on CPU: the algorithmic work per stage (the roofline's numerator) against a
row-by-row count from the layouts' definitions, and the synthetic inputs' reproducibility."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from sparse_attention_indexer_tcgen05_gb300 import synth  # noqa: E402


def _rows_geometry(cfg, inp):
    """(visible keys v, window rows w) of every row, walking the layout's definition row by row."""
    out = []
    if cfg.layout == "thd":
        cu, cur = inp.cu_seqlens_q, inp.cu_seqlens_q_unpadded
        for b in range(len(cu) - 1):
            real = cur[b + 1] - cur[b]
            for s in range(cu[b + 1] - cu[b]):
                out.append(((s + 1) // cfg.ratio, min(cfg.window, s + 1)) if s < real else (0, 0))
    else:
        order = [(b, s) for b in range(cfg.batch) for s in range(cfg.seqlen)]
        if cfg.layout == "sbhd":
            order = [(b, s) for s in range(cfg.seqlen) for b in range(cfg.batch)]
        for b, s in order:
            out.append(((s + 1) // cfg.ratio, min(cfg.window, s + 1)))
    return out


@pytest.mark.parametrize("layout", ["bshd", "sbhd", "thd"])
def test_algorithmic_flops_match_a_row_by_row_count(layout):
    import bench
    kw = dict(layout=layout, batch=2, seqlen=90, ratio=4, heads=3, head_dim=8, idx_heads=4, idx_dim=16, topk=7,
              window=6, seed=5)
    if layout == "thd":
        kw.update(batch=1, seqlen=300, doc_len=(40, 120))
    cfg = synth.tiny(**kw)
    inp = synth.generate(cfg)
    geo = _rows_geometry(cfg, inp)
    K = min(cfg.topk, max(v for v, _ in geo)) if cfg.layout != "thd" else None
    if K is None:  # THD: K = min(topk, key width of the longest unpadded segment)
        cur = inp.cu_seqlens_q_unpadded
        K = min(cfg.topk, int(max(np.diff(cur))) // cfg.ratio)
    fl, by, ex = bench.algorithmic(cfg, inp, K, len(geo))
    score = sum(2 * cfg.idx_heads * cfg.idx_dim * v for v, _ in geo)
    k_of = [min(v, K) for v, _ in geo]
    w_of = [w if v > 0 else 0 for v, w in geo]
    teacher = sum(2 * cfg.heads * cfg.head_dim * (k + w) for k, w in zip(k_of, w_of))
    grads = sum(6 * cfg.idx_heads * cfg.idx_dim * k for k in k_of)
    exps = sum(cfg.heads * (1 + w + 2 * k) for (v, _), k, w in zip(geo, k_of, w_of) if v > 0)
    assert fl["score_topk"] == score
    assert fl["teacher"] == teacher
    assert fl["teacher_from_lse"] == sum(2 * cfg.heads * cfg.head_dim * k for k in k_of)
    assert fl["kl_grad"] == grads
    assert ex == exps


def test_synthetic_inputs_are_reproducible():
    cfg = synth.tiny(layout="bshd", batch=2, seqlen=64, heads=2, head_dim=16, seed=9)
    a, b = synth.generate(cfg), synth.generate(cfg)
    for name in ("q_idx", "w", "k_idx", "q", "kv", "kv_c", "sink"):
        x, y = getattr(a, name), getattr(b, name)
        x = x.values if hasattr(x, "values") else x
        y = y.values if hasattr(y, "values") else y
        assert np.array_equal(x, y), name
    c = synth.generate(synth.tiny(layout="bshd", batch=2, seqlen=64, heads=2, head_dim=16, seed=10))
    assert not np.array_equal(a.q.values, c.q.values)
