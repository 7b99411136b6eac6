"""Comparison helpers for the GPU-vs-oracle parity tests (imported by the test files only).

Acceptance (the step's stated tolerances):
  * top-k ids: bit-exact against the oracle's selection applied to the GPU's own fp32 scores; against the
    oracle's float64 selection, a swap is allowed only between keys whose float64 scores lie within the
    row's measured fp32 score error of the selection threshold (a rounding near-tie);
  * GPU fp32 scores vs float64: within 2 (D_I + H_I) u_fp32 sum_j w_j sum_d |q_jd k_d| per (row, key), twice the
    first-order worst case of any fp32 summation order;
  * teacher (per row L1 error / L1 norm) and loss (relative): 1e-4 in fp32 mode, 2e-2 in bf16 mode;
  * dq_idx, dw, dk_idx: relative L2 error <= 2e-2.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from sparse_attention_indexer_tcgen05_gb300 import binding as B
from sparse_attention_indexer_tcgen05_gb300 import workload

U32 = 2.0 ** -24
GRAD_TOL = 2e-2


def value_tol(dtype: str) -> float:
    return 1e-4 if dtype == "f32" else 2e-2


def gpu_step(d: workload.DeviceInputs, want_teacher=True):
    """The natural pipeline through the C ABI: fwd -> teacher -> bwd (teacher recomputed inside bwd)."""
    p = d.params
    ids, sel = B.csa_indexer_fwd(p, *d.indexer)
    out = dict(ids=ids, sel=sel, fwd_path=B.csa_last_path())
    if want_teacher:
        out["teacher"] = B.csa_teacher(p, *d.teacher_side, ids)
        out["teacher_path"] = B.csa_last_path()
    row_loss = torch.empty(p.rows, dtype=torch.float32, device=ids.device)
    loss, dq, dw, dk = B.csa_indexer_bwd(p, *d.indexer, *d.teacher_side, ids, sel, row_loss=row_loss)
    torch.cuda.synchronize()
    B.csa_check_device_status()
    out.update(loss=float(loss), dq=dq, dw=dw, dk=dk, row_loss=row_loss, bwd_path=B.csa_last_path())
    return out


def to_np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def row_geometry(inp, rows):
    """(first global id, visible count) of each listed row, decoded from the layout (test-side plumbing)."""
    c = inp.cfg
    rows = np.asarray(rows, np.int64)
    if c.layout == "thd":
        cu, cur = inp.cu_seqlens_q.astype(np.int64), inp.cu_seqlens_q_unpadded.astype(np.int64)
        b = np.searchsorted(cu, rows, side="right") - 1
        b = np.minimum(b, len(cu) - 2)
        cu_c = np.concatenate([[0], np.cumsum(np.diff(cur) // c.ratio)])
        s = rows - cu[b]
        real = (cur[b + 1] - cur[b])
        v = np.where(s < real, (s + 1) // c.ratio, 0)
        return cu_c[b], v
    nc = c.seqlen // c.ratio
    b, s = (rows // c.seqlen, rows % c.seqlen) if c.layout == "bshd" else (rows % c.batch, rows // c.batch)
    return b * nc, (s + 1) // c.ratio


def key_memory_rows(inp, gids):
    c = inp.cfg
    if c.layout == "sbhd":
        nc = c.seqlen // c.ratio
        return (gids % nc) * c.batch + gids // nc
    return gids


def score_bound(inp, rows):
    """Per (row, local key) rounding bound 2 (D_I + H_I) u sum_j w_j sum_d |q_jd k_d| (float64), [rows, key width]."""
    P = O.Problem.from_inputs(inp)
    NC = P.key_width
    qi = np.abs(inp.q_idx.rows_f32(rows).astype(np.float64))
    w = inp.w.rows_f32(rows).astype(np.float64)
    DI = inp.cfg.idx_dim
    ki = np.abs(inp.k_idx.values.astype(np.float64)).reshape(-1, DI)
    a = np.einsum("rj,rjd->rd", w.reshape(len(rows), -1), qi.reshape(len(rows), -1, DI))   # [rows, DI]
    first, v = row_geometry(inp, rows)
    out = np.zeros((len(rows), NC))
    for i in range(len(rows)):
        if v[i] == 0:
            continue
        kr = key_memory_rows(inp, first[i] + np.arange(v[i]))
        out[i, :v[i]] = 2.0 * (DI + inp.cfg.idx_heads) * U32 * (ki[kr] @ a[i])
    return out


def check_scores(gpu_scores, ref_scores, inp, rows):
    """GPU fp32 scores against float64: same visibility, error within the rounding bound.  Returns |error|."""
    vis = np.isfinite(ref_scores)
    assert np.array_equal(vis, np.isfinite(gpu_scores)), "visibility pattern differs"
    err = np.where(vis, np.abs(gpu_scores.astype(np.float64) - np.where(vis, ref_scores, 0.0)), 0.0)
    bound = score_bound(inp, rows) + 1e-30
    ratio = np.max(err / bound)
    assert ratio <= 1.0, f"score error {ratio:.3g} x the rounding bound"
    return err


def check_ids(gpu_ids, gpu_scores, ref_scores, inp, P: O.Problem, rows, err):
    """Strict (same fp32 scores) and end-to-end (float64) top-k checks; returns (mean, min) recall."""
    strict = P.topk(gpu_scores.astype(np.float64), rows)
    bad = np.any(strict != gpu_ids, axis=1)
    assert not bad.any(), f"ids differ from the oracle's selection on the GPU's own fp32 scores in {bad.sum()} rows"
    ref_ids = P.topk(ref_scores, rows)
    first, v = row_geometry(inp, rows)
    recalls = []
    for i in range(len(rows)):
        g = set(gpu_ids[i][gpu_ids[i] >= 0].tolist())
        o = set(ref_ids[i][ref_ids[i] >= 0].tolist())
        assert len(g) == len(o), f"row {rows[i]}: {len(g)} ids vs {len(o)}"
        recalls.append(1.0 if not o else len(g & o) / len(o))
        if g == o:
            continue
        vis = ref_scores[i][: v[i]]
        kth = np.sort(vis)[::-1][len(o) - 1]
        E = 2.0 * np.max(err[i][: v[i]])
        for gid in g ^ o:
            s = ref_scores[i][gid - first[i]]
            assert abs(s - kth) <= E, f"row {rows[i]}: key {gid} swapped at {abs(s - kth):.3g} from the threshold > {E:.3g}"
    return float(np.mean(recalls)), float(np.min(recalls))


def rel_l2(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-300))


def row_l1(a, b):
    num = np.abs(np.asarray(a, np.float64) - b).sum(axis=1)
    den = np.abs(b).sum(axis=1)
    ok = den > 0
    return float(np.max(num[ok] / den[ok])) if np.any(ok) else 0.0


def gpu_scores(d, rows):
    """GPU fp32 scores of the listed rows (csa_scores_debug over each contiguous run of rows)."""
    rows = np.asarray(rows, np.int64)
    out = np.empty((len(rows), d.params.key_width), np.float32)
    i = 0
    while i < len(rows):
        j = i
        while j + 1 < len(rows) and rows[j + 1] == rows[j] + 1:
            j += 1
        out[i:j + 1] = B.csa_scores_debug(d.params, *d.indexer, int(rows[i]), j - i + 1).cpu().numpy()
        i = j + 1
    return out


def sample_rows(n_rows, k=256, seed=0, must=()):
    """Stratified row sample: evenly spread rows, the last rows (most keys), and the given rows."""
    rng = np.random.default_rng(seed)
    even = np.linspace(0, n_rows - 1, k // 2).astype(np.int64)
    rand = rng.integers(0, n_rows, k // 4)
    tail = np.arange(max(0, n_rows - k // 4), n_rows)
    return np.unique(np.concatenate([even, rand, tail, np.asarray(must, np.int64)])).astype(np.int32)


def check_step(inp, d=None, rows=None, full_dk=True, report=None):
    """Run the GPU pipeline and check every output against the oracle (own float64 selection).

    rows=None: every row (dk compared in full).  Otherwise only the listed rows are checked row-wise, and dk
    through the homogeneity invariant sum_s k_s . dK_s = sum_t sum_j q_tj . dQ_tj on the GPU outputs."""
    c = inp.cfg
    tol = value_tol(c.dtype)
    d = d if d is not None else workload.to_device(inp)
    gpu = gpu_step(d)
    P = O.Problem.from_inputs(inp)
    ref = P.step(inp, rows=rows, want_dk=rows is None)
    rws = ref["rows"]
    gs = gpu_scores(d, rws)
    err = check_scores(gs, ref["scores"], inp, rws)
    ids_g = gpu["ids"].cpu().numpy()[rws]
    recall = check_ids(ids_g, gs, ref["scores"], inp, P, rws, err)
    same = np.all(ids_g == ref["ids"], axis=1)
    # teacher: the GPU pipeline's own teacher on rows whose selection matches, and the GPU teacher of the
    # oracle's ids on every row
    te_g = gpu["teacher"].cpu().numpy()[rws]
    t_err = row_l1(te_g[same], ref["teacher"][same]) if same.any() else 0.0
    assert t_err <= tol, f"teacher row L1 error {t_err}"
    ids_o = np.full((d.params.rows, d.params.K), -1, np.int32)
    ids_o[rws] = ref["ids"]
    te_o = B.csa_teacher(d.params, *d.teacher_side, torch.from_numpy(ids_o).to(d.q.device)).cpu().numpy()[rws]
    t_err2 = row_l1(te_o, ref["teacher"])
    assert t_err2 <= tol, f"teacher (oracle ids) row L1 error {t_err2}"
    # per-row KL and the loss
    rl = gpu["row_loss"].cpu().numpy()[rws]
    # relative to the row's own KL, floored at the mean row KL (a row's KL can be a near-cancelling difference)
    floor = max(float(np.mean(np.abs(ref["loss_rows"]))), 1e-12)
    l_err = float(np.max(np.abs(rl[same] - ref["loss_rows"][same]) / np.maximum(np.abs(ref["loss_rows"][same]), floor)))
    assert l_err <= tol, f"per-row KL error {l_err}"
    if rows is None:
        loss_err = abs(gpu["loss"] - ref["loss"]) / abs(ref["loss"])
        assert loss_err <= tol, f"loss {gpu['loss']} vs {ref['loss']}"
    # gradients
    dq = to_np(gpu["dq"]).reshape(P.rows, c.idx_heads, c.idx_dim)[rws]
    dw = to_np(gpu["dw"]).reshape(P.rows, c.idx_heads)[rws]
    e_dq = rel_l2(dq[same], ref["dq"][same])
    e_dw = rel_l2(dw[same], ref["dw"][same])
    assert e_dq <= GRAD_TOL and e_dw <= GRAD_TOL, f"dq {e_dq} dw {e_dw}"
    out = dict(recall=recall, teacher_err=max(t_err, t_err2), dq_err=e_dq, dw_err=e_dw, rows=len(rws),
               same_rows=int(same.sum()), path=gpu["fwd_path"], fwd_path=gpu["fwd_path"],
               teacher_path=gpu["teacher_path"], bwd_path=gpu["bwd_path"],
               _oracle_teacher=ref["teacher"], _gpu_teacher_oracle_ids=te_o,
               _oracle_loss_rows=ref["loss_rows"], _gpu_loss_rows=rl)
    dk = to_np(gpu["dk"]).reshape(-1, c.idx_dim)
    if rows is None:
        e_dk = rel_l2(dk, ref["dk"])
        assert e_dk <= GRAD_TOL, f"dk {e_dk}"
        out["dk_err"] = e_dk
        out["loss_err"] = loss_err
    else:
        out.update(check_sampled_dk(inp, d, P, rws, gpu["ids"]))
    if report is not None:
        report.update(out)
    return out


def check_sampled_dk(inp, d, P, rws, ids_gpu):
    """dK element by element on a row sample: the GPU step is run again with w zeroed on every row outside the
    sample.  Those rows then score every key 0 and, since dK takes each row's contribution through w, add nothing
    to dK (dK_s = sum_t sum_j g_ts w_tj 1[x_tjs > 0] q_tj), while the sampled rows keep their scores, ids, teacher
    and gradient.  The oracle computes the sampled rows' dK from the same ids (the GPU's), with its own teacher and
    float64 scores.  Also compares the sampled rows' summed loss."""
    c = inp.cfg
    p = d.params
    keep = torch.zeros(p.rows, dtype=torch.bool, device=d.w.device)
    keep[torch.from_numpy(np.asarray(rws, np.int64)).to(d.w.device)] = True
    w_m = torch.where(keep.view((p.rows,) + (1,) * 1), d.w.reshape(p.rows, -1), torch.zeros((), device=d.w.device))
    w_m = w_m.reshape(d.w.shape).contiguous()
    dm = workload.DeviceInputs(p, d.q_idx, w_m, d.k_idx, d.q, d.kv, d.kv_c, d.sink, d.cu, d.cur)
    ids_m, sel_m = B.csa_indexer_fwd(p, *dm.indexer)
    rl = torch.empty(p.rows, dtype=torch.float32, device=ids_m.device)
    _, _, _, dk_m = B.csa_indexer_bwd(p, *dm.indexer, *dm.teacher_side, ids_m, sel_m, row_loss=rl)
    torch.cuda.synchronize()
    B.csa_check_device_status()
    ids_s = ids_m.cpu().numpy()[rws]
    assert np.array_equal(ids_s, ids_gpu.cpu().numpy()[rws]), "masking other rows changed the sampled rows' ids"
    qq = inp.q.rows_f32(rws)
    te_s = P.teacher(qq, inp.kv.values, inp.kv_c.values, inp.sink.values, ids_s, rws, compact=True)
    qi, ww = inp.q_idx.rows_f32(rws), inp.w.rows_f32(rws)
    loss_o, lr_o, _, _, dk_o = P.loss_grads(qi, ww, inp.k_idx.values, ids_s, te_s, rws, want_dk=True, compact=True)
    e_dk = rel_l2(to_np(dk_m).reshape(-1, c.idx_dim), dk_o)
    assert e_dk <= GRAD_TOL, f"dk (sampled rows) {e_dk}"
    loss_g = float(rl.cpu().numpy()[rws].astype(np.float64).sum()) * P.loss_factor
    e_loss = abs(loss_g - loss_o) / max(abs(loss_o), 1e-30)
    assert e_loss <= value_tol(c.dtype), f"sampled-row loss {loss_g} vs {loss_o}"
    return dict(dk_err=e_dk, sampled_loss_err=e_loss)
