"""Pins of the float64 oracle to what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a value derived from the pages'
equations (tests/golden), a textbook special case computed with a library routine, brute force on
tiny inputs, an invariant, or finite differences.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax, logsumexp

from oracle import oracle as O
from sparse_attention_indexer_tcgen05_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(x):
    if isinstance(x, str):
        if x.startswith("ln"):
            return math.log(float(x[2:]))
        return float(Fraction(x))
    return float(x)


def small(layout="bshd", **kw):
    base = dict(batch=2, seqlen=48, ratio=4, heads=3, head_dim=8, idx_heads=3, idx_dim=8, topk=5, window=6,
                seed=11)
    base.update(kw)
    return synth.tiny(layout=layout, **base)


def problem(inp, **over):
    return O.Problem.from_inputs(inp, **over)


# --------------------------------------------------------------------------- mask (step 1)

@pytest.mark.parametrize("ratio,seqlen", [(4, 48), (3, 50), (1, 9), (5, 23)])
def test_mask_matches_page_expression(ratio, seqlen):
    """Visibility equals the page's mask expression: -inf where arange(n_c) >= arange(1, sq+1) // ratio."""
    inp = synth.generate(small(ratio=ratio, seqlen=seqlen, batch=1))
    P = problem(inp)
    sc = P.scores(inp.q_idx.values, inp.w.values, inp.k_idx.values)
    n_c = seqlen // ratio
    positions = np.arange(1, seqlen + 1)[:, None]
    mask = np.where(np.arange(n_c)[None, :] >= positions // ratio, -np.inf, 0.0)
    assert np.array_equal(np.isfinite(sc), np.isfinite(mask))
    assert not np.isfinite(sc[: ratio - 1]).any()          # rows i < r see no key
    assert np.isfinite(sc[-1]).sum() == seqlen // ratio     # the last row sees every key


# --------------------------------------------------------------------------- scores (step 1)

def test_scores_reduce_to_matmul():
    """One head, w = 1, all dot products positive: I is the plain matrix product q_idx @ k_idx^T."""
    cfg = small(batch=1, idx_heads=1, seqlen=40)
    inp = synth.generate(cfg)
    inp.q_idx.values[:] = np.abs(inp.q_idx.values)
    inp.k_idx.values[:] = np.abs(inp.k_idx.values)
    inp.w.values[:] = 1.0
    P = problem(inp)
    sc = P.scores(inp.q_idx.values, inp.w.values, inp.k_idx.values)
    ref = inp.q_idx.values[0, :, 0, :].astype(np.float64) @ inp.k_idx.values[0].astype(np.float64).T
    vis = np.isfinite(sc)
    np.testing.assert_allclose(sc[vis], ref[vis], rtol=1e-13)


def test_scores_relu_and_homogeneity():
    """ReLU drops negative heads; I is linear in w and positively 1-homogeneous in q_idx."""
    inp = synth.generate(small(batch=1))
    P = problem(inp)
    qi, w, ki = inp.q_idx.values.astype(np.float64), inp.w.values.astype(np.float64), inp.k_idx.values
    base = P.scores(qi, w, ki)
    vis = np.isfinite(base)
    # all-negative dot products -> zero score
    qpos = np.abs(qi)
    zero = P.scores(qpos, w, -np.abs(ki))
    assert np.all(zero[vis] == 0.0)
    # linear in w
    w2 = np.random.default_rng(0).random(w.shape)
    np.testing.assert_allclose(P.scores(qi, w + w2, ki)[vis], base[vis] + P.scores(qi, w2, ki)[vis],
                               rtol=1e-12, atol=1e-14)
    # 1-homogeneous in q_idx for positive factors
    np.testing.assert_allclose(P.scores(2.5 * qi, w, ki)[vis], 2.5 * base[vis], rtol=1e-13)
    # a head with w = 0 contributes nothing: dropping it changes nothing
    w3 = w.copy()
    w3[..., 0] = 0.0
    qi3 = qi.copy()
    qi3[..., 0, :] = 1e3 * np.random.default_rng(1).standard_normal(qi3[..., 0, :].shape)
    np.testing.assert_allclose(P.scores(qi3, w3, ki)[vis], P.scores(qi, w3, ki)[vis], rtol=1e-13)


# --------------------------------------------------------------------------- top-k (step 2)

def _brute_topk(scores_row, v, K, gid_of):
    order = sorted(range(v), key=lambda j: (-scores_row[j], j))[: min(K, v)]
    ids = sorted(gid_of(j) for j in order)
    return ids + [-1] * (K - len(ids))


@pytest.mark.parametrize("layout", ["bshd", "sbhd"])
def test_topk_brute_force_with_ties(layout):
    cfg = small(layout="bshd", batch=2, seqlen=64, topk=6)
    inp = synth.generate(cfg)
    # forced ties: duplicate compressed keys, and keys whose every dot product is negative (score 0)
    inp.k_idx.values[:, 5] = inp.k_idx.values[:, 2]
    inp.k_idx.values[:, 9] = inp.k_idx.values[:, 2]
    inp.q_idx.values[0, 40:] = np.abs(inp.q_idx.values[0, 40:])
    inp.k_idx.values[0, 11] = -np.abs(inp.k_idx.values[0, 11])
    inp.k_idx.values[0, 12] = -np.abs(inp.k_idx.values[0, 12])
    if layout == "sbhd":
        inp = synth.to_sbhd(inp)
    P = problem(inp)
    sc = P.scores(inp.q_idx.values, inp.w.values, inp.k_idx.values)
    ids = P.topk(sc)
    n_c, K, B, S = 16, P.K, 2, 64
    for r in range(B * S):
        b, s = (r // S, r % S) if layout == "bshd" else (r % B, r // B)
        v = (s + 1) // 4
        assert ids[r].tolist() == _brute_topk(sc[r], v, K, lambda j: b * n_c + j), r
    # ties really occurred and went to the lower index
    r = 0 * S + 63 if layout == "bshd" else 63 * B + 0
    assert (sc[r, 11] == 0.0) and (sc[r, 12] == 0.0)


def test_topk_negative_zero_ties_positive_zero():
    """-0.0 and +0.0 are the same score: the lower index wins."""
    inp = synth.generate(small(batch=1, seqlen=32, topk=2))
    P = problem(inp)
    sc = np.full((32, 8), -np.inf)
    sc[31, :] = [1.0, -0.0, 0.0, -1.0, 0.0, -0.0, 0.5, -2.0]
    ids = P.topk(sc)
    assert ids[31].tolist() == [0, 6]
    sc[31, :] = [-1.0, 0.0, -0.0, -1.0, -3.0, -0.0, -0.5, -2.0]
    ids = P.topk(sc)
    assert ids[31].tolist() == [1, 2]


def test_global_ids_batch_split():
    """BSHD b=2 ids are the two b=1 calls' ids with a b * n_c offset ([PR] item 1)."""
    cfg = small(batch=2, seqlen=40)
    inp = synth.generate(cfg)
    P = problem(inp)
    ids = P.topk(P.scores(inp.q_idx.values, inp.w.values, inp.k_idx.values))
    n_c = 10
    for b in range(2):
        sub = synth.Inputs(cfg.replace(batch=1), *(synth.Tensor(t.values[b:b + 1]) for t in
                                                   (inp.q_idx, inp.w, inp.k_idx, inp.q, inp.kv, inp.kv_c)),
                           inp.sink)
        P1 = problem(sub)
        ids1 = P1.topk(P1.scores(sub.q_idx.values, sub.w.values, sub.k_idx.values))
        exp = np.where(ids1 >= 0, ids1 + b * n_c, -1)
        assert np.array_equal(ids[b * 40:(b + 1) * 40], exp)


# --------------------------------------------------------------------------- teacher (step 3)

def _golden_problem(sink, window):
    # BSHD, B=1, S=2, ratio 1, topk 2, sigma 1, D 3 (construction in the golden file)
    cfg = synth.tiny(batch=1, seqlen=2, ratio=1, heads=2, head_dim=3, idx_heads=1, idx_dim=4, topk=2,
                     window=window, softmax_scale=1.0)
    inp = synth.generate(cfg)
    q = np.zeros((1, 2, 2, 3))
    q[0, 1, 0] = [0.0, math.log(3), math.log(5)]
    q[0, 1, 1] = [math.log(3), 0.0, 0.0]
    kv = np.zeros((1, 2, 3))
    kv[0, 1] = [0, 0, 1]
    kvc = np.zeros((1, 2, 3))
    kvc[0, 0] = [1, 0, 0]
    kvc[0, 1] = [0, 1, 0]
    P = problem(inp)
    ids = np.array([[0, 1]], np.int32)
    return P, q, kv, kvc, np.array(sink, np.float64), ids


def test_teacher_golden_two_heads():
    g = json.load(open(os.path.join(GOLDEN, "teacher_two_head.json")))
    for case in g["cases"]:
        sink = [_frac(x) for x in case["sink"]]
        P, q, kv, kvc, sk, ids = _golden_problem(sink, case["window"])
        t = P.teacher(q, kv, kvc, sk, ids, rows=[1])
        np.testing.assert_allclose(t[0], [_frac(x) for x in case["teacher"]], rtol=1e-14, err_msg=case["name"])
        # the compressed-only teacher (no window, sink = -inf) is the same in every case
        P0, q, kv, kvc, _, ids = _golden_problem(sink, 0)
        t0 = P0.teacher(q, kv, kvc, np.array([-np.inf, -np.inf]), ids, rows=[1])
        np.testing.assert_allclose(t0[0], [_frac(x) for x in case["compressed_only"]], rtol=1e-14)


def _teacher_case(layout="bshd", **kw):
    inp = synth.generate(small(layout=layout, **kw))
    P = problem(inp)
    ids = P.topk(P.scores(inp.q_idx.values, inp.w.values, inp.k_idx.values))
    return inp, P, ids


def test_teacher_sums_to_one():
    """I1: each valid row's teacher sums to 1; rows with no visible key are all zero."""
    inp, P, ids = _teacher_case(seqlen=64, heads=4)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    valid = (ids >= 0).any(axis=1)
    np.testing.assert_allclose(t[valid].sum(axis=1), 1.0, rtol=1e-13)
    assert np.all(t[~valid] == 0.0)
    assert np.all(t[ids < 0] == 0.0)


def _logits(inp, row_q, gids, scale):
    """sigma * q . key rows (library matmul) for a BSHD row."""
    b, s = row_q
    qh = inp.q.values[b, s].astype(np.float64)                      # [H, D]
    keys = inp.kv_c.values.reshape(-1, inp.kv_c.values.shape[-1])[gids].astype(np.float64)
    return scale * qh @ keys.T                                       # [H, n]


def test_teacher_single_head_is_softmax_over_C():
    """I2: with one head, t = softmax over C of the compressed logits, whatever the sink and window."""
    inp, P, ids = _teacher_case(heads=1, seqlen=64, window=10)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    t2 = P.teacher(inp.q.values, inp.kv.values * 7.0, inp.kv_c.values, inp.sink.values + 5.0, ids)
    np.testing.assert_allclose(t, t2, rtol=1e-12, atol=1e-15)
    for r in (30, 47, 64 + 63):
        b, s = divmod(r, 64)
        sel = ids[r][ids[r] >= 0]
        ref = softmax(_logits(inp, (b, s), sel, P.p.scale)[0])
        np.testing.assert_allclose(t[r, :len(sel)], ref, rtol=1e-12)


def test_teacher_without_window_and_sink_is_compressed_only():
    """I3: W = 0 and sink = -inf give the compressed-only teacher: per-head softmax over C, head sum, L1."""
    inp, P, ids = _teacher_case(heads=4, seqlen=64, window=0)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, np.full(4, -np.inf), ids)
    for r in (20, 40, 64 + 50):
        b, s = divmod(r, 64)
        sel = ids[r][ids[r] >= 0]
        per_head = softmax(_logits(inp, (b, s), sel, P.p.scale), axis=1).sum(axis=0)
        np.testing.assert_allclose(t[r, :len(sel)], per_head / per_head.sum(), rtol=1e-12)


def test_teacher_factored_lse_form_equals_direct_form():
    """I6: the follow-up proposal's factored form u_h, l_h, p_hj = exp(c_hj - l_h) gives the same t."""
    inp, P, ids = _teacher_case(heads=5, seqlen=64, window=7)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    W = 7
    for r in (10, 33, 63, 64 + 63):
        b, s = divmod(r, 64)
        sel = ids[r][ids[r] >= 0]
        c = _logits(inp, (b, s), sel, P.p.scale)                     # [H, n]
        p0 = max(0, s - W + 1)
        win = inp.kv.values[b, p0:s + 1].astype(np.float64)
        wl = P.p.scale * inp.q.values[b, s].astype(np.float64) @ win.T
        u = logsumexp(np.concatenate([inp.sink.values[:, None].astype(np.float64), wl], axis=1), axis=1)
        ell = logsumexp(np.concatenate([u[:, None], c], axis=1), axis=1)
        T = np.exp(c - ell[:, None]).sum(axis=0)
        np.testing.assert_allclose(t[r, :len(sel)], T / max(T.sum(), 1e-10), rtol=1e-13)


def test_noncompressed_lse_is_sink_and_window_logsumexp():
    """u_h = log(exp(a_h) + sum over the window of exp(sigma q.kv)), by scipy's logsumexp over the logits taken
    with a library matmul; with no window it is the sink itself, with neither it is -inf."""
    inp, P, ids = _teacher_case(heads=4, seqlen=64, window=7)
    u = P.noncompressed_lse(inp.q.values, inp.kv.values, inp.sink.values)
    assert u.shape == (P.rows, 4)
    for r in (0, 5, 33, 63, 64 + 2, 64 + 63):
        b, s = divmod(r, 64)
        win = inp.kv.values[b, max(0, s - 6):s + 1].astype(np.float64)
        wl = P.p.scale * inp.q.values[b, s].astype(np.float64) @ win.T
        ref = logsumexp(np.concatenate([inp.sink.values[:, None].astype(np.float64), wl], axis=1), axis=1)
        np.testing.assert_allclose(u[r], ref, rtol=1e-13)
    inp0, P0, _ = _teacher_case(heads=4, seqlen=64, window=0)
    u0 = P0.noncompressed_lse(inp0.q.values, inp0.kv.values, inp0.sink.values)
    assert np.array_equal(u0, np.broadcast_to(inp0.sink.values.astype(np.float64), u0.shape))
    assert np.all(P0.noncompressed_lse(inp0.q.values, inp0.kv.values, np.full(4, -np.inf)) == -np.inf)


@pytest.mark.parametrize("layout", ["bshd", "sbhd", "thd"])
def test_teacher_from_noncompressed_lse_equals_full_teacher(layout):
    """The teacher from a given u_h (the non-compressed log-sum-exp the proposal would take from the attention
    forward) equals the full-CSA teacher when u_h is the sink-and-window log-sum-exp of the same inputs, and
    the compressed-only teacher when u_h = -inf."""
    inp, P, ids = _teacher_case(layout=layout, heads=4, seqlen=64, window=9)
    q, kv, kv_c, sink = inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values
    t = P.teacher(q, kv, kv_c, sink, ids)
    u = P.noncompressed_lse(q, kv, sink)
    np.testing.assert_allclose(P.teacher_from_lse(q, kv_c, u, ids), t, rtol=1e-12, atol=1e-15)
    P0 = problem(inp, window=0)
    t0 = P0.teacher(q, kv, kv_c, np.full(4, -np.inf), ids)
    np.testing.assert_allclose(P.teacher_from_lse(q, kv_c, np.full_like(u, -np.inf), ids), t0, rtol=1e-12, atol=1e-15)


def test_attention_with_identical_rows_has_closed_form():
    """Every key/value row equal to one vector v: each of the n = |C| + |W| logits is x = sigma q.v, so
    l = log(e^a + n e^x) and O = n e^x / (e^a + n e^x) v (the sink takes the rest of the mass)."""
    inp, P, ids = _teacher_case(heads=3, seqlen=64, window=5)
    rng = np.random.default_rng(3)
    v = rng.standard_normal(inp.kv.values.shape[-1])
    kv = np.broadcast_to(v, inp.kv.values.shape).copy()
    kv_c = np.broadcast_to(v, inp.kv_c.values.shape).copy()
    O, lse = P.attention(inp.q.values, kv, kv_c, inp.sink.values, ids)
    for r in (3, 17, 40, 63, 64 + 30):
        b, s = divmod(r, 64)
        n = int((ids[r] >= 0).sum()) + min(5, s + 1)
        x = P.p.scale * inp.q.values[b, s].astype(np.float64) @ v          # [H]
        a = inp.sink.values.astype(np.float64)
        ell = np.logaddexp(a, np.log(n) + x)
        np.testing.assert_allclose(lse[r], ell, rtol=1e-13)
        np.testing.assert_allclose(O[r], (np.exp(np.log(n) + x - ell))[:, None] * v[None, :], rtol=1e-12, atol=1e-15)


def test_attention_single_key_no_sink_no_window_returns_its_value():
    """One visible compressed key, no window, no sink: the attention puts all mass on it, O = kv_c[key]."""
    inp, P, ids = _teacher_case(heads=2, seqlen=64, window=0)
    O, lse = P.attention(inp.q.values, inp.kv.values, inp.kv_c.values, np.full(2, -np.inf), ids)
    kvc = inp.kv_c.values.reshape(-1, inp.kv_c.values.shape[-1]).astype(np.float64)
    for r in (3, 4, 5, 6, 64 + 5):                     # positions 4..7: exactly one visible key (ratio 4)
        sel = ids[r][ids[r] >= 0]
        assert len(sel) == 1
        np.testing.assert_allclose(O[r], np.broadcast_to(kvc[sel[0]], O[r].shape), rtol=1e-14)
    assert np.all(lse[:3] == -np.inf) and np.all(O[:3] == 0.0)   # no key, no window, no sink


def test_attention_lse_reproduces_the_teacher():
    """The attention's l_h is the teacher's denominator: T_j = sum_h exp(c_hj - l_h), normalised, is the
    full-CSA teacher of the same inputs."""
    inp, P, ids = _teacher_case(heads=4, seqlen=64, window=9)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    _, lse = P.attention(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    for r in (10, 33, 63, 64 + 63):
        b, s = divmod(r, 64)
        sel = ids[r][ids[r] >= 0]
        c = _logits(inp, (b, s), sel, P.p.scale)                     # [H, n]
        T = np.exp(c - lse[r][:, None]).sum(axis=0)
        np.testing.assert_allclose(t[r, :len(sel)], T / T.sum(), rtol=1e-12)


def test_teacher_perturbations():
    """I5: with H > 1, changing only the window values or one head's sink changes the teacher, and leaves
    the selection and the predictor unchanged."""
    inp, P, ids = _teacher_case(heads=4, seqlen=64, window=8)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    sink2 = inp.sink.values.copy()
    sink2[2] += 3.0
    t_sink = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, sink2, ids)
    t_win = P.teacher(inp.q.values, inp.kv.values + 0.5, inp.kv_c.values, inp.sink.values, ids)
    many = (ids >= 0).sum(axis=1) >= 2
    assert np.abs(t_sink - t).max(axis=1)[many].min() > 1e-9
    assert np.abs(t_win - t).max(axis=1)[many].min() > 1e-9
    # compressed-only teacher is blind to both ([BUG] static reproduction)
    t0 = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, np.full(4, -np.inf), ids)
    P0 = O.Problem.from_inputs(inp, window=0)
    a = P0.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, np.full(4, -np.inf), ids)
    b = P0.teacher(inp.q.values, inp.kv.values + 0.5, inp.kv_c.values, np.full(4, -np.inf), ids)
    np.testing.assert_array_equal(a, b)
    # ids do not depend on the teacher-side inputs at all (scores only read q_idx, w, k_idx)
    ids2 = P.topk(P.scores(inp.q_idx.values, inp.w.values, inp.k_idx.values))
    np.testing.assert_array_equal(ids, ids2)


def test_teacher_single_head_sink_dominated_stays_finite():
    inp, P, ids = _teacher_case(heads=2, seqlen=64)
    t = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, np.array([80.0, -80.0]), ids)
    valid = (ids >= 0).any(axis=1)
    assert np.isfinite(t).all()
    np.testing.assert_allclose(t[valid].sum(axis=1), 1.0, rtol=1e-12)


# --------------------------------------------------------------------------- KL (step 4)

def test_kl_zero_when_predictor_equals_teacher():
    rng = np.random.default_rng(3)
    t = rng.random(9)
    t /= t.sum()
    L, g, p = O.kl_row(t, np.log(t) + 4.2)
    np.testing.assert_allclose(p, t, rtol=1e-13)
    assert abs(L) < 1e-14
    np.testing.assert_allclose(g, 0.0, atol=1e-9)


def test_kl_nonnegative_and_matches_scipy_entropy():
    from scipy.stats import entropy
    rng = np.random.default_rng(4)
    for n in (1, 2, 7, 40):
        t = rng.random(n)
        t /= t.sum()
        I = rng.standard_normal(n) * 3
        L, g, p = O.kl_row(t, I)
        assert L >= -1e-12
        # the 1e-10 guards move L from the textbook KL divergence by at most eps * sum(1 + t/p)
        p_ref = softmax(I)
        bound = 1e-10 * np.sum(1.0 + t / p_ref) + 1e-13
        assert abs(L - entropy(t, p_ref)) <= bound
        np.testing.assert_allclose(g.sum(), 0.0, atol=1e-12)


def test_kl_gradient_finite_differences():
    rng = np.random.default_rng(5)
    t = rng.random(12)
    t /= t.sum()
    I = rng.standard_normal(12)
    _, g, _ = O.kl_row(t, I)
    h = 1e-6
    fd = np.array([(O.kl_row(t, I + h * e, False)[0] - O.kl_row(t, I - h * e, False)[0]) / (2 * h)
                   for e in np.eye(12)])
    np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-10)


# --------------------------------------------------------------------------- backward (step 5)

def _fd_setup(layout="bshd", sparse=True, **kw):
    cfg = small(layout=layout, batch=2, seqlen=24, ratio=3, idx_heads=2, idx_dim=4, heads=2, head_dim=4,
                topk=3, window=4, sparse=sparse, **kw)
    inp = synth.generate(cfg)
    qi = inp.q_idx.values.astype(np.float64)
    w = inp.w.values.astype(np.float64)
    ki = inp.k_idx.values.astype(np.float64)
    P = problem(inp)
    ids = P.topk(P.scores(qi, w, ki))
    te = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    # reject points near a ReLU kink
    x = np.einsum("bshd,bcd->bshc", qi, ki)
    assert np.abs(x).min() > 1e-4
    return P, qi, w, ki, ids, te


@pytest.mark.parametrize("sparse", [True, False])
def test_gradients_finite_differences(sparse):
    P, qi, w, ki, ids, te = _fd_setup(sparse=sparse, coeff=1.7)
    loss, _, dq, dw, dk = P.loss_grads(qi, w, ki, ids, te)
    dq = dq.reshape(qi.shape)
    dw = dw.reshape(w.shape)
    dk = dk.reshape(ki.shape)
    h = 1e-6
    for arr, grad in ((qi, dq), (w, dw), (ki, dk)):
        fd = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for e in range(flat.size):
            old = flat[e]
            flat[e] = old + h
            lp = P.loss_grads(qi, w, ki, ids, te, want_dk=False)[0]
            flat[e] = old - h
            lm = P.loss_grads(qi, w, ki, ids, te, want_dk=False)[0]
            flat[e] = old
            fd.reshape(-1)[e] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - grad) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, err
        assert np.linalg.norm(grad) > 0


def test_gradient_homogeneity_invariants():
    """sum_j w dW = sum_j q_idx . dQ per row (both equal sum_s g_ts I_ts) and sum_s k . dK = sum over rows."""
    inp = synth.generate(small(seqlen=64, heads=2, idx_heads=4, idx_dim=16, topk=6))
    P = problem(inp)
    qi, w, ki = (t.values.astype(np.float64) for t in (inp.q_idx, inp.w, inp.k_idx))
    ids = P.topk(P.scores(qi, w, ki))
    te = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids)
    loss, lr, dq, dw, dk = P.loss_grads(qi, w, ki, ids, te)
    a = (w.reshape(dw.shape) * dw).sum(axis=1)
    b = (qi.reshape(dq.shape) * dq).sum(axis=(1, 2))
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-16)
    np.testing.assert_allclose((ki.reshape(dk.shape) * dk).sum(), b.sum(), rtol=1e-10)


def test_batch_split_equivalence():
    """dK of a b=2 call equals the two b=1 calls', scaled for the row mean ([PR] test plan)."""
    cfg = small(batch=2, seqlen=40)
    inp = synth.generate(cfg)
    P = problem(inp)
    full = P.step(inp)
    n_c = 10
    for b in range(2):
        sub = synth.Inputs(cfg.replace(batch=1), *(synth.Tensor(t.values[b:b + 1]) for t in
                                                   (inp.q_idx, inp.w, inp.k_idx, inp.q, inp.kv, inp.kv_c)),
                           inp.sink)
        one = problem(sub).step(sub)
        np.testing.assert_allclose(full["dk"][b * n_c:(b + 1) * n_c], one["dk"] / 2, rtol=1e-12, atol=1e-18)
        np.testing.assert_allclose(full["dq"][b * 40:(b + 1) * 40], one["dq"] / 2, rtol=1e-12, atol=1e-18)
        np.testing.assert_allclose(full["teacher"][b * 40:(b + 1) * 40], one["teacher"], rtol=1e-13)


# --------------------------------------------------------------------------- layouts and padding

def _all_outputs(inp):
    return problem(inp).step(inp)


def test_sbhd_bshd_thd_agree():
    cfg = small(batch=2, seqlen=44, ratio=4)
    bshd = synth.generate(cfg)
    a = _all_outputs(bshd)
    s = _all_outputs(synth.to_sbhd(bshd))
    t = _all_outputs(synth.to_thd(bshd))
    B, S = 2, 44
    perm = np.array([(r % B) * S + r // B for r in range(B * S)])  # SBHD row -> BSHD row
    for k in ("ids", "teacher", "dq", "dw"):
        np.testing.assert_array_equal(s[k], a[k][perm]) if k == "ids" else \
            np.testing.assert_allclose(s[k], a[k][perm], rtol=1e-12, atol=1e-18)
        np.testing.assert_array_equal(t[k], a[k]) if k == "ids" else \
            np.testing.assert_allclose(t[k], a[k], rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(s["loss"], a["loss"], rtol=1e-12)
    np.testing.assert_allclose(t["loss"], a["loss"], rtol=1e-12)
    # SBHD compressed rows are [n_c, B]: dk row j*B+b <-> BSHD row b*n_c+j
    n_c = S // 4
    permk = np.array([(r % B) * n_c + r // B for r in range(B * n_c)])
    np.testing.assert_allclose(s["dk"], a["dk"][permk], rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(t["dk"], a["dk"], rtol=1e-12, atol=1e-18)


def test_thd_segments_are_independent_bshd_calls():
    """Each THD segment behaves as its own b=1 sequence: per-segment mask and packed global ids."""
    cfg = synth.tiny(layout="thd", seqlen=100, ratio=4, heads=2, head_dim=8, idx_heads=2, idx_dim=8, topk=4,
                     window=5, doc_len=(13, 40), seed=5)
    inp = synth.generate(cfg)
    cu, cur = inp.cu_seqlens_q, inp.cu_seqlens_q_unpadded
    P = problem(inp)
    full = P.step(inp)
    c_base = 0
    for b in range(len(cu) - 1):
        L = int(cur[b + 1] - cur[b])
        r0 = int(cu[b])
        sl = slice(r0, r0 + L)
        cfg1 = cfg.replace(layout="bshd", batch=1, seqlen=L)
        nc = L // 4
        sub = synth.Inputs(cfg1, synth.Tensor(inp.q_idx.values[None, sl]), synth.Tensor(inp.w.values[None, sl]),
                           synth.Tensor(inp.k_idx.values[None, c_base:c_base + nc]), synth.Tensor(inp.q.values[None, sl]),
                           synth.Tensor(inp.kv.values[None, sl]), synth.Tensor(inp.kv_c.values[None, c_base:c_base + nc]),
                           inp.sink)
        P1 = problem(sub)
        one = P1.step(sub)
        K1 = P1.K
        ids = full["ids"][sl]
        assert np.all(ids[:, K1:] == -1)
        np.testing.assert_array_equal(ids[:, :K1], np.where(one["ids"] >= 0, one["ids"] + c_base, -1))
        np.testing.assert_allclose(full["teacher"][sl][:, :K1], one["teacher"], rtol=1e-13, atol=1e-300)
        scale = cfg1.seqlen / inp.rows  # mean over each call's own physical rows
        np.testing.assert_allclose(full["dq"][sl], one["dq"] * scale, rtol=1e-12, atol=1e-18)
        c_base += nc


def test_thd_padding_rows_are_inert():
    """Padding rows ([BUG] fused-path excerpt) get ids -1, teacher 0, no loss and no gradient, but count in
    the mean's divisor (the review's physical-row contract)."""
    cfg = synth.tiny(layout="thd", seqlen=120, ratio=4, heads=2, head_dim=8, idx_heads=2, idx_dim=8, topk=4,
                     window=5, doc_len=(20, 50), seed=6)
    inp = synth.generate(cfg)
    cu, cur = inp.cu_seqlens_q, inp.cu_seqlens_q_unpadded
    assert cu[-1] > cur[-1], "fixture must carry padding"
    P = problem(inp)
    out = P.step(inp)
    pad = np.arange(cur[-1], cu[-1])
    assert np.all(out["ids"][pad] == -1)
    assert np.all(out["teacher"][pad] == 0)
    assert np.all(out["dq"][pad] == 0) and np.all(out["dw"][pad] == 0)
    assert np.all(out["loss_rows"][pad] == 0)
    # same step without padding: sum mode agrees exactly, mean mode by the divisor ratio
    real = int(cur[-1])
    inp2 = synth.Inputs(cfg.replace(seqlen=real), *(synth.Tensor(t.values[:real]) for t in
                                                    (inp.q_idx, inp.w)), inp.k_idx,
                        synth.Tensor(inp.q.values[:real]), synth.Tensor(inp.kv.values[:real]), inp.kv_c, inp.sink,
                        cur.copy(), cur.copy(), int(np.max(np.diff(cur))))
    P2 = O.Problem.from_inputs(inp2, max_seqlen_q=inp.max_seqlen_q)
    out2 = P2.step(inp2)
    np.testing.assert_allclose(out["loss"] * cu[-1], out2["loss"] * real, rtol=1e-12)
    Ps = O.Problem.from_inputs(inp, reduction="sum")
    Ps2 = O.Problem.from_inputs(inp2, reduction="sum", max_seqlen_q=inp.max_seqlen_q)
    np.testing.assert_allclose(Ps.step(inp)["loss"], Ps2.step(inp2)["loss"], rtol=1e-12)


def test_dense_equals_sparse_when_every_key_is_selected():
    cfg = small(seqlen=48, topk=12)  # topk = n_c: every visible key is selected
    inp = synth.generate(cfg)
    a = problem(inp).step(inp)
    b = O.Problem.from_inputs(inp, sparse=False).step(inp)
    np.testing.assert_array_equal(a["ids"], b["ids"])
    np.testing.assert_allclose(a["teacher"], b["teacher"], rtol=1e-13)
    np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-13)
    np.testing.assert_allclose(a["dk"], b["dk"], rtol=1e-12, atol=1e-18)


def test_dense_support_is_every_visible_key():
    cfg = small(seqlen=48, topk=3, sparse=False)
    inp = synth.generate(cfg)
    P = problem(inp)
    out = P.step(inp)
    assert P.teacher_width == 12
    for r in (20, 47):
        v = (r + 1) // 4
        assert np.all(out["teacher"][r, :v] > 0) and np.all(out["teacher"][r, v:] == 0)
        np.testing.assert_allclose(out["teacher"][r].sum(), 1.0, rtol=1e-13)


def test_loss_reduction_modes():
    inp = synth.generate(small(seqlen=40))
    m = problem(inp).step(inp)
    s = O.Problem.from_inputs(inp, reduction="sum").step(inp)
    np.testing.assert_allclose(m["loss"] * 80, s["loss"], rtol=1e-13)
    np.testing.assert_allclose(m["loss_rows"], s["loss_rows"], rtol=1e-13)
    np.testing.assert_allclose(m["dk"] * 80, s["dk"], rtol=1e-12)
