"""GPU path vs the float64 oracle, element by element, through the C ABI (needs a GB300)."""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import oracle as O  # noqa: E402
from sparse_attention_indexer_tcgen05_gb300 import synth  # noqa: E402

if torch.cuda.is_available():
    from sparse_attention_indexer_tcgen05_gb300 import binding as B  # noqa: E402
    from sparse_attention_indexer_tcgen05_gb300 import workload  # noqa: E402
    import parity_util as U  # noqa: E402

# per-case parity figures (errors, recall, path) are appended here as JSON lines
REPORT = os.environ.get("CSA_PARITY_REPORT_DIR",
                        os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "parity_reports"))


def _report(name, out):
    os.makedirs(REPORT, exist_ok=True)
    with open(os.path.join(REPORT, "parity_report.jsonl"), "a") as f:
        f.write(json.dumps({"case": name, **{k: v for k, v in out.items() if not k.startswith("_")}}) + "\n")


def small(**kw):
    base = dict(name="small", layout="bshd", dtype="bf16", batch=2, seqlen=300, ratio=4, heads=8, head_dim=64,
                idx_heads=8, idx_dim=32, topk=24, window=16, seed=21)
    base.update(kw)
    return synth.Config(**base)


# ------------------------------------------------------------------ the five workloads

def test_tiny_fp32_config():
    """tiny_fp32 in full: fp32 mode, tolerances 1e-4; ids must equal the float64 oracle's exactly."""
    inp = synth.generate(synth.CONFIGS["tiny_fp32"])
    out = U.check_step(inp)
    assert out["recall"] == (1.0, 1.0)
    _report("tiny_fp32", out)


def test_bshd_bf16_config_full():
    inp = synth.generate(synth.CONFIGS["bshd_bf16"])
    _report("bshd_bf16", U.check_step(inp))


def test_thd_bf16_config_full():
    inp = synth.generate(synth.CONFIGS["thd_bf16"])
    assert inp.cu_seqlens_q[-1] > inp.cu_seqlens_q_unpadded[-1]  # carries padding
    _report("thd_bf16", U.check_step(inp))


def test_long_bf16_config_sampled():
    """64k long context (16384 compressed keys, topk 2048, 128 main heads of 512): every stage on the tensor-core
    kernels; sampled rows against the oracle, dK element by element over the sampled rows' contributions."""
    inp = synth.generate(synth.CONFIGS["long_bf16"])
    rows = U.sample_rows(inp.rows, k=192, seed=3, must=(0, 3, 4, 8191, 8192))
    out = U.check_step(inp, rows=rows)
    assert (out["fwd_path"], out["teacher_path"], out["bwd_path"]) == ("tcgen05",) * 3, out
    _report("long_bf16", out)


def test_dense_bf16_config_full():
    """The dense-loss workload (32768 rows, every visible key in the support) on every row: ids, teacher, per-row
    KL, the whole-step loss and all three gradients element by element."""
    inp = synth.generate(synth.CONFIGS["dense_bf16"])
    out = U.check_step(inp)
    assert (out["fwd_path"], out["teacher_path"], out["bwd_path"]) == ("tcgen05",) * 3, out
    _report("dense_bf16", out)


def _variant_devices(d0, inp):
    return workload.DeviceInputs(d0.params, d0.q_idx, d0.w, d0.k_idx, d0.q,
                                 workload.tensor_to_torch(inp.kv, "bf16", "cuda:0"), d0.kv_c,
                                 workload.tensor_to_torch(inp.sink, "f32", "cuda:0"))


def test_dense_bf16_config_variants():
    """The dense-loss workload's 8 sensitivity variants (window values or one head's sink moved by +-3), sampled rows
    of each against the oracle.  With this workload's draws every attention logit is near zero, so a single head's
    sink barely moves the L1-normalised teacher; the change itself is tracked on the order-one-logit input below."""
    base = synth.generate(synth.CONFIGS["dense_bf16"])
    rows = U.sample_rows(base.rows, k=96, seed=4, must=(127, 128, 129, 32767))
    d0 = workload.to_device(base)
    for v in range(8):
        inp = synth.dense_variant(base, v)
        out = U.check_step(inp, d=_variant_devices(d0, inp), rows=rows)
        _report(f"dense_bf16_v{v}", out)


def test_teacher_sensitivity_sweep_tracks_the_oracle():
    """The dense-loss shape (128 heads of 512, window 512, ratio 128) on a shorter sequence with q, kv, kv_c ~ N(0, 1)
    so the attention logits are of order one, and sinks ~ N(6.5, 1), of the order of the other terms' log-sum-exp
    (about log(544) + 1/2 over the 512 window and 32 compressed logits), so that raising or lowering one head's sink
    both move its denominator: each of the 8 variants (every window value +-3, or one head's sink +-3) moves the
    teacher well above fp32 resolution, and the GPU must reproduce the oracle's change for every one of them
    (relative L2 of the change <= 0.25) and its change of every row's KL."""
    cfg = synth.CONFIGS["dense_bf16"].replace(name="dense_sharp", seqlen=4096, qk_std=1.0, sink_mean=6.5, seed=5)
    base = synth.generate(cfg)
    rows = U.sample_rows(base.rows, k=64, seed=6, must=(127, 128, 129, 4095))
    d0 = workload.to_device(base)
    out0 = U.check_step(base, d=d0, rows=rows)
    lr0_o = out0["_oracle_loss_rows"]
    lr0_g = out0["_gpu_loss_rows"]
    for v in range(8):
        inp = synth.dense_variant(base, v)
        out = U.check_step(inp, d=_variant_devices(d0, inp), rows=rows)
        d_ora = out["_oracle_teacher"] - out0["_oracle_teacher"]
        d_gpu = out["_gpu_teacher_oracle_ids"].astype(np.float64) - out0["_gpu_teacher_oracle_ids"]
        change = float(np.abs(d_ora).sum() / np.abs(out0["_oracle_teacher"]).sum())
        assert change > 1e-4, f"variant {v} moves the oracle's teacher by only {change}"
        err = U.rel_l2(d_gpu, d_ora)
        assert err <= 0.25, f"variant {v}: GPU teacher change off by {err}"
        dl_err = U.rel_l2(out["_gpu_loss_rows"].astype(np.float64) - lr0_g, out["_oracle_loss_rows"] - lr0_o)
        assert dl_err <= 0.25, f"variant {v}: GPU per-row KL change off by {dl_err}"
        _report(f"dense_sharp_v{v}", dict(out, teacher_change=change, teacher_change_err=err, kl_change_err=dl_err))


# ------------------------------------------------------------------ layouts, ragged shapes, edge cases

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["bshd", "sbhd"])
def test_layouts_small(layout, dtype):
    cfg = small(layout=layout, dtype=dtype)
    _report(f"small_{layout}_{dtype}", U.check_step(synth.generate(cfg)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_thd_ragged_with_padding(dtype):
    cfg = small(layout="thd", dtype=dtype, seqlen=700, ratio=3, doc_len=(37, 260), seed=5)
    inp = synth.generate(cfg)
    assert inp.cu_seqlens_q[-1] > inp.cu_seqlens_q_unpadded[-1]
    _report(f"thd_ragged_{dtype}", U.check_step(inp))


def test_tensor_core_shape_multi_tile():
    """H_I = 64, D_I = 128 (the tensor-core shape) with a ragged key tail (n_c = 250)."""
    cfg = small(seqlen=1000, heads=16, head_dim=64, idx_heads=64, idx_dim=128, topk=96, window=40, seed=8)
    _report("tc_shape_bshd", U.check_step(synth.generate(cfg)))


@pytest.mark.parametrize("layout", ["bshd", "sbhd"])
def test_tensor_core_shape_odd_length(layout):
    """The tensor-core shapes (H = 64 teacher heads, H_I = 64, D_I = 128) with an odd sequence length, so the
    last row pair of each sequence has one row, in both position-major and sequence-major layouts."""
    cfg = small(layout=layout, seqlen=999, heads=64, head_dim=64, idx_heads=64, idx_dim=128, topk=96, window=40,
                seed=10)
    out = U.check_step(synth.generate(cfg))
    assert out["path"] == "tcgen05" and out["bwd_path"] == "tcgen05", (out["path"], out["bwd_path"])
    _report(f"tc_shape_odd_{layout}", out)


def test_tensor_core_shape_thd():
    cfg = small(layout="thd", seqlen=2600, heads=16, head_dim=64, idx_heads=64, idx_dim=128, topk=128, window=40,
                doc_len=(300, 1200), seed=9)
    _report("tc_shape_thd", U.check_step(synth.generate(cfg)))


# ------------------------------------------------------------------ long key axis (streaming top-k)

def _long_axis(**kw):
    """Key axes past 1024 (ratio 1, so every position is a compressed key): the score kernel streams its score
    tiles into per-row candidate buffers, which are cut back to the top K whenever they fill up (rows with
    more than ~3968 visible keys see several cuts)."""
    base = dict(batch=2, seqlen=4608, ratio=1, heads=16, head_dim=64, idx_heads=64, idx_dim=128, topk=300,
                window=32, seed=40)
    base.update(kw)
    return small(**base)


@pytest.mark.parametrize("layout", ["bshd", "sbhd"])
def test_long_key_axis_streaming_topk(layout):
    inp = synth.generate(_long_axis(layout=layout))
    rows = U.sample_rows(inp.rows, k=96, seed=41, must=(0, 299, 300, 4607, 4608, 9215))
    out = U.check_step(inp, rows=rows)
    assert out["fwd_path"] == "tcgen05"
    _report(f"long_axis_{layout}", out)


def test_long_key_axis_exact_ties_across_cuts():
    """k_idx repeats every 37 rows, so every score value recurs about v / 37 times in a row: the selection must
    keep the lowest keys of each tied value across every cut of the candidate buffer (strict check: ids equal
    the oracle's top-k of the GPU's own fp32 scores)."""
    inp = synth.generate(_long_axis(batch=1, seqlen=5000, topk=500, seed=42))
    bits = inp.k_idx.bits
    idx = np.arange(bits.shape[1]) % 37
    inp.k_idx = synth.Tensor(bits=np.ascontiguousarray(bits[:, idx]), lead=2)
    rows = U.sample_rows(inp.rows, k=64, seed=43, must=(36, 37, 499, 500, 4999))
    out = U.check_step(inp, rows=rows)
    _report("long_axis_ties", out)


def test_long_key_axis_thd():
    cfg = _long_axis(layout="thd", seqlen=9000, doc_len=(2500, 5000), topk=256, seed=44)
    inp = synth.generate(cfg)
    rows = U.sample_rows(inp.rows, k=96, seed=45, must=(0, inp.rows - 1))
    out = U.check_step(inp, rows=rows)
    _report("long_axis_thd", out)


# ------------------------------------------------------------------ 128 main heads (one row per MMA tile)

def _h128(**kw):
    """128 main heads: one query row's heads fill the MMA's 128 lanes; the selected compressed keys are gathered.
    K = 300 spans three 128-key tiles (the last one ragged) and the window of 200 positions two tiles."""
    base = dict(batch=2, seqlen=1200, ratio=2, heads=128, head_dim=512, idx_heads=64, idx_dim=128, topk=300,
                window=200, seed=50)
    base.update(kw)
    return small(**base)


@pytest.mark.parametrize("layout,head_dim", [("bshd", 512), ("sbhd", 256), ("thd", 512)])
def test_teacher_128_heads(layout, head_dim):
    kw = dict(layout=layout, head_dim=head_dim)
    if layout == "thd":
        kw.update(seqlen=2600, doc_len=(500, 1500))
    out = U.check_step(synth.generate(_h128(**kw)))
    assert out["teacher_path"] == "tcgen05" and out["fwd_path"] == "tcgen05", out
    _report(f"h128_{layout}_d{head_dim}", out)


def test_teacher_128_heads_dense_loss():
    """Dense loss: every visible key (n_c = 187 <= topk) in contiguous tiles, the teacher indexed by key."""
    cfg = _h128(batch=1, seqlen=1500, ratio=8, topk=256, window=300, sparse=False, seed=51)
    out = U.check_step(synth.generate(cfg))
    assert out["teacher_path"] == "tcgen05", out
    _report("h128_dense", out)


def test_teacher_128_heads_modes():
    """The teacher from a given non-compressed log-sum-exp and the compressed-only teacher on the 128-head path."""
    inp = synth.generate(_h128(seqlen=700, seed=52))
    d = workload.to_device(inp)
    p = d.params
    ids, _ = B.csa_indexer_fwd(p, *d.indexer)
    ids_np = ids.cpu().numpy()
    P = O.Problem.from_inputs(inp)
    u = P.noncompressed_lse(inp.q.values, inp.kv.values, inp.sink.values)
    lse = torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).to(d.q.device)
    got = B.csa_teacher_from_lse(p, d.q, d.kv_c, lse, ids)
    torch.cuda.synchronize()
    B.csa_check_device_status()
    assert B.csa_last_path() == "tcgen05"
    ref = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids_np)
    e_lse = U.row_l1(got.cpu().numpy(), ref)
    assert e_lse <= 2e-2, e_lse
    d_comp = workload.to_device(inp, teacher_mode="compressed_only")
    t_comp = B.csa_teacher(d_comp.params, *d_comp.teacher_side, ids).cpu().numpy()
    B.csa_check_device_status()
    assert B.csa_last_path() == "tcgen05"
    ref_c = O.Problem.from_inputs(inp, window=0).teacher(inp.q.values, inp.kv.values, inp.kv_c.values,
                                                         np.full(inp.cfg.heads, -np.inf), ids_np)
    e_comp = U.row_l1(t_comp, ref_c)
    assert e_comp <= 2e-2, e_comp
    _report("h128_modes", dict(teacher_from_lse_err=e_lse, compressed_only_err=e_comp))


def test_dense_loss_with_unselected_keys():
    """Dense support (every visible key) while top-k keeps fewer: the backward rescoring path."""
    cfg = small(sparse=False, topk=10, seqlen=200)
    _report("dense_rescore", U.check_step(synth.generate(cfg)))


def test_no_window_no_sink_and_sum_reduction():
    cfg = small(window=0, reduction="sum", coeff=0.37)
    inp = synth.generate(cfg)
    inp.sink._values = np.full(cfg.heads, -np.inf, np.float32)
    _report("no_window_no_sink_sum", U.check_step(inp))


@pytest.mark.parametrize("dtype,wide", [("f32", False), ("bf16", True)])
def test_compressed_only_teacher_is_a_negative_control(dtype, wide):
    """teacher_mode="compressed_only" is the teacher the issue reports as the bug (a per-head softmax over the
    selected compressed keys alone).  It must equal the oracle's teacher with no window and no sink, and be
    blind to the window values and the sink, both of which move the full-CSA teacher.  wide=True takes the
    tensor-core teacher (64 heads), wide=False the CUDA-core one."""
    if wide:
        cfg = small(dtype=dtype, heads=64, head_dim=64, idx_heads=64, idx_dim=128, seqlen=600, topk=64, window=32)
    else:
        cfg = small(dtype=dtype)
    base = synth.generate(cfg)
    d_full = workload.to_device(base)
    d_comp = workload.to_device(base, teacher_mode="compressed_only")
    ids, _ = B.csa_indexer_fwd(d_full.params, *d_full.indexer)
    t_full = B.csa_teacher(d_full.params, *d_full.teacher_side, ids).cpu().numpy()
    t_comp = B.csa_teacher(d_comp.params, *d_comp.teacher_side, ids).cpu().numpy()
    B.csa_check_device_status()
    ref = O.Problem.from_inputs(base, window=0).teacher(base.q.values, base.kv.values, base.kv_c.values,
                                                        np.full(cfg.heads, -np.inf), ids.cpu().numpy())
    err = U.row_l1(t_comp, ref)
    assert err <= U.value_tol(dtype), f"compressed-only teacher row L1 error {err}"
    moved = 0.0
    for v in (0, 4):  # every window value moved by +-3; one head's sink moved by +3
        inp = synth.dense_variant(base, v)
        kv = workload.tensor_to_torch(inp.kv, dtype, "cuda:0")
        sink = workload.tensor_to_torch(inp.sink, "f32", "cuda:0")
        t_comp2 = B.csa_teacher(d_comp.params, d_comp.q, kv, d_comp.kv_c, sink, ids).cpu().numpy()
        t_full2 = B.csa_teacher(d_full.params, d_full.q, kv, d_full.kv_c, sink, ids).cpu().numpy()
        assert np.array_equal(t_comp2, t_comp), f"variant {v} moved the compressed-only teacher"
        moved = max(moved, float(np.abs(t_full2 - t_full).sum() / np.abs(t_full).sum()))
    assert moved > 1e-6, "the full teacher ignored the window and the sink"
    _report(f"compressed_only_teacher_{dtype}", dict(teacher_err=err, full_teacher_change=moved,
                                                     path=B.csa_last_path()))


def test_window_longer_than_sequence_and_topk_above_keys():
    cfg = small(seqlen=64, window=500, topk=1000)
    _report("window_gt_seq", U.check_step(synth.generate(cfg)))


def test_sequence_shorter_than_ratio_has_no_keys():
    cfg = small(seqlen=3, ratio=4)
    inp = synth.generate(cfg)
    d = workload.to_device(inp)
    p = d.params
    assert p.K == 0
    ids, sel = B.csa_indexer_fwd(p, *d.indexer)
    loss, dq, dw, dk = B.csa_indexer_bwd(p, *d.indexer, *d.teacher_side, ids, sel)
    assert ids.numel() == 0 and float(loss) == 0.0
    assert float(dq.float().abs().sum()) == 0.0 and float(dw.abs().sum()) == 0.0


def test_thd_single_segment_equals_bshd():
    cfg = small(batch=1, seqlen=400, idx_heads=64, idx_dim=128, seed=12)
    bshd = synth.generate(cfg)
    thd = synth.to_thd(bshd)
    a = U.gpu_step(workload.to_device(bshd))
    b = U.gpu_step(workload.to_device(thd))
    assert torch.equal(a["ids"], b["ids"])
    torch.testing.assert_close(a["teacher"], b["teacher"], rtol=1e-5, atol=1e-7)
    assert abs(a["loss"] - b["loss"]) <= 1e-5 * abs(a["loss"])


@pytest.mark.parametrize("dtype,wide,layout", [("f32", False, "bshd"), ("bf16", True, "bshd"), ("bf16", True, "sbhd"),
                                                ("bf16", True, "thd")])
def test_teacher_from_noncompressed_lse(dtype, wide, layout):
    """csa_teacher_from_lse with u_h = the oracle's sink-and-window log-sum-exp equals the oracle's full-CSA
    teacher (and the GPU's own full teacher) for the GPU's ids, on the CUDA-core (f32) and tensor-core paths."""
    kw = dict(layout=layout, dtype=dtype, seed=16)
    if wide:
        kw.update(seqlen=999, heads=64, head_dim=64, idx_heads=64, idx_dim=128, topk=96, window=40)
    if layout == "thd":
        kw.update(seqlen=2600, doc_len=(300, 1200))
    inp = synth.generate(small(**kw))
    d = workload.to_device(inp)
    p = d.params
    ids, _ = B.csa_indexer_fwd(p, *d.indexer)
    P = O.Problem.from_inputs(inp)
    ids_np = ids.cpu().numpy()
    u = P.noncompressed_lse(inp.q.values, inp.kv.values, inp.sink.values)
    lse = torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).to(d.q.device)
    got = B.csa_teacher_from_lse(p, d.q, d.kv_c, lse, ids)
    torch.cuda.synchronize()
    B.csa_check_device_status()
    assert B.csa_last_path() == ("tcgen05" if wide else "generic")
    got = got.cpu().numpy()
    ref = P.teacher(inp.q.values, inp.kv.values, inp.kv_c.values, inp.sink.values, ids_np)
    tol = U.value_tol(dtype)
    err = U.row_l1(got, ref)
    assert err <= tol, err
    full = B.csa_teacher(p, *d.teacher_side, ids).cpu().numpy()
    assert U.row_l1(got, full) <= tol
    _report(f"teacher_from_lse_{layout}_{dtype}", dict(teacher_err=err, path=B.csa_last_path()))


@pytest.mark.parametrize("layout", ["bshd", "sbhd", "thd"])
def test_backward_with_and_without_given_teacher(layout):
    """The backward that computes the teacher itself and the one given csa_teacher's rows run the same kernels
    on the same values: the loss, the per-row KL, dQ_idx and dW agree bit for bit; dK_idx sums key-tile
    partials with fp32 atomics in whatever order the CTAs finish, so it agrees to rounding."""
    kw = dict(layout=layout, seqlen=999, heads=64, head_dim=64, idx_heads=64, idx_dim=128, topk=96, window=40,
              seed=15)
    if layout == "thd":
        kw.update(seqlen=2600, doc_len=(300, 1200))
    d = workload.to_device(synth.generate(small(**kw)))
    p = d.params
    ids, sel = B.csa_indexer_fwd(p, *d.indexer)
    outs = []
    for teacher in (None, B.csa_teacher(p, *d.teacher_side, ids)):
        rl = torch.empty(p.rows, dtype=torch.float32, device=ids.device)
        loss, dq, dw, dk = B.csa_indexer_bwd(p, *d.indexer, *d.teacher_side, ids, sel, teacher=teacher, row_loss=rl)
        torch.cuda.synchronize()
        B.csa_check_device_status()
        assert B.csa_last_path() == "tcgen05"
        outs.append((loss, rl, dq, dw, dk))
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert torch.equal(a, b)
    dk0, dk1 = outs[0][4].double(), outs[1][4].double()
    assert float((dk0 - dk1).norm() / dk1.norm()) <= 1e-3


@pytest.mark.parametrize("axis", ["short", "long"])
def test_backward_128_heads_kl_inside_the_teacher(axis):
    """With 128 heads and the sparse loss the backward takes the KL step inside the teacher kernel (by key on
    short key axes, by slot on long ones).  Given csa_teacher's rows instead, it runs the separate KL kernel on
    the same values: the two agree to fp32 rounding (the max and the normaliser are reduced in another order),
    which is 1e-5 on the loss and the per-row KL.  The backward rounds g-derived MMA operands to bf16, and dQ_idx
    and dK_idx are bf16 outputs, so there a rounding difference can move a value by one bf16 unit (2^-8
    relative); a few such flips are allowed (2e-3 relative-L2 on dQ_idx, dW and dK_idx).
    The fused step matches the oracle on sampled rows."""
    kw = dict(batch=1, seqlen=1200, ratio=2, head_dim=128, topk=300, window=64, seed=53)
    if axis == "long":
        kw.update(seqlen=2600, topk=256)  # 1300 compressed keys: the long-axis backward over g by slot
    inp = synth.generate(_h128(**kw))
    d = workload.to_device(inp)
    p = d.params
    ids, sel = B.csa_indexer_fwd(p, *d.indexer)
    outs = []
    for teacher in (None, B.csa_teacher(p, *d.teacher_side, ids)):
        rl = torch.empty(p.rows, dtype=torch.float32, device=ids.device)
        loss, dq, dw, dk = B.csa_indexer_bwd(p, *d.indexer, *d.teacher_side, ids, sel, teacher=teacher, row_loss=rl)
        torch.cuda.synchronize()
        B.csa_check_device_status()
        assert B.csa_last_path() == "tcgen05"
        outs.append([x.double() for x in (loss, rl, dq, dw, dk)])
    (l0, r0, q0, w0, k0), (l1, r1, q1, w1, k1) = outs
    assert abs(float(l0 - l1)) <= 1e-5 * abs(float(l1)) + 1e-12
    assert float((r0 - r1).abs().max()) <= 1e-5 * float(r1.abs().max()) + 1e-9
    for a, b, tol in ((q0, q1, 2e-3), (w0, w1, 2e-3), (k0, k1, 2e-3)):
        assert float((a - b).norm()) <= tol * float(b.norm()) + 1e-12, (tol, float((a - b).norm() / b.norm()))
    rows = U.sample_rows(inp.rows, k=48, seed=54, must=(0, inp.rows - 1))
    out = U.check_step(inp, rows=rows)
    assert out["teacher_path"] == "tcgen05", out
    _report(f"h128_kl_in_teacher_{axis}", out)


def test_batch_split_dk():
    """BSHD b=2 against two b=1 calls scaled for the row mean: the [PR] test plan's dK check (<= 8e-6 there)."""
    cfg = small(batch=2, seqlen=512, idx_heads=64, idx_dim=128, topk=64, seed=13, dtype="f32")
    inp = synth.generate(cfg)
    full = U.gpu_step(workload.to_device(inp))
    n_c = 128
    for b in range(2):
        sub = synth.Inputs(cfg.replace(batch=1), *(synth.Tensor(t.values[b:b + 1], lead=2) for t in
                                                   (inp.q_idx, inp.w, inp.k_idx, inp.q, inp.kv, inp.kv_c)), inp.sink)
        one = U.gpu_step(workload.to_device(sub))
        got = full["dk"].reshape(-1, 128)[b * n_c:(b + 1) * n_c].double()
        exp = one["dk"].reshape(-1, 128).double() / 2
        rel = float((got - exp).norm() / exp.norm())
        assert rel <= 1e-5, rel
        ids_b = full["ids"][b * 512:(b + 1) * 512]
        assert torch.equal(ids_b, torch.where(one["ids"] >= 0, one["ids"] + b * n_c, one["ids"]))


def test_autograd_function():
    cfg = small(idx_heads=64, idx_dim=128, dtype="f32", seed=14)
    inp = synth.generate(cfg)
    d = workload.to_device(inp)
    qi = d.q_idx.clone().requires_grad_(True)
    w = d.w.clone().requires_grad_(True)
    ki = d.k_idx.clone().requires_grad_(True)
    q = d.q.clone().requires_grad_(True)
    ids, loss = B.csa_indexer_loss(qi, w, ki, q, d.kv, d.kv_c, d.sink, d.params)
    (3.0 * loss).backward()
    ref = U.gpu_step(d)
    torch.testing.assert_close(qi.grad, 3.0 * ref["dq"], rtol=1e-5, atol=1e-9)
    torch.testing.assert_close(w.grad, 3.0 * ref["dw"], rtol=1e-5, atol=1e-9)
    torch.testing.assert_close(ki.grad, 3.0 * ref["dk"], rtol=1e-5, atol=1e-9)
    assert q.grad is None  # no gradient to the teacher side


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """A device-side bounded wait that runs out (csa_selftest_bounded_wait: the tensor-core kernels' wait, limited
    to about 1 ms, on a barrier nothing arrives on) is reported on the host as CSA_ERR_TIMEOUT by the next
    csa_check_device_status, which clears it; the CUDA context stays usable and the next step is correct."""
    stream = torch.cuda.current_stream().cuda_stream
    assert B._lib.csa_selftest_bounded_wait(stream) == 0
    assert B._lib.csa_check_device_status(stream) == 6      # CSA_ERR_TIMEOUT
    assert B.csa_last_timeout_site() == 990                 # the self-test (9), its wait site 90
    assert B._lib.csa_check_device_status(stream) == 0      # read and cleared
    out = U.check_step(synth.generate(small(idx_heads=64, idx_dim=128, heads=64, seed=17)))
    assert out["fwd_path"] == "tcgen05"
    _report("after_timeout", out)


def test_require_tensor_cores_runs_every_step_on_tcgen05():
    """With require_tensor_cores set, a shape the tcgen05 kernels take runs as usual; one they do not take (8
    indexer heads) is refused with CSA_ERR_UNSUPPORTED and nothing runs."""
    inp = synth.generate(small(idx_heads=64, idx_dim=128, heads=64, seed=18))
    d = workload.to_device(inp, require_tensor_cores=True)
    ids, sel = B.csa_indexer_fwd(d.params, *d.indexer)
    B.csa_indexer_bwd(d.params, *d.indexer, *d.teacher_side, ids, sel)
    torch.cuda.synchronize()
    assert B.csa_last_path() == "tcgen05"
    d8 = workload.to_device(synth.generate(small(seed=18)), require_tensor_cores=True)
    with pytest.raises(B.CSAError) as e:
        B.csa_indexer_fwd(d8.params, *d8.indexer)
    assert e.value.status == 2
    B.csa_check_device_status()


def test_errors_fail_closed():
    cfg = small()
    d = workload.to_device(synth.generate(cfg))
    p = d.params
    with pytest.raises(B.CSAError) as e:
        B.csa_indexer_fwd(p, *d.indexer, workspace=torch.empty(1, dtype=torch.uint8, device="cuda:0"))
    assert e.value.status == 4
    B.csa_check_device_status()
