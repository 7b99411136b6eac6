"""The C-ABI library on a machine without a GPU: it loads, exports every symbol the header declares, and
its host-side logic (sizes, argument validation, fault injection) behaves; no compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa_indexer.h")


def _no_gpu():
    """Tests that hand made-up device addresses to the library run only where no GPU exists: on a GPU machine a
    regression in the host-side validation would otherwise launch kernels on those addresses."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("passes made-up device addresses: run only where no GPU exists")


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_tcgen05_gb300 import build
    build.build()
    from sparse_attention_indexer_tcgen05_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(csa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_step(B):
    names = declared_functions()
    for n in ("csa_indexer_fwd", "csa_teacher", "csa_indexer_bwd", "csa_workspace_size", "csa_topk_width"):
        assert n in names


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(B.EXPORTED) | set(declared_functions())


def _params(B, **kw):
    base = dict(layout="bshd", dtype="bf16", batch=2, seqlen=4096, compress_ratio=4, window=128, topk=512, heads=64,
                head_dim=192, idx_heads=64, idx_dim=128, softmax_scale=0.072)
    base.update(kw)
    return B.Params(**base)


def test_sizes(B):
    p = _params(B)
    assert (p.K, p.key_width, p.teacher_width, p.rows, p.compressed_rows) == (512, 1024, 512, 8192, 2048)
    assert p.workspace_bytes >= 2 * 8192 * 512 * 4 + 2048 * 128 * 4
    assert _params(B, topk=5000).K == 1024                         # K = min(topk, n_c)
    assert _params(B, sparse_loss=False, topk=16).teacher_width == 1024  # dense teacher spans the key axis
    assert _params(B, seqlen=3).K == 0                              # no compressed key at all
    assert _params(B, layout="sbhd").compressed_rows == 2048


def test_bench_workload_fits_the_no_allocation_scratch(B):
    """The bshd_bf16 workload (the default bench case) runs through csa_indexer_bwd_noalloc: its workspace
    (teacher rows, the by-key gradient rows of the tensor-core backward, dK accumulator, per-row loss) stays
    inside the library's fixed scratch of CSA_NOALLOC_SCRATCH_BYTES."""
    m = re.search(r"#define CSA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", open(HEADER).read())
    scratch = int(m.group(1)) << int(m.group(2))
    p = _params(B)
    assert 8192 * 512 * 4 + 8192 * 1024 * 4 <= p.workspace_bytes <= scratch


@pytest.mark.parametrize("field,value", [("compress_ratio", 0), ("topk", 0), ("window", -1), ("heads", 0),
                                         ("batch", 0), ("seqlen", -5), ("reduction", 2), ("sparse_loss", 3),
                                         ("layout", 7), ("dtype", 9), ("key_rows", 5), ("teacher_mode", 2)])
def test_invalid_params_rejected(B, field, value):
    _no_gpu()
    p = _params(B)
    setattr(p.c, field, value)
    assert p.K == -1 and p.workspace_bytes == 0
    st = B._lib.csa_indexer_fwd(p.ref, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 1 << 40, None)
    assert st == 1


def test_teacher_mode_accepted(B):
    """The compressed-only teacher changes no width: it is the same step with the sink and window dropped."""
    full, comp = _params(B), _params(B, teacher_mode="compressed_only")
    assert comp.c.teacher_mode == 1 and full.c.teacher_mode == 0
    assert (comp.K, comp.teacher_width, comp.workspace_bytes) == (full.K, full.teacher_width, full.workspace_bytes)


def test_thd_requires_offsets(B):
    p = _params(B, layout="thd", batch=3, seqlen=100, max_seqlen_q=50, key_rows=25)
    assert p.K == -1  # no cu_seqlens_q
    p.c.cu_seqlens_q = 0x7000
    assert p.K == 12
    p.c.max_seqlen_q = 101
    assert p.K == -1  # a segment cannot be longer than all rows


def test_pointer_validation_before_any_launch(B):
    _no_gpu()
    p = _params(B)
    big = 1 << 40
    f = B._lib.csa_indexer_fwd
    assert f(p.ref, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, big, None) == 1       # null input
    assert f(p.ref, 0x1000, 0x2000, 0x3008, 0x4000, 0x5000, 0x6000, big, None) == 3     # misaligned
    assert f(p.ref, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 16, None) == 4      # small workspace
    assert f(None, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, big, None) == 1      # no params
    bwd = B._lib.csa_indexer_bwd
    args = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 0x9000, None]
    assert bwd(p.ref, *args, None, None, 0xa000, 0xb000, 0xc000, 0xd000, big, None) == 1  # no loss_out
    assert bwd(p.ref, *args, 0xe002, None, 0xa000, 0xb000, 0xc000, 0xd000, big, None) == 3  # misaligned loss
    tl = B._lib.csa_teacher_from_lse
    assert tl(p.ref, 0x1000, 0x2000, None, 0x4000, 0x5000, 0x6000, big, None) == 1     # no lse_nc
    assert tl(p.ref, 0x1000, 0x2000, 0x3004, 0x4000, 0x5000, 0x6000, big, None) == 3   # misaligned lse_nc
    assert tl(p.ref, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 16, None) == 4    # small workspace


def test_no_gpu_is_a_cuda_error_not_a_crash(B):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = _params(B)
    st = B._lib.csa_indexer_fwd(p.ref, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 1 << 40, None)
    assert st == 5


@pytest.mark.parametrize("site,status", [("invalid_arg", 1), ("unsupported", 2), ("alignment", 3),
                                         ("workspace", 4), ("cuda", 5), ("timeout", 6)])
def test_fault_injection(B, monkeypatch, site, status):
    _no_gpu()
    monkeypatch.setenv("CSA_FAULT", site)
    p = _params(B)
    assert B._lib.csa_indexer_fwd(p.ref, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 1 << 40, None) == status
    assert B._lib.csa_check_device_status(None) == status
    err = B.CSAError(status, "csa_indexer_fwd")
    assert B.STATUS[status] in str(err)


def test_noalloc_rejects_problems_beyond_the_scratch(B):
    """The 64k long-context shape needs far more than the fixed scratch of csa_indexer_bwd_noalloc: refused with
    CSA_ERR_WORKSPACE by the host-side size check, before anything is enqueued."""
    _no_gpu()
    p = B.Params("bshd", "bf16", 1, 65536, 4, 128, 2048, 128, 512, 64, 128, 0.044)
    assert p.workspace_bytes > B.NOALLOC_SCRATCH_BYTES
    fake = [0x10000 * (i + 1) for i in range(13)]
    # q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore | teacher | loss | row_loss | dq_idx, dw, dk_idx | stream
    st = B._lib.csa_indexer_bwd_noalloc(p.ref, *fake[:9], None, fake[9], None, fake[10], fake[11], fake[12], None)
    assert st == 4  # CSA_ERR_WORKSPACE


def test_require_tensor_cores_refuses_the_cuda_core_kernels(B):
    """With require_tensor_cores set, a call whose shape the tensor-core kernels do not take (here 8 indexer
    heads) returns CSA_ERR_UNSUPPORTED before anything is enqueued; fp32 values are refused the same way."""
    _no_gpu()
    big = 1 << 40
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, big, None)
    p = _params(B, idx_heads=8, require_tensor_cores=True)
    assert p.c.require_tensor_cores == 1
    assert B._lib.csa_indexer_fwd(p.ref, *args) == 2
    assert B._lib.csa_indexer_fwd(_params(B, dtype="f32", require_tensor_cores=True).ref, *args) == 2
    # without the flag the same call gets past the path choice (and fails only for want of a GPU)
    assert B._lib.csa_indexer_fwd(_params(B, idx_heads=8).ref, *args) == 5


def test_status_strings(B):
    for s, name in B.STATUS.items():
        assert B._lib.csa_status_string(s).decode().startswith(name)
