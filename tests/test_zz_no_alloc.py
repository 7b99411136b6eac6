"""csa_indexer_bwd_noalloc: the backward for callers that cannot allocate device memory (no workspace
argument; the library's own fixed device scratch is used instead).  Collected last on purpose."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from sparse_attention_indexer_tcgen05_gb300 import synth  # noqa: E402

GRAD_TOL = 2e-2   # the parity tests' gradient tolerance (relative L2)
LOSS_TOL = 2e-2   # the parity tests' bf16 loss tolerance (relative)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-300))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_noalloc_backward_matches_workspace_backward_twice():
    from sparse_attention_indexer_tcgen05_gb300 import binding as B
    from sparse_attention_indexer_tcgen05_gb300 import workload

    cfg = synth.Config("noalloc", "bshd", "bf16", 2, 1024, 4, 16, 64, 64, 128, 128, 64, seed=31)
    d = workload.to_device(synth.generate(cfg))
    p = d.params
    assert p.workspace_bytes <= B.NOALLOC_SCRATCH_BYTES
    ids, sel = B.csa_indexer_fwd(p, *d.indexer)
    ref = B.csa_indexer_bwd(p, *d.indexer, *d.teacher_side, ids, sel)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share (and reuse) the library's scratch
        got = B.csa_indexer_bwd_noalloc(p, *d.indexer, *d.teacher_side, ids, sel)
        torch.cuda.synchronize()
        assert abs(float(got[0]) - float(ref[0])) <= LOSS_TOL * abs(float(ref[0]))
        for g, r in zip(got[1:], ref[1:]):
            assert _rel(g, r) <= GRAD_TOL
    B.csa_check_device_status()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_noalloc_rejects_problems_beyond_the_scratch():
    from sparse_attention_indexer_tcgen05_gb300 import binding as B

    # the 64k long-context shape needs far more than the fixed scratch: refused before anything runs
    p = B.Params("bshd", "bf16", 1, 65536, 4, 128, 2048, 128, 512, 64, 128, 0.044)
    assert p.workspace_bytes > B.NOALLOC_SCRATCH_BYTES
    fake = [0x10000 * (i + 1) for i in range(13)]
    # q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore | teacher | loss | row_loss | dq_idx, dw, dk_idx | stream
    st = B._lib.csa_indexer_bwd_noalloc(p.ref, *fake[:9], None, fake[9], None, fake[10], fake[11], fake[12], None)
    assert st == 4  # CSA_ERR_WORKSPACE
