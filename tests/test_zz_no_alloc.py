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

    # a larger problem with other values goes through the scratch first, so that anything the backward read from
    # the scratch without writing it first would differ from the workspace reference below
    other = synth.Config("noalloc_other", "bshd", "bf16", 2, 3000, 4, 16, 64, 64, 128, 256, 64, seed=37)
    do = workload.to_device(synth.generate(other))
    assert do.params.workspace_bytes <= B.NOALLOC_SCRATCH_BYTES
    ids_o, sel_o = B.csa_indexer_fwd(do.params, *do.indexer)
    B.csa_indexer_bwd_noalloc(do.params, *do.indexer, *do.teacher_side, ids_o, sel_o)
    torch.cuda.synchronize()
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
