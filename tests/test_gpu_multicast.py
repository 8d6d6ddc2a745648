"""Operand multicast between CTA pairs (4-CTA clusters preferred) against plain
CTA pairs.

With cluster multicast on, a pair launch whose tiles pair up runs the walk in
which the two pairs of a 4-CTA cluster compute two tiles sharing one operand
and multicast it; any four CTAs the hardware groups as two 2-CTA clusters run
the same tiles without multicast.  Every output tile is still computed by one
pair over the same k-blocks in the same order with the same MMA shape, so the
results must equal the plain-pair results bit for bit.  The cases cover the
walks: row-block pairs sharing B (forward, dZ recompute, and dW / dX when the
column-block count is odd), column-block pairs sharing A (dW / dX), row-block
bands and vocabulary groups in the forward, and shapes that do not pair up
(which must fall back to plain pairs).
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, tensor_f64, to_device

pytestmark = pytest.mark.gpu


def _run(wl, mcast, chunk, **kw):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    X, W, y = to_device(wl)
    o = B.make_options(wl.spec.ignore_index, wl.spec.smoothing, cluster_multicast=mcast,
                       vocab_chunk=chunk, cta_pair=True, backward_merge=0, **kw)
    out = B.flce_fwd_bwd_ex(X, W, y, o)
    n_mc = B.last_multicast_launches()
    torch.cuda.synchronize()
    assert int(out[5].item()) == 0
    return out, n_mc


CASES = [
    # (N, H, V, chunk, n_ignore, smoothing, seed, multicast launches expected?)
    (1024, 512, 4096, 1024, 40, 0.1, 51, True),    # dW / dX: column-block pairs share A
    (1024, 768, 3000, 512, 30, 0.0, 52, True),     # 3 column blocks: row-block pairs share B
    (2048, 256, 5000, 1024, 0, 0.0, 53, True),     # ragged V, one column block for dW / dX
    (700, 136, 3000, 512, 20, 0.1, 54, False),     # 3 row blocks, 1 column block: no pairs
]


@pytest.mark.parametrize("case", CASES, ids=[f"N{c[0]}-H{c[1]}-V{c[2]}-cv{c[3]}" for c in CASES])
def test_multicast_equals_plain_pairs(case):
    import torch
    N, H, V, chunk, n_ign, eps, seed, expect_mc = case
    wl = I.make_workload(I.custom_spec("mcast", N=N, H=H, V=V, dtype="bf16", n_ignore=n_ign,
                                       smoothing=eps), seed=seed)
    a, n_a = _run(wl, True, chunk)
    b, n_b = _run(wl, False, chunk)
    assert n_b == 0
    assert (n_a > 0) == expect_mc, n_a
    for i, name in enumerate(("loss", "lse", "nv", "dX", "dW")):
        assert torch.equal(a[i], b[i]), name


def test_multicast_parity_with_oracle():
    wl = I.make_workload(I.custom_spec("mcast_parity", N=1024, H=768, V=3000, dtype="bf16",
                                       n_ignore=50, smoothing=0.1), seed=55)
    (loss, lse, nv, dX, dW, _), n_mc = _run(wl, True, 512, z_loss=1e-4)
    assert n_mc > 0
    f = O.forward(wl.x, wl.w, wl.labels, -100, 0.1, z_loss=1e-4)
    b = O.backward(wl.x, wl.w, wl.labels, -100, 0.1, z_loss=1e-4)
    assert int(nv.item()) == f.n_valid
    assert rel_err(float(loss.item()), f.loss) <= LOSS_REL
    assert np.max(np.abs(tensor_f64(lse) - f.lse)) <= LSE_ABS
    assert rel_fro(tensor_f64(dX), b.dX) <= GRAD_REL_FRO
    assert rel_fro(tensor_f64(dW), b.dW) <= GRAD_REL_FRO


def test_multicast_bands_and_vocab_groups():
    """Forward with two row-block bands (X > 48 MiB) and vocabulary groups of
    two tiles (partials > 32 MiB); both walks give the same bits."""
    import torch
    wl = I.make_workload(I.custom_spec("mcast_bands", N=100352, H=256, V=6000, dtype="bf16",
                                       n_ignore=300), seed=56)
    a, n_a = _run(wl, True, 1024)
    b, _ = _run(wl, False, 1024)
    assert n_a > 0
    for i, name in enumerate(("loss", "lse", "nv", "dX", "dW")):
        assert torch.equal(a[i], b[i]), name


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("shape", [(512, 1024, 384), (1024, 768, 200)],
                         ids=["share_a", "share_b"])
def test_gemm_core_multicast_layouts(a_mn, b_mn, shape):
    """The GEMM core alone: both operand layouts on both sides, with column-block
    pairs sharing A (4 column blocks) or row-block pairs sharing B (3 column
    blocks), against plain pairs and against torch."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    M, Nn, K = shape
    g = torch.Generator().manual_seed(57)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    Bm = torch.randn(Nn, K, generator=g).to(torch.bfloat16).cuda()
    a_in = A.t().contiguous() if a_mn else A
    b_in = Bm.t().contiguous() if b_mn else Bm
    outs = []
    try:
        for on in (True, False):
            B.flce_set_cluster_multicast(on)
            D, err = B.flce_debug_gemm(a_in, b_in, M, Nn, K, bool(a_mn), bool(b_mn))
            n_mc = B.last_multicast_launches()
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert (n_mc > 0) == on
            outs.append(D.cpu())
    finally:
        B.flce_set_cluster_multicast(True)
    assert torch.equal(outs[0], outs[1])
    ref = A.float().cpu() @ Bm.float().cpu().t()
    assert torch.allclose(outs[0], ref, rtol=1e-3, atol=1e-2)
