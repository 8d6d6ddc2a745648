"""Operand multicast between CTA pairs against plain CTA pairs.

With cluster multicast on, a pair launch whose tiles group exactly walks them
in groups of G pairs (G = 4 with 8-CTA clusters preferred, else G = 2 with
4-CTA clusters preferred) that compute G tiles sharing one operand and
multicast it; CTAs the hardware places in smaller clusters share with fewer
pairs or none.  Every output tile is still computed by one pair over the same
k-blocks in the same order with the same MMA shape, so every mode must equal
the plain-pair results bit for bit.  The cases cover groups of four and of two
pairs, sharing A and sharing B, the shared operand K-major (cut into 32-row
pieces for groups of four) and MN-major (cut into 16-k-row pieces), row-block
bands and vocabulary groups in the forward, and shapes that group in no way
(which must fall back to plain pairs).
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, tensor_f64, to_device

pytestmark = pytest.mark.gpu


def _run(wl, mode, chunk, **kw):
    """mode: 0 plain pairs, 1 groups of up to four pairs, 2 groups of two pairs.
    Returns the outputs and the launches that took groups of (2, 4) pairs."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    X, W, y = to_device(wl)
    o = B.make_options(wl.spec.ignore_index, wl.spec.smoothing, cluster_multicast=mode,
                       vocab_chunk=chunk, cta_pair=True, backward_merge=0, **kw)
    out = B.flce_fwd_bwd_ex(X, W, y, o)
    n = (B.last_multicast_launches(2), B.last_multicast_launches(4))
    torch.cuda.synchronize()
    assert int(out[5].item()) == 0
    return out, n


CASES = [
    # (N, H, V, chunk, n_ignore, smoothing, seed, groups of 4 expected, groups of 2 expected)
    # 4 row blocks, 4 column blocks: groups of four everywhere; dW and dX share A
    (1024, 1024, 4096, 1024, 40, 0.1, 51, True, False),
    # 3 column blocks: dW and dX group row blocks in fours and share B (MN-major pieces)
    (2048, 768, 3000, 1024, 30, 0.0, 52, True, False),
    # 6 row blocks, 2 column blocks: only groups of two
    (1536, 512, 3000, 512, 0, 0.0, 53, False, True),
    # 3 row blocks, 1 column block: no groups at all
    (700, 136, 3000, 512, 20, 0.1, 54, False, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"N{c[0]}-H{c[1]}-V{c[2]}-cv{c[3]}" for c in CASES])
def test_multicast_equals_plain_pairs(case):
    import torch
    N, H, V, chunk, n_ign, eps, seed, want4, want2 = case
    wl = I.make_workload(I.custom_spec("mcast", N=N, H=H, V=V, dtype="bf16", n_ignore=n_ign,
                                       smoothing=eps), seed=seed)
    base, n0 = _run(wl, 0, chunk)
    assert n0 == (0, 0)
    up_to_4, n1 = _run(wl, 1, chunk)
    pairs_of_2, n2 = _run(wl, 2, chunk)
    assert (n1[1] > 0) == want4 and (n1[0] > 0) == want2, n1
    assert n2[1] == 0 and (n2[0] > 0) == (want4 or want2), n2
    for out in (up_to_4, pairs_of_2):
        for i, name in enumerate(("loss", "lse", "nv", "dX", "dW")):
            assert torch.equal(out[i], base[i]), name


def test_multicast_parity_with_oracle():
    """Groups of four pairs sharing B (MN-major for dW and dX) against the oracle."""
    wl = I.make_workload(I.custom_spec("mcast_parity", N=2048, H=768, V=3000, dtype="bf16",
                                       n_ignore=50, smoothing=0.1), seed=55)
    (loss, lse, nv, dX, dW, _), n = _run(wl, 1, 1024, z_loss=1e-4)
    assert n[1] > 0
    f = O.forward(wl.x, wl.w, wl.labels, -100, 0.1, z_loss=1e-4)
    b = O.backward(wl.x, wl.w, wl.labels, -100, 0.1, z_loss=1e-4)
    assert int(nv.item()) == f.n_valid
    assert rel_err(float(loss.item()), f.loss) <= LOSS_REL
    assert np.max(np.abs(tensor_f64(lse) - f.lse)) <= LSE_ABS
    assert rel_fro(tensor_f64(dX), b.dX) <= GRAD_REL_FRO
    assert rel_fro(tensor_f64(dW), b.dW) <= GRAD_REL_FRO


def test_multicast_bands_and_vocab_groups():
    """Forward with two row-block bands (X > 48 MiB) and vocabulary groups of
    two tiles (partials > 32 MiB), walked in groups of four row blocks; every
    mode gives the same bits."""
    import torch
    wl = I.make_workload(I.custom_spec("mcast_bands", N=100352, H=256, V=6000, dtype="bf16",
                                       n_ignore=300), seed=56)
    base, _ = _run(wl, 0, 1024)
    up_to_4, n1 = _run(wl, 1, 1024)
    pairs_of_2, n2 = _run(wl, 2, 1024)
    assert n1[1] > 0 and n2[0] > 0
    for out in (up_to_4, pairs_of_2):
        for i, name in enumerate(("loss", "lse", "nv", "dX", "dW")):
            assert torch.equal(out[i], base[i]), name


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("shape,group", [((512, 1024, 384), 4), ((1024, 768, 200), 4),
                                         ((512, 512, 256), 2)],
                         ids=["share_a_4", "share_b_4", "share_a_2"])
def test_gemm_core_multicast_layouts(a_mn, b_mn, shape, group):
    """The GEMM core alone: both operand layouts on both sides, groups of four
    pairs sharing A (4 column blocks) or B (3 column blocks, 4 row blocks) and
    groups of two, against plain pairs and against torch."""
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
        for mode in (1, 0):
            B.flce_set_cluster_multicast(mode)
            D, err = B.flce_debug_gemm(a_in, b_in, M, Nn, K, bool(a_mn), bool(b_mn))
            n_g = B.last_multicast_launches(group)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert (n_g > 0) == (mode == 1)
            outs.append(D.cpu())
    finally:
        B.flce_set_cluster_multicast(1)
    assert torch.equal(outs[0], outs[1])
    ref = A.float().cpu() @ Bm.float().cpu().t()
    assert torch.allclose(outs[0], ref, rtol=1e-3, atol=1e-2)
