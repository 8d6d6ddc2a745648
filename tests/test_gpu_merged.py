"""The merged backward launch against the three-launch backward.

With merging on (flce_set_backward_merge(1)) the backward runs the dZ recompute of chunk 0
alone and then one launch per vocabulary chunk holding the dW and dX GEMMs of
that chunk and the dZ recompute of the next, with tiles taken from one list.
Every output tile is computed by one CTA pair over the same k-blocks in the same
order as in the separate launches, so at the same chunk width the two paths
must agree bit for bit.  The cases cover several chunks (both dZ buffers used
in turn), launches handed out wholly dynamically and launches with round-robin
rounds first, ragged N, H and V tails, H below one tile, smoothing, z-loss, sum
reduction with an upstream gradient, dW accumulation, fp32 inputs and the
vocabulary-parallel backward, and one parity case against the oracle.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_cta_pair(1)
    yield
    B.flce_set_backward_merge(0)
    B.flce_set_vocab_chunk(0)
    B.flce_set_cta_pair(1)


def _run(wl, merge, chunk, reduction="mean", grad=None, dW0=None, z_loss=0.0):
    """merge: 0 three launches per chunk, 1 dW(c) + dX(c) + dZ(c+1) merged,
    2 dZ(c) alone then dW(c) + dX(c) merged."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_backward_merge(merge)
    B.flce_set_vocab_chunk(chunk)
    assert B.flce_vocab_chunk(wl.N, wl.spec.H, wl.spec.V) == chunk  # same Cv on both paths
    X, W, y = to_device(wl)
    g = None if grad is None else torch.tensor([grad], dtype=torch.float32, device="cuda")
    dW = None if dW0 is None else torch.from_numpy(dW0).cuda()
    B.flce_profile_reset()
    B.flce_profile_enable(True)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(
        X, W, y, wl.spec.ignore_index, wl.spec.smoothing, reduction, grad_loss=g, dW=dW,
        accumulate_dW=dW0 is not None, z_loss=z_loss)
    torch.cuda.synchronize()
    B.flce_profile_enable(False)
    prof = B.flce_profile_read()
    assert int(err.item()) == 0
    return dict(loss=loss.cpu(), lse=lse.cpu(), nv=nv.cpu(), dX=dX.cpu(), dW=dW.cpu()), prof


CASES = [
    # (N, H, V, n_ignore, smoothing, z_loss, chunk, dtype, seed)
    (700, 136, 5000, 40, 0.1, 1e-4, 1024, "bf16", 31),   # 5 chunks, H < one tile, ragged V
    (513, 264, 3000, 0, 0.0, 0.0, 512, "bf16", 32),       # 6 chunks, ragged H and N
    (1024, 512, 2560, 100, 0.0, 0.0, 256, "bf16", 33),    # 10 chunks of one tile each
    (300, 128, 3200, 10, 0.05, 0.0, 768, "fp32", 34),     # fp32 inputs, 5 chunks
    (2304, 1024, 9000, 64, 0.0, 1e-3, 2048, "bf16", 35),  # 140 tiles per launch, all dynamic
    # enough tiles per launch (384, 320) for round-robin rounds before the
    # dynamically handed-out last rounds
    (4096, 1024, 20000, 0, 0.0, 0.0, 4096, "bf16", 39),
    (6000, 1024, 16000, 100, 0.1, 1e-4, 2048, "bf16", 40),
    # degenerate: one chunk (a merged launch with no dZ tiles), one token
    (300, 128, 200, 20, 0.1, 0.0, 256, "bf16", 42),
    (1, 64, 1000, 0, 0.0, 0.0, 256, "bf16", 43),
]


@pytest.mark.parametrize("mode", [1, 2], ids=["dw_dx_dznext", "dw_dx"])
@pytest.mark.parametrize("case", CASES, ids=[f"N{c[0]}-H{c[1]}-V{c[2]}-cv{c[6]}-{c[7]}"
                                              for c in CASES])
def test_merged_equals_separate_launches(case, mode):
    import torch
    N, H, V, n_ign, eps, zl, chunk, dt, seed = case
    spec = I.custom_spec("merged", N=N, H=H, V=V, dtype=dt, n_ignore=n_ign, smoothing=eps)
    wl = I.make_workload(spec, seed=seed)
    a, pa = _run(wl, mode, chunk, z_loss=zl)
    b, pb = _run(wl, 0, chunk, z_loss=zl)
    n_chunks = -(-V // chunk)
    # the merged kernel ran once per chunk and no separate dW / dX launch did;
    # the dZ recompute ran alone for chunk 0 (mode 1) or for every chunk (mode 2)
    assert pa["bwd_merged"][1] == n_chunks
    assert pa["bwd_dz_recompute"][1] == (1 if mode == 1 else n_chunks)
    assert pa["bwd_dw_gemm"][1] == 0 and pa["bwd_dx_gemm"][1] == 0
    assert pb["bwd_merged"][1] == 0 and pb["bwd_dw_gemm"][1] == n_chunks
    for k in ("loss", "lse", "nv", "dX", "dW"):
        assert torch.equal(a[k], b[k]), k
    assert float(a["dW"].abs().sum()) > 0 and float(a["dX"].float().abs().sum()) > 0


@pytest.mark.parametrize("mode", [1, 2], ids=["dw_dx_dznext", "dw_dx"])
def test_merged_sum_reduction_and_dw_accumulation(mode):
    import torch
    spec = I.custom_spec("merged_acc", N=600, H=192, V=3300, dtype="bf16", n_ignore=25)
    wl = I.make_workload(spec, seed=36)
    dW0 = np.random.default_rng(7).standard_normal((3300, 192)).astype(np.float32)
    a, _ = _run(wl, mode, 512, reduction="sum", grad=0.37, dW0=dW0)
    b, _ = _run(wl, False, 512, reduction="sum", grad=0.37, dW0=dW0)
    for k in ("loss", "lse", "dX", "dW"):
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["dW"], torch.from_numpy(dW0))


def test_merged_vocab_shard_backward():
    """Vocabulary-parallel backward (fp32 partial dX, shard's dW rows) through
    both paths, for the second of two shards (non-zero vocabulary offset)."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    spec = I.custom_spec("merged_shard", N=500, H=256, V=4000, dtype="bf16", n_ignore=20,
                         smoothing=0.1)
    wl = I.make_workload(spec, seed=37)
    X, W, y = to_device(wl)
    opt = B.make_options(smoothing=0.1, z_loss=1e-4)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(X, W, y, -100, 0.1, "mean", z_loss=1e-4)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    outs = []
    for merge in (1, 2, 0):
        B.flce_set_backward_merge(merge)
        B.flce_set_vocab_chunk(512)
        assert B.flce_vocab_chunk(500, 256, 2200) == 512
        dxp, dwp, e = B.flce_backward_vocab_shard(X, W[1800:], y, 1800, 4000, lse, nv, opt)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        outs.append((dxp.cpu(), dwp.cpu()))
    for o in outs[1:]:
        assert torch.equal(outs[0][0], o[0]) and torch.equal(outs[0][1], o[1])


def test_optional_features_take_the_separate_launches():
    """skip_ignored_blocks needs the feature-carrying kernels: no merged launch."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    spec = I.custom_spec("merged_skip", N=600, H=128, V=2000, dtype="bf16", n_ignore=0)
    wl = I.make_workload(spec, seed=38)
    X, W, y = to_device(wl)
    y[:256] = -100
    B.flce_set_vocab_chunk(256)
    B.flce_profile_reset()
    B.flce_profile_enable(True)
    out = B.flce_fwd_bwd(X, W, y, skip_ignored_blocks=True)
    torch.cuda.synchronize()
    B.flce_profile_enable(False)
    prof = B.flce_profile_read()
    assert int(out[-1].item()) == 0
    assert prof["bwd_merged"][1] == 0 and prof["bwd_dw_gemm"][1] == 8


def test_merged_parity_with_oracle():
    """The merged path against the fp64 oracle (not only against the other
    path): several chunks, ragged tails, smoothing and z-loss."""
    from oracle import flce_oracle as O
    from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro
    spec = I.custom_spec("merged_parity", N=700, H=200, V=3000, dtype="bf16", n_ignore=30,
                         smoothing=0.1)
    wl = I.make_workload(spec, seed=41)
    got, prof = _run(wl, True, 512, z_loss=1e-4)
    assert prof["bwd_merged"][1] == 6
    f = O.forward(wl.x, wl.w, wl.labels, -100, 0.1, "mean", z_loss=1e-4)
    b = O.backward(wl.x, wl.w, wl.labels, -100, 0.1, "mean", z_loss=1e-4)
    assert int(got["nv"].item()) == f.n_valid
    assert rel_err(float(got["loss"].item()), f.loss) <= LOSS_REL
    assert np.max(np.abs(got["lse"].double().numpy() - f.lse)) <= LSE_ABS
    assert rel_fro(got["dX"].double().numpy(), b.dX) <= GRAD_REL_FRO
    assert rel_fro(got["dW"].double().numpy(), b.dW) <= GRAD_REL_FRO


@pytest.mark.slow
def test_merged_equals_separate_launches_full_size():
    """At the Llama-3 benchmark shape (N=8192, H=4096, V=128256) and Cv = 4096,
    where merging pays: 32 merged launches of up to 1280 tiles, most of them round
    robin, the last rounds handed out dynamically; same bits as three
    launches per chunk."""
    import torch
    wl = I.make_workload(I.CONFIGS["llama3_n8192"], seed=0)
    a, pa = _run(wl, True, 4096)
    b, pb = _run(wl, False, 4096)
    assert pa["bwd_merged"][1] == 32 and pb["bwd_dw_gemm"][1] == 32
    for k in ("loss", "lse", "nv", "dX", "dW"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.slow
def test_dw_dx_merged_equals_separate_launches_full_size():
    """At the Llama-3 benchmark shape with the default chunk width (14592: 8
    chunks and a last one of 11520): dZ(c) alone, then dW(c) and dX(c) from
    one tile list of 912 + 512 tiles; same bits as three launches per chunk."""
    import torch
    wl = I.make_workload(I.CONFIGS["llama3_n8192"], seed=0)
    a, pa = _run(wl, 2, 14592)
    b, pb = _run(wl, 0, 14592)
    assert pa["bwd_merged"][1] == 9 and pa["bwd_dz_recompute"][1] == 9
    for k in ("loss", "lse", "nv", "dX", "dW"):
        assert torch.equal(a[k], b[k]), k
