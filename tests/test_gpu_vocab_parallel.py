"""Vocabulary-parallel layout, its shards emulated one after another on one GPU.

Each shard runs flce_forward_vocab_shard on its rows of W; the partials are
stacked (the exchange) and combined with flce_combine_vocab_shards; each
shard's flce_backward_vocab_shard gives a partial dX (summed over shards, the
all-reduce) and its own dW rows.  Checked against the fp64 oracle and against
the unsharded path.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, tensor_f64, to_device

pytestmark = pytest.mark.gpu


def run_sharded(wl, bounds, z_loss=0.0, reduction="mean"):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    X, W, y = to_device(wl)
    V = wl.V
    opt = B.make_options(wl.spec.ignore_index, wl.spec.smoothing, reduction, z_loss)
    parts = []
    for v0, v1 in zip(bounds, bounds[1:]):
        part, err = B.flce_forward_vocab_shard(X, W[v0:v1], y, v0, V, opt)
        parts.append(part)
    allp = torch.stack(parts)  # [P, N, 4]: the exchange
    loss, lse, nv, err_c = B.flce_combine_vocab_shards(allp, y, V, opt)
    dX = torch.zeros(wl.N, wl.H, dtype=torch.float32, device="cuda")
    dWs = []
    for v0, v1 in zip(bounds, bounds[1:]):
        dxp, dwp, err_b = B.flce_backward_vocab_shard(X, W[v0:v1], y, v0, V, lse, nv, opt)
        dX += dxp  # the all-reduce
        dWs.append(dwp)
    torch.cuda.synchronize()
    return dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
                dX=tensor_f64(dX), dW=tensor_f64(torch.cat(dWs)),
                err=int(err.item()) | int(err_c.item()) | int(err_b.item()))


def check(wl, got, z_loss=0.0, reduction="mean"):
    ii, eps = wl.spec.ignore_index, wl.spec.smoothing
    f, b = O.fwd_bwd(wl.x, wl.w, wl.labels, ii, eps, reduction, z_loss=z_loss)
    assert got["err"] == 0 and got["nv"] == f.n_valid
    assert rel_err(got["loss"], f.loss) <= LOSS_REL
    assert np.max(np.abs(got["lse"] - f.lse)) <= LSE_ABS
    assert rel_fro(got["dX"], b.dX) <= GRAD_REL_FRO
    assert rel_fro(got["dW"], b.dW) <= GRAD_REL_FRO


@pytest.mark.parametrize("pair", [1, 0], ids=["cta_pair", "single_cta"])
def test_three_uneven_shards(pair):
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_cta_pair(pair)
    try:
        wl = I.make_workload(I.custom_spec("vp", N=700, H=192, V=5000, dtype="bf16", n_ignore=40,
                                           smoothing=0.1, w_std=0.05), seed=40)
        check(wl, run_sharded(wl, [0, 1700, 3400, 5000], z_loss=1e-3), z_loss=1e-3)
    finally:
        B.flce_set_cta_pair(1)


def test_tiny_shard_and_sum_reduction():
    wl = I.make_workload(I.custom_spec("vp", N=300, H=64, V=1029, dtype="bf16", n_ignore=10,
                                       labels="zipf"), seed=41)
    check(wl, run_sharded(wl, [0, 5, 1029], reduction="sum"), reduction="sum")


def test_fp32_inputs_two_shards():
    wl = I.make_workload("tiny", seed=0)
    check(wl, run_sharded(wl, [0, 2048, 4096]))


def test_sharded_equals_unsharded():
    from linear_cross_entropy_logit_gb300 import binding as B
    import torch
    wl = I.make_workload(I.custom_spec("vp", N=512, H=128, V=3000, dtype="bf16", n_ignore=30,
                                       smoothing=0.1), seed=42)
    got = run_sharded(wl, [0, 1024, 3000])
    X, W, y = to_device(wl)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(X, W, y, -100, 0.1)
    torch.cuda.synchronize()
    assert rel_err(got["loss"], loss.item()) <= 1e-5
    assert np.max(np.abs(got["lse"] - tensor_f64(lse))) <= 1e-4
    assert rel_fro(got["dX"], tensor_f64(dX)) <= 5e-3
    assert rel_fro(got["dW"], tensor_f64(dW)) <= 5e-3
