"""Parity at the full workload sizes, in the launch configuration bench.py times.

One flce_fwd_bwd call per workload (default vocabulary chunk).  Against the
fp64 oracle:
  * the loss and the lse of every token row (the oracle's full forward);
  * dX on sampled token rows, ignored rows included (exactly zero there): the
    first and last row of every row-block band the forward and dZ launches
    walk (and an ignored row inside each band), the last row N-1, and random
    rows;
  * dW on sampled vocabulary rows: the first and last row of every vocabulary
    chunk of the backward (the partial last chunk included), the most
    frequent labels, random rows, and for the Gemma-shaped workload the
    x8-scaled rows nearest a chunk edge and some others, each computed by the
    oracle one by one from its own lse;
  * the property sum_j dW_j = 0 (with z-loss: sum_i 2 c alpha lse_i x_i) on
    the whole GPU dW, relative to sum_j |dW_j|.
Each case takes from ~20 s (Llama shape) to ~2 min (Gemma shape) of oracle time
on the host.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, to_device

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WORKLOADS = [("llama3_n8192", 0.0), ("llama3_long_n16384", 0.0), ("qwen25_n16384", 0.0),
             ("gemma2_n32768", 0.0), ("llama3_n8192", 1e-4)]


def band_edge_rows(N, H, labels, ii):
    """Token rows at the edges of the row-block bands the forward and dZ
    launches walk (X above 48 MiB is split into ceil(X / 40 MiB) bands of
    256-row blocks, at most 4), plus one ignored row inside each band."""
    blocks = -(-N // 256)
    x_bytes = N * H * 2
    bands = min(4, -(-x_bytes // (40 << 20))) if x_bytes > (48 << 20) else 1
    per = -(-blocks // bands) * 256
    rows = []
    for b0 in range(0, N, per):
        b1 = min(N, b0 + per)
        rows += [b0, b1 - 1]
        ign = np.flatnonzero(labels[b0:b1] == ii)
        if ign.size:
            rows.append(b0 + int(ign[len(ign) // 2]))
    return rows + [N - 1]


def chunk_edge_rows(V, cv):
    """First and last vocabulary row of every backward chunk of width cv."""
    rows = []
    for v0 in range(0, V, cv):
        rows += [v0, min(V, v0 + cv) - 1]
    return rows


@pytest.mark.parametrize("name,z_loss", WORKLOADS,
                         ids=[n + (f"-zloss{z:g}" if z else "") for n, z in WORKLOADS])
def test_full_size_parity(name, z_loss):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B

    B.flce_set_vocab_chunk(0)
    spec = I.CONFIGS[name]
    wl = I.make_workload(spec, seed=0)
    N, V = spec.N, spec.V
    ii, eps = spec.ignore_index, spec.smoothing
    X, W, y = to_device(wl)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(X, W, y, ii, eps, spec.reduction,
                                                z_loss=z_loss)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got_lse = lse.double().cpu().numpy()

    rng = np.random.default_rng(1234)
    ignored = np.flatnonzero(wl.labels == ii)
    rows = np.unique(np.concatenate([ignored[:8], rng.choice(N, 56, replace=False),
                                     band_edge_rows(N, spec.H, wl.labels, ii)]))
    labels_valid = wl.labels[wl.labels != ii]
    counts = np.bincount(labels_valid, minlength=V)
    cv = B.flce_vocab_chunk(N, spec.H, V)
    edges = np.array(chunk_edge_rows(V, cv))
    vrows = [np.argsort(-counts)[:8], rng.choice(V, 40, replace=False), edges]
    if spec.n_scaled_w_rows:
        scaled = I._rng(0, 5).permutation(V)[:spec.n_scaled_w_rows]
        # the scaled rows nearest a chunk edge, and a few others
        dist = np.min(np.abs(scaled[:, None] - edges[None, :]), axis=1)
        vrows += [scaled[np.argsort(dist)[:8]], scaled[:8]]
    vrows = np.unique(np.concatenate(vrows))
    got_dx = dX[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    got_dw = dW[torch.from_numpy(vrows).cuda()].double().cpu().numpy()
    # sum_j dW_j on the whole GPU output (0, or sum_i 2 c alpha lse_i x_i with
    # z-loss), relative to sum_j |dW_j|
    col_sum = dW.double().sum(dim=0).cpu().numpy()
    row_norm_sum = dW.double().norm(dim=1).sum().item()
    del X, W, dX, dW
    torch.cuda.empty_cache()

    f = O.forward(wl.x, wl.w, wl.labels, ii, eps, spec.reduction, z_loss=z_loss)
    assert int(nv.item()) == f.n_valid
    assert rel_err(loss.item(), f.loss) <= LOSS_REL, (loss.item(), f.loss)
    assert np.max(np.abs(got_lse - f.lse)) <= LSE_ABS
    c = O.grad_scale(f.n_valid, spec.reduction)
    want_dx = O.dx_rows(wl.x, wl.w, wl.labels, rows, c, ii, eps, z_loss)
    assert rel_fro(got_dx, want_dx) <= GRAD_REL_FRO
    assert np.all(got_dx[np.isin(rows, ignored)] == 0.0)
    want_dw = O.dw_rows(wl.x, wl.w, wl.labels, vrows, f.lse, c, ii, eps, z_loss)
    assert rel_fro(got_dw, want_dw) <= GRAD_REL_FRO
    valid = (wl.labels != ii).astype(np.float64)
    want_col = 2.0 * c * z_loss * (valid * f.lse) @ O.upcast(wl.x) if z_loss else 0.0
    assert np.linalg.norm(col_sum - want_col) / row_norm_sum <= 1e-3
