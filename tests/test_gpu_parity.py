"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Element-by-element comparisons on seeded inputs that span several tiles and
ragged tails in every dimension, plus the method's edge cases: masking,
smoothing, sum reduction with an upstream gradient, dW accumulation, all
tokens ignored, N = 0, N = 1, a vocabulary smaller than one tile, an invalid
label, logits far above the fp32 exp overflow point, and token shards that
compose to the whole batch.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import (GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, tensor_f64,
                            to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _auto_chunk():
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_vocab_chunk(0)
    B.flce_set_cta_pair(1)
    yield
    B.flce_set_vocab_chunk(0)
    B.flce_set_cta_pair(1)


def run_fwd_bwd(wl, reduction="mean", grad=None, chunk=0, dW0=None, z_loss=0.0,
                row_loss=False, skip=False):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_vocab_chunk(chunk)
    X, W, y = to_device(wl)
    g = None if grad is None else torch.tensor([grad], dtype=torch.float32, device="cuda")
    dW = None if dW0 is None else torch.from_numpy(dW0.astype(np.float32)).cuda()
    rl = torch.full((wl.N,), float("nan"), device="cuda") if row_loss else None
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(
        X, W, y, wl.spec.ignore_index, wl.spec.smoothing, reduction, grad_loss=g, dW=dW,
        accumulate_dW=dW0 is not None, z_loss=z_loss, row_loss=rl, skip_ignored_blocks=skip)
    torch.cuda.synchronize()
    out = dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
               dX=tensor_f64(dX), dW=tensor_f64(dW), err=int(err.item()))
    if row_loss:
        out["row_loss"] = tensor_f64(rl)
    return out


def check_against_oracle(wl, got, reduction="mean", grad=1.0, dW0=None, z_loss=0.0,
                         lse_rows="all"):
    f = O.forward(wl.x, wl.w, wl.labels, wl.spec.ignore_index, wl.spec.smoothing, reduction,
                  z_loss=z_loss)
    b = O.backward(wl.x, wl.w, wl.labels, wl.spec.ignore_index, wl.spec.smoothing, reduction,
                   grad_loss=grad, dW_in=dW0, z_loss=z_loss)
    assert got["err"] == 0
    assert got["nv"] == f.n_valid
    assert rel_err(got["loss"], f.loss) <= LOSS_REL, (got["loss"], f.loss)
    if wl.N:
        keep = np.isfinite(got["lse"]) if lse_rows == "finite" else slice(None)
        assert np.max(np.abs(got["lse"][keep] - f.lse[keep])) <= LSE_ABS
        assert rel_fro(got["dX"], b.dX) <= GRAD_REL_FRO
    assert rel_fro(got["dW"], b.dW) <= GRAD_REL_FRO
    return f, b


def spec(**kw):
    kw.setdefault("dtype", "bf16")
    return I.custom_spec("case", **kw)


def test_tiny_config_fp32():
    wl = I.make_workload("tiny", seed=0)
    check_against_oracle(wl, run_fwd_bwd(wl))


@pytest.mark.parametrize("pair", [1, 0], ids=["cta_pair", "single_cta"])
@pytest.mark.parametrize("chunk", [0, 256, 512])
def test_ragged_multi_tile(chunk, pair):
    # 3 row blocks (last ragged), 4 vocabulary tiles (last ragged), K tail of 8
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_cta_pair(pair)
    wl = I.make_workload(spec(N=300, H=136, V=1000, n_ignore=30, smoothing=0.1), seed=1)
    check_against_oracle(wl, run_fwd_bwd(wl, chunk=chunk))


def test_tile_shapes_agree():
    """CTA-pair and single-CTA tiles give the same results up to fp32 summation order."""
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=700, H=264, V=3000, n_ignore=50, smoothing=0.1), seed=15)
    B.flce_set_cta_pair(1)
    a = run_fwd_bwd(wl)
    B.flce_set_cta_pair(0)
    b = run_fwd_bwd(wl)
    assert rel_err(a["loss"], b["loss"]) <= 1e-5
    assert np.max(np.abs(a["lse"] - b["lse"])) <= 1e-4
    assert rel_fro(a["dX"], b["dX"]) <= 5e-3 and rel_fro(a["dW"], b["dW"]) <= 5e-3


def test_sum_reduction_with_upstream_grad():
    wl = I.make_workload(spec(N=257, H=64, V=777, n_ignore=20, smoothing=0.05), seed=2)
    got = run_fwd_bwd(wl, reduction="sum", grad=0.37)
    check_against_oracle(wl, got, reduction="sum", grad=0.37)


def test_accumulate_dw():
    wl = I.make_workload(spec(N=200, H=96, V=600, n_ignore=10), seed=3)
    dW0 = np.random.default_rng(4).standard_normal((600, 96)) * 1e-3
    got = run_fwd_bwd(wl, dW0=dW0)
    check_against_oracle(wl, got, dW0=dW0.astype(np.float32).astype(np.float64))


def test_separate_calls_match_fused():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=384, H=128, V=1500, n_ignore=40, smoothing=0.1), seed=5)
    X, W, y = to_device(wl)
    loss, lse, nv, err = B.flce_forward(X, W, y, -100, 0.1)
    dX, dW, err2 = B.flce_backward(X, W, y, lse, nv, -100, 0.1)
    torch.cuda.synchronize()
    fused = run_fwd_bwd(wl)
    assert int(err.item()) == 0 and int(err2.item()) == 0
    assert float(loss.item()) == fused["loss"]
    assert np.array_equal(tensor_f64(lse), fused["lse"])
    assert np.array_equal(tensor_f64(dX), fused["dX"])
    assert np.array_equal(tensor_f64(dW), fused["dW"])


def test_deterministic_repeat():
    wl = I.make_workload(spec(N=512, H=256, V=3000, n_ignore=50, smoothing=0.1), seed=6)
    a = run_fwd_bwd(wl)
    b = run_fwd_bwd(wl)
    assert a["loss"] == b["loss"]
    for k in ("lse", "dX", "dW"):
        assert np.array_equal(a[k], b[k])


def test_all_ignored():
    wl = I.make_workload(spec(N=130, H=64, V=300, n_ignore=130, smoothing=0.1), seed=7)
    got = run_fwd_bwd(wl)
    assert got["err"] == 0 and got["nv"] == 0 and got["loss"] == 0.0
    assert np.all(got["dX"] == 0.0) and np.all(got["dW"] == 0.0)
    f = O.forward(wl.x, wl.w, wl.labels, -100, 0.1)
    assert np.max(np.abs(got["lse"] - f.lse)) <= LSE_ABS


def test_empty_batch():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(300, 64, device="cuda").to(torch.bfloat16)
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    dW = torch.full((300, 64), 7.0, device="cuda")
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(X, W, y, dW=dW)
    torch.cuda.synchronize()
    assert float(loss.item()) == 0.0 and int(nv.item()) == 0 and int(err.item()) == 0
    assert torch.all(dW == 0)


def test_single_token():
    wl = I.make_workload(spec(N=1, H=32, V=700), seed=8)
    check_against_oracle(wl, run_fwd_bwd(wl))


def test_vocab_smaller_than_a_tile():
    wl = I.make_workload(spec(N=70, H=48, V=5, n_ignore=3, smoothing=0.2, w_std=0.5), seed=9)
    check_against_oracle(wl, run_fwd_bwd(wl))


def test_invalid_label_sets_error_word():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=64, H=32, V=100), seed=10)
    wl.labels[5] = 100
    X, W, y = to_device(wl)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd(X, W, y)
    torch.cuda.synchronize()
    assert int(err.item()) == B.FLCE_ERR_LABEL
    assert int(nv.item()) == 63


BAD_LABELS = {5: "V", 300: -1, 599: "V+7"}


@pytest.mark.parametrize("path", ["three_launch", "merged", "vocab_shard"])
def test_invalid_labels_count_as_ignored(path):
    """A label outside [0, V) that is not ignore_index sets FLCE_ERR_LABEL and
    its row counts as ignored in the forward AND the backward: loss, lse, dX
    and dW equal the oracle's on the same labels with those entries replaced
    by ignore_index, and the bad rows of dX are exactly zero ("Fused
    cross-entropy -- the memory kernel", "Numerical traps": the ignore_index
    mask folded into the fused pass)."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    V = 1000
    wl = I.make_workload(spec(N=600, H=136, V=V, n_ignore=30, smoothing=0.1), seed=23)
    bad = np.array(sorted(BAD_LABELS))
    for r, v in BAD_LABELS.items():
        wl.labels[r] = {"V": V, "V+7": V + 7}.get(v, v)
    ref_labels = wl.labels.copy()
    ref_labels[bad] = -100
    X, W, y = to_device(wl)
    eps = wl.spec.smoothing
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if path == "vocab_shard":
        opt = B.make_options(-100, eps)
        bounds = [0, 512, V]
        parts = torch.empty(2, wl.N, 4, dtype=torch.float32, device="cuda")
        for i, (b0, b1) in enumerate(zip(bounds, bounds[1:])):
            B.flce_forward_vocab_shard(X, W[b0:b1].contiguous(), y, b0, V, opt,
                                       partials=parts[i], err_word=err)
        loss, lse, nv, _ = B.flce_combine_vocab_shards(parts, y, V, opt, err_word=err)
        dX = torch.zeros(wl.N, wl.H, dtype=torch.float32, device="cuda")
        dWs = []
        for b0, b1 in zip(bounds, bounds[1:]):
            dxp, dws, _ = B.flce_backward_vocab_shard(X, W[b0:b1].contiguous(), y, b0, V, lse,
                                                      nv, opt, err_word=err)
            dX += dxp
            dWs.append(dws)
        dW = torch.cat(dWs)
    else:
        merged = path == "merged"
        opt = B.make_options(-100, eps, backward_merge=merged, vocab_chunk=256 if merged else 0)
        loss, lse, nv, dX, dW, _ = B.flce_fwd_bwd_ex(X, W, y, opt, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.FLCE_ERR_LABEL
    got = dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
               dX=tensor_f64(dX), dW=tensor_f64(dW), err=0)
    f = O.forward(wl.x, wl.w, ref_labels, -100, eps)
    b = O.backward(wl.x, wl.w, ref_labels, -100, eps)
    assert got["nv"] == f.n_valid == wl.N - np.count_nonzero(ref_labels == -100)
    assert rel_err(got["loss"], f.loss) <= LOSS_REL
    assert np.max(np.abs(got["lse"] - f.lse)) <= LSE_ABS
    assert rel_fro(got["dX"], b.dX) <= GRAD_REL_FRO
    assert rel_fro(got["dW"], b.dW) <= GRAD_REL_FRO
    assert np.all(got["dX"][bad] == 0.0)


def test_large_logits_max_subtraction():
    """Logits far above 88.7 (where exp overflows fp32) stay finite and exact."""
    wl = I.make_workload(spec(N=256, H=64, V=900, n_ignore=8, w_std=1.0, x_std=4.0), seed=11)
    f = O.forward(wl.x, wl.w, wl.labels)
    assert f.m.max() > 100.0
    check_against_oracle(wl, run_fwd_bwd(wl))


def test_scaled_rows_gemma_like():
    wl = I.make_workload(spec(N=512, H=128, V=4000, labels="zipf", n_ignore=25,
                              n_scaled_w_rows=40, w_row_scale=8.0, w_std=0.1), seed=12)
    check_against_oracle(wl, run_fwd_bwd(wl))


def test_token_shards_compose_on_one_gpu():
    """Data-parallel algebra: shards run with the sum reduction and the global
    1/N_valid as upstream gradient add up to the unsharded result."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=600, H=128, V=2000, n_ignore=60, smoothing=0.1), seed=13)
    X, W, y = to_device(wl)
    full = run_fwd_bwd(wl)
    nv = full["nv"]
    g = torch.tensor([1.0 / nv], device="cuda")
    loss_sum, dW_sum, dX_parts = 0.0, None, []
    for idx in np.array_split(np.arange(wl.N), 3):
        sl = slice(int(idx[0]), int(idx[-1]) + 1)
        loss, lse, c, dX, dW, err = B.flce_fwd_bwd(X[sl].contiguous(), W, y[sl].contiguous(),
                                                   -100, 0.1, "sum", grad_loss=g)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        loss_sum += float(loss.item())
        dW_sum = tensor_f64(dW) if dW_sum is None else dW_sum + tensor_f64(dW)
        dX_parts.append(tensor_f64(dX))
    assert rel_err(loss_sum / nv, full["loss"]) <= 1e-5
    assert rel_fro(np.concatenate(dX_parts), full["dX"]) <= 1e-3
    assert rel_fro(dW_sum, full["dW"]) <= 1e-3


def test_autograd_wrapper():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=160, H=64, V=500, n_ignore=12), seed=14)
    X, W, y = to_device(wl)
    X.requires_grad_(True)
    W.requires_grad_(True)
    loss = B.linear_cross_entropy(X.view(2, 80, 64), W, y.view(2, 80))
    loss.backward()
    torch.cuda.synchronize()
    f = O.forward(wl.x, wl.w, wl.labels)
    b = O.backward(wl.x, wl.w, wl.labels)
    assert rel_err(loss.item(), f.loss) <= LOSS_REL
    assert rel_fro(tensor_f64(X.grad), b.dX) <= GRAD_REL_FRO
    assert rel_fro(tensor_f64(W.grad), b.dW) <= GRAD_REL_FRO


def test_l2_hints_do_not_change_results():
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=640, H=256, V=4000, n_ignore=30, smoothing=0.1), seed=16)
    try:
        B.flce_set_l2_hints(True)
        a = run_fwd_bwd(wl)
        B.flce_set_l2_hints(False)
        b = run_fwd_bwd(wl)
    finally:
        B.flce_set_l2_hints(False)
    assert a["loss"] == b["loss"]
    for k in ("lse", "dX", "dW"):
        assert np.array_equal(a[k], b[k])


@pytest.mark.parametrize("z_loss", [1e-4, 0.05])
def test_z_loss(z_loss):
    """z-loss: each valid token adds alpha * lse^2; the dZ softmax term is
    scaled by 1 + 2 alpha lse."""
    wl = I.make_workload(spec(N=400, H=192, V=2500, n_ignore=25, smoothing=0.1, w_std=0.1),
                         seed=17)
    got = run_fwd_bwd(wl, z_loss=z_loss)
    check_against_oracle(wl, got, z_loss=z_loss)


def test_z_loss_separate_calls_and_sum():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=300, H=128, V=1800, n_ignore=20), seed=18)
    X, W, y = to_device(wl)
    loss, lse, nv, err = B.flce_forward(X, W, y, -100, 0.0, "sum", z_loss=0.01)
    dX, dW, err2 = B.flce_backward(X, W, y, lse, nv, -100, 0.0, "sum", z_loss=0.01)
    torch.cuda.synchronize()
    got = dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
               dX=tensor_f64(dX), dW=tensor_f64(dW), err=int(err.item()) | int(err2.item()))
    check_against_oracle(wl, got, reduction="sum", z_loss=0.01)


def test_per_token_loss():
    """reduction 'none': every token's loss, 0 on ignored rows."""
    wl = I.make_workload(spec(N=333, H=96, V=1200, n_ignore=33, smoothing=0.1), seed=19)
    got = run_fwd_bwd(wl, row_loss=True, z_loss=0.001)
    f = O.forward(wl.x, wl.w, wl.labels, -100, 0.1, z_loss=0.001)
    assert np.max(np.abs(got["row_loss"] - f.row_loss)) <= LSE_ABS
    assert np.all(got["row_loss"][wl.labels == -100] == 0.0)
    assert rel_err(got["row_loss"].sum() / f.n_valid, f.loss) <= LOSS_REL


@pytest.mark.parametrize("pair", [1, 0], ids=["cta_pair", "single_cta"])
def test_skip_ignored_blocks_sft(pair):
    """Whole token blocks whose labels are all ignored are skipped: loss, dX, dW
    as the oracle's; lse equal on kept rows and NaN on skipped ones."""
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_cta_pair(pair)
    wl = I.make_workload(spec(N=2048, H=192, V=3000, labels="sft", seq_len=512,
                              prompt_frac=(0.3, 0.9), smoothing=0.1), seed=20)
    got = run_fwd_bwd(wl, skip=True, z_loss=1e-3, row_loss=True)
    f, _ = check_against_oracle(wl, got, z_loss=1e-3, lse_rows="finite")
    rows = 256 if pair else 128
    blocks = wl.labels.reshape(-1, rows)
    skipped = np.all(blocks == -100, axis=1).repeat(rows)
    assert skipped.any() and not skipped.all()
    assert np.all(np.isnan(got["lse"][skipped])) and np.all(np.isfinite(got["lse"][~skipped]))
    assert np.all(got["row_loss"][skipped] == 0.0)
    full = run_fwd_bwd(wl, z_loss=1e-3)
    assert rel_err(got["loss"], full["loss"]) <= 1e-6
    assert rel_fro(got["dX"], full["dX"]) <= 1e-6 and rel_fro(got["dW"], full["dW"]) <= 1e-6


def test_skip_ignored_blocks_all_ignored():
    wl = I.make_workload(spec(N=600, H=64, V=700, n_ignore=600), seed=21)
    got = run_fwd_bwd(wl, skip=True)
    assert got["err"] == 0 and got["nv"] == 0 and got["loss"] == 0.0
    assert np.all(got["dX"] == 0.0) and np.all(got["dW"] == 0.0)
    assert np.all(np.isnan(got["lse"]))


def test_skip_with_separate_calls_and_chunks():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_vocab_chunk(512)
    wl = I.make_workload(spec(N=1500, H=136, V=2100, labels="sft", seq_len=500), seed=22)
    X, W, y = to_device(wl)
    loss, lse, nv, err = B.flce_forward(X, W, y, skip_ignored_blocks=True)
    dX, dW, err2 = B.flce_backward(X, W, y, lse, nv, skip_ignored_blocks=True)
    torch.cuda.synchronize()
    got = dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
               dX=tensor_f64(dX), dW=tensor_f64(dW), err=int(err.item()) | int(err2.item()))
    check_against_oracle(wl, got, lse_rows="finite")
