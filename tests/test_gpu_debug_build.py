"""The FLCE_DEBUG build (libflce_debug.so) on the small ragged and odd-shape
cases.

That build range-checks the device-side index math the release build trusts:
the unit and tile coordinates of the persistent walks (row-block bands,
vocabulary groups, the merged backward's tile list), the token-block skip
lists, the gradient-filter mask reads and stores, and the forward's partial
slots.  An out-of-range index sets FLCE_ERR_BOUNDS in the error word and the
access is skipped; on the host the workspace plan's regions are checked
before anything is launched.  Every case here must leave the error word at 0
and still match the fp64 oracle within the parity tolerances.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, tensor_f64, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def debug_library():
    from linear_cross_entropy_logit_gb300 import binding as B
    from linear_cross_entropy_logit_gb300 import build as libbuild
    libbuild.build()
    prev = B.use_library(B.load(B.DEBUG_LIB_PATH))
    yield
    B.use_library(prev)


def spec(**kw):
    kw.setdefault("dtype", "bf16")
    return I.custom_spec("debug", **kw)


def run(wl, **opt):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    X, W, y = to_device(wl)
    o = B.make_options(wl.spec.ignore_index, wl.spec.smoothing, **opt)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd_ex(X, W, y, o)
    torch.cuda.synchronize()
    return dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
                dX=tensor_f64(dX), dW=tensor_f64(dW), err=int(err.item()))


def check(wl, got, z_loss=0.0, exact_grads=True):
    from linear_cross_entropy_logit_gb300 import binding as B
    assert got["err"] == 0, B.lib().flce_status_string(got["err"]).decode()
    f, b = O.fwd_bwd(wl.x, wl.w, wl.labels, wl.spec.ignore_index, wl.spec.smoothing,
                     z_loss=z_loss)
    assert got["nv"] == f.n_valid
    assert rel_err(got["loss"], f.loss) <= LOSS_REL
    keep = np.isfinite(got["lse"])
    if wl.N:
        assert np.max(np.abs(got["lse"][keep] - f.lse[keep])) <= LSE_ABS
    if exact_grads:
        assert rel_fro(got["dX"], b.dX) <= GRAD_REL_FRO
        assert rel_fro(got["dW"], b.dW) <= GRAD_REL_FRO


def test_debug_library_is_the_one_called():
    from linear_cross_entropy_logit_gb300 import binding as B
    assert B.lib()._name == B.DEBUG_LIB_PATH


@pytest.mark.parametrize("pair", [True, False], ids=["cta_pair", "single_cta"])
@pytest.mark.parametrize("chunk", [0, 256])
def test_ragged_multi_tile(pair, chunk):
    wl = I.make_workload(spec(N=300, H=136, V=1000, n_ignore=30, smoothing=0.1), seed=1)
    check(wl, run(wl, cta_pair=pair, vocab_chunk=chunk))


def test_row_bands_and_vocab_groups():
    """X above 48 MiB (N = 100000, H = 256: 51.2 MB): the forward and dZ
    launches walk two row-block bands; forward partials above 32 MiB (24
    vocabulary tiles x 100096 padded rows): the forward groups two vocabulary
    tiles per unit.  lse of every row, the loss, and dX / dW rows at the band
    and chunk edges against the oracle's row-by-row definitions."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=100000, H=256, V=6000, n_ignore=500), seed=2)
    X, W, y = to_device(wl)
    o = B.make_options(vocab_chunk=1024)
    loss, lse, nv, dX, dW, err = B.flce_fwd_bwd_ex(X, W, y, o)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    f = O.forward(wl.x, wl.w, wl.labels)
    assert int(nv.item()) == f.n_valid
    assert rel_err(float(loss.item()), f.loss) <= LOSS_REL
    assert np.max(np.abs(tensor_f64(lse) - f.lse)) <= LSE_ABS
    band = 196 * 256  # ceil(391 row blocks / 2 bands) blocks of 256 rows
    rows = np.array([0, band - 1, band, wl.N - 1, 12345, 77777])
    vrows = np.array([0, 1023, 1024, 2047, 5119, 5120, 5999])
    c = O.grad_scale(f.n_valid, "mean")
    want_dx = O.dx_rows(wl.x, wl.w, wl.labels, rows, c)
    want_dw = O.dw_rows(wl.x, wl.w, wl.labels, vrows, f.lse, c)
    got_dx = tensor_f64(dX[torch.from_numpy(rows).cuda()])
    got_dw = tensor_f64(dW[torch.from_numpy(vrows).cuda()])
    assert rel_fro(got_dx, want_dx) <= GRAD_REL_FRO
    assert rel_fro(got_dw, want_dw) <= GRAD_REL_FRO


@pytest.mark.parametrize("pair", [True, False], ids=["cta_pair", "single_cta"])
def test_skip_lists(pair):
    wl = I.make_workload(spec(N=2048, H=192, V=3000, labels="sft", seq_len=512,
                              prompt_frac=(0.3, 0.9), smoothing=0.1), seed=3)
    check(wl, run(wl, cta_pair=pair, skip_ignored_blocks=True, z_loss=1e-3), z_loss=1e-3)


@pytest.mark.parametrize("pair", [True, False], ids=["cta_pair", "single_cta"])
def test_filter_masks(pair):
    """Gradient filtering: the keep masks are written by the dZ epilogue and
    read by the filtered dX / dW k-loops (the loss stays exact)."""
    wl = I.make_workload(I.custom_spec("peaked", N=512, H=256, V=8000, dtype="bf16",
                                       n_ignore=25, x_align=3.0), seed=4)
    check(wl, run(wl, cta_pair=pair, grad_filter=2.0 ** -12), exact_grads=False)


def test_filter_with_skip_lists():
    wl = I.make_workload(I.custom_spec("peaked", N=1024, H=128, V=3000, dtype="bf16",
                                       n_ignore=51, x_align=3.0, labels="sft", seq_len=256),
                         seed=5)
    check(wl, run(wl, grad_filter=0.2, skip_ignored_blocks=True), exact_grads=False)


@pytest.mark.parametrize("chunk", [256, 1024])
def test_merged_backward_tile_list(chunk):
    wl = I.make_workload(spec(N=700, H=136, V=5000, n_ignore=40, smoothing=0.1), seed=6)
    check(wl, run(wl, backward_merge=True, vocab_chunk=chunk))


def test_vocab_shards():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    wl = I.make_workload(spec(N=500, H=128, V=2300, n_ignore=20, smoothing=0.1), seed=7)
    X, W, y = to_device(wl)
    opt = B.make_options(-100, 0.1)
    bounds = [0, 768, 1536, 2300]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    parts = torch.empty(3, wl.N, 4, dtype=torch.float32, device="cuda")
    for i, (b0, b1) in enumerate(zip(bounds, bounds[1:])):
        B.flce_forward_vocab_shard(X, W[b0:b1], y, b0, wl.V, opt, partials=parts[i], err_word=err)
    loss, lse, nv, _ = B.flce_combine_vocab_shards(parts, y, wl.V, opt, err_word=err)
    dX = torch.zeros(wl.N, wl.H, dtype=torch.float32, device="cuda")
    dWs = []
    for b0, b1 in zip(bounds, bounds[1:]):
        dxp, dws, _ = B.flce_backward_vocab_shard(X, W[b0:b1], y, b0, wl.V, lse, nv, opt,
                                                  err_word=err)
        dX += dxp
        dWs.append(dws)
    torch.cuda.synchronize()
    got = dict(loss=float(loss.item()), lse=tensor_f64(lse), nv=int(nv.item()),
               dX=tensor_f64(dX), dW=tensor_f64(torch.cat(dWs)), err=int(err.item()))
    check(wl, got)


@pytest.mark.parametrize("case", ["tiny_fp32", "single_token", "vocab_below_tile",
                                  "all_ignored"])
def test_odd_shapes(case):
    if case == "tiny_fp32":
        wl = I.make_workload("tiny", seed=0)
    elif case == "single_token":
        wl = I.make_workload(spec(N=1, H=32, V=700), seed=8)
    elif case == "vocab_below_tile":
        wl = I.make_workload(spec(N=70, H=48, V=5, n_ignore=3, smoothing=0.2, w_std=0.5), seed=9)
    else:
        wl = I.make_workload(spec(N=130, H=64, V=300, n_ignore=130, smoothing=0.1), seed=10)
    got = run(wl)
    if case == "all_ignored":
        assert got["err"] == 0 and got["nv"] == 0 and got["loss"] == 0.0
        assert np.all(got["dX"] == 0.0) and np.all(got["dW"] == 0.0)
    else:
        check(wl, got)
