"""flce_forward_noalloc: the forward for callers that cannot allocate.

Some callers cannot call cudaMalloc or keep a workspace: code inside an
application that owns all device memory through its own fixed pool, code on a
path that must not allocate after start-up, C callers without an allocator.
For them the library offers a forward whose scratch is a fixed device array
inside the library.  These tests call it through the C ABI and check that it
gives what the regular flce_forward gives, within the parity tolerances, on two
calls in a row with different inputs (the shared array keeps the previous
call's contents, which must not leak into the next result).

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from tests.gpu_util import LOSS_REL, LSE_ABS, rel_err, to_device

pytestmark = pytest.mark.gpu


def _noalloc(L, X, W, y, N, H, V, ii, eps, red):
    import torch
    dev = X.device
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    nv = torch.full((1,), -1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = L.flce_forward_noalloc(X.data_ptr(), W.data_ptr(), y.data_ptr(), N, H, V, ii, eps, red,
                                loss.data_ptr(), lse.data_ptr(), nv.data_ptr(), err.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == 0, L.flce_noalloc_last_error().decode()
    return loss, lse, nv, err


CASES = [
    # (N, H, V, n_ignore, smoothing, reduction code, seed): several row blocks,
    # ragged vocabulary and K tails
    (700, 256, 5000, 40, 0.1, 0, 21),
    (300, 136, 3000, 0, 0.0, 1, 22),
    # partials of 501 vocabulary tiles x 4096 rows (32 MiB) do not fit the
    # 16 MiB array one per tile: the call groups two tiles per partial
    (4096, 256, 128256, 200, 0.0, 0, 24),
]


def test_noalloc_matches_forward_two_calls_in_a_row():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    L = B.lib()
    for (N, H, V, n_ign, eps, red, seed) in CASES:
        spec = I.custom_spec("noalloc", N=N, H=H, V=V, dtype="bf16", n_ignore=n_ign,
                             smoothing=eps)
        wl = I.make_workload(spec, seed=seed)
        X, W, y = to_device(wl)
        loss_a, lse_a, nv_a, err_a = _noalloc(L, X, W, y, N, H, V, -100, eps, red)
        loss_b, lse_b, nv_b, err_b = B.flce_forward(X, W, y, -100, eps,
                                                    "sum" if red else "mean")
        torch.cuda.synchronize()
        assert int(err_a.item()) == 0 and int(err_b.item()) == 0
        assert int(nv_a.item()) == int(nv_b.item()) == N - n_ign
        assert rel_err(loss_a.item(), loss_b.item()) <= LOSS_REL
        assert float((lse_a - lse_b).abs().max().item()) <= LSE_ABS


def test_noalloc_rejects_too_many_tokens():
    """Forward partials of ~1.1M tokens do not fit the fixed scratch: the call
    is refused on the host before anything is launched."""
    from linear_cross_entropy_logit_gb300 import binding as B
    L = B.lib()
    fake = 1 << 20  # aligned stand-in addresses; the call returns before using them
    P = ctypes.c_void_p
    st = L.flce_forward_noalloc(P(fake), P(fake), P(fake), 1_100_000, 64, 1000, -100, 0.0, 0,
                                P(fake), P(fake), P(fake), P(fake), None)
    assert st == B.FLCE_ERR_WORKSPACE
    assert "scratch" in L.flce_noalloc_last_error().decode()
