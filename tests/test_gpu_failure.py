"""Failure detection on the GPU without a fault.

Every wait in the library's kernels is bounded.  Here the bounded wait runs on
an mbarrier that nothing ever arrives on (a flag nothing sets): it has to give
up after its short limit, report FLCE_ERR_TIMEOUT through the error word, and
leave the context usable -- the fused forward+backward still runs and matches
the oracle afterwards.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, rel_err, rel_fro, tensor_f64, to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_context_survives():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    L = B.lib()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = L.flce_debug_wait_timeout(err.data_ptr(), 50_000_000, waited.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == B.FLCE_OK
    torch.cuda.synchronize()
    assert int(err.item()) == B.FLCE_ERR_TIMEOUT
    assert 50_000 <= int(waited.item()) < 2_000_000  # gave up after ~50 ms, not never
    # the context is intact: a full fused step still matches the oracle
    wl = I.make_workload(I.custom_spec("after", N=256, H=128, V=1000, dtype="bf16",
                                       n_ignore=10), seed=50)
    X, W, y = to_device(wl)
    loss, lse, nv, dX, dW, err2 = B.flce_fwd_bwd(X, W, y)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    f, b = O.fwd_bwd(wl.x, wl.w, wl.labels)
    assert rel_err(loss.item(), f.loss) <= LOSS_REL
    assert rel_fro(tensor_f64(dX), b.dX) <= GRAD_REL_FRO
    assert rel_fro(tensor_f64(dW), b.dW) <= GRAD_REL_FRO


def test_error_word_is_sticky_first_error_wins():
    """A later label error does not overwrite an earlier timeout."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    L = B.lib()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.flce_debug_wait_timeout(err.data_ptr(), 1_000_000, waited.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    wl = I.make_workload(I.custom_spec("bad", N=64, H=32, V=50, dtype="bf16"), seed=51)
    wl.labels[3] = 50
    X, W, y = to_device(wl)
    B.flce_fwd_bwd(X, W, y, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.FLCE_ERR_TIMEOUT
