"""Per-call launch settings (flce_options: cta_pair, backward_merge, l2_hints,
vocab_chunk) on the GPU.

Two host threads run fused steps on their own streams with different tile
shapes, backward layouts and chunk widths, each sizing its workspace with
flce_workspace_size_ex from its own options, while a third thread keeps
flipping the process-wide defaults.  No call may fail (a workspace sized
under one setting and used under another would return FLCE_ERR_WORKSPACE),
and each thread's results match the oracle.
"""
import threading

import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from oracle import flce_oracle as O
from tests.gpu_util import GRAD_REL_FRO, LOSS_REL, LSE_ABS, rel_err, rel_fro, tensor_f64, to_device

pytestmark = pytest.mark.gpu


def test_two_threads_with_their_own_settings():
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    spec = I.custom_spec("opts", N=700, H=264, V=3000, dtype="bf16", n_ignore=50, smoothing=0.1)
    wl = I.make_workload(spec, seed=31)
    X, W, y = to_device(wl)
    settings = {
        "pair_merged_512": dict(cta_pair=True, backward_merge=True, vocab_chunk=512),
        "single_cta_1024": dict(cta_pair=False, backward_merge=False, vocab_chunk=1024),
    }
    results, errors = {}, []
    stop = threading.Event()

    def flipper():
        i = 0
        while not stop.is_set():
            B.flce_set_backward_merge(i % 2 == 0)
            B.flce_set_cta_pair(i % 3 != 0)
            B.flce_set_vocab_chunk((i % 4) * 256)
            i += 1

    def worker(name, kw):
        try:
            torch.cuda.set_device(0)
            opt = B.make_options(-100, 0.1, **kw)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                ws = B.workspace(wl.N, wl.H, wl.V, B.FLCE_BF16, B.MODE_FWD_BWD, X.device, opt)
                outs = []
                for _ in range(4):
                    err = torch.zeros(1, dtype=torch.int32, device="cuda")
                    outs.append(B.flce_fwd_bwd_ex(X, W, y, opt, workspace_buf=ws, err_word=err,
                                                  stream=st))
                st.synchronize()
            for o in outs:
                assert int(o[5].item()) == 0
            loss, lse, nv, dX, dW, _ = outs[-1]
            # repeated calls with the same settings are bitwise identical
            for o in outs[:-1]:
                assert torch.equal(o[0], loss) and torch.equal(o[3], dX) and torch.equal(o[4], dW)
            results[name] = dict(loss=float(loss.item()), lse=tensor_f64(lse),
                                 nv=int(nv.item()), dX=tensor_f64(dX), dW=tensor_f64(dW))
        except Exception as e:  # noqa: BLE001 -- reported by the main thread
            errors.append((name, repr(e)))

    t0 = threading.Thread(target=flipper)
    ts = [threading.Thread(target=worker, args=(k, v)) for k, v in settings.items()]
    t0.start()
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    stop.set()
    t0.join()
    B.flce_set_backward_merge(False)
    B.flce_set_cta_pair(True)
    B.flce_set_vocab_chunk(0)
    assert not errors, errors
    f = O.forward(wl.x, wl.w, wl.labels, -100, 0.1)
    b = O.backward(wl.x, wl.w, wl.labels, -100, 0.1)
    for name, got in results.items():
        assert got["nv"] == f.n_valid, name
        assert rel_err(got["loss"], f.loss) <= LOSS_REL, name
        assert np.max(np.abs(got["lse"] - f.lse)) <= LSE_ABS, name
        assert rel_fro(got["dX"], b.dX) <= GRAD_REL_FRO, name
        assert rel_fro(got["dW"], b.dW) <= GRAD_REL_FRO, name


def test_options_override_process_defaults():
    """An explicit per-call setting wins over the process-wide one: the
    merged backward chosen by options gives the same bits as the merged
    backward chosen process-wide, at the same chunk width."""
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    spec = I.custom_spec("opts2", N=600, H=256, V=2500, dtype="bf16", n_ignore=20, smoothing=0.0)
    wl = I.make_workload(spec, seed=32)
    X, W, y = to_device(wl)
    try:
        B.flce_set_backward_merge(False)
        a = B.flce_fwd_bwd_ex(X, W, y, B.make_options(backward_merge=True, vocab_chunk=512))
        B.flce_set_backward_merge(True)
        B.flce_set_vocab_chunk(512)
        b = B.flce_fwd_bwd(X, W, y)
        torch.cuda.synchronize()
    finally:
        B.flce_set_backward_merge(False)
        B.flce_set_vocab_chunk(0)
    assert int(a[5].item()) == 0 and int(b[5].item()) == 0
    for i in (0, 1, 3, 4):
        assert torch.equal(a[i], b[i])
