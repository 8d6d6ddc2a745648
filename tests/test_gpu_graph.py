"""The fused call inside a CUDA graph.

flce_fwd_bwd enqueues its kernels, memsets and nothing else on the caller's
stream: no host synchronisation, no allocation.  So a training loop can capture
it once into a CUDA graph and replay it with new inputs copied into the captured
buffers.  These tests capture the call (after one eager call, which sets the
kernels' attributes), replay it on fresh inputs and require the same bits as
eager calls on those inputs, for the default backward and the merged one.
"""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    from linear_cross_entropy_logit_gb300 import binding as B
    yield
    B.flce_set_backward_merge(0)
    B.flce_set_vocab_chunk(0)


@pytest.mark.parametrize("merge", [0, 1], ids=["three_launches", "merged"])
def test_fused_call_replays_in_a_cuda_graph(merge):
    import torch
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_backward_merge(merge)
    B.flce_set_vocab_chunk(1024)
    N, H, V = 1000, 384, 5000
    specs = [I.custom_spec("graph", N=N, H=H, V=V, dtype="bf16", n_ignore=50, smoothing=0.1)
             for _ in range(3)]
    wls = [I.make_workload(s, seed=50 + i) for i, s in enumerate(specs)]
    dev = torch.device("cuda")
    X, W, y = (t.clone() for t in to_device(wls[0]))
    g_loss = torch.tensor([0.5], dtype=torch.float32, device=dev)
    outs = dict(loss=torch.empty(1, dtype=torch.float32, device=dev),
                lse=torch.empty(N, dtype=torch.float32, device=dev),
                valid_count=torch.empty(1, dtype=torch.int32, device=dev),
                dX=torch.empty_like(X), dW=torch.empty(V, H, dtype=torch.float32, device=dev))
    ws = B.workspace(N, H, V, B.FLCE_BF16, B.MODE_FWD_BWD, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def call(stream=None):
        B.flce_fwd_bwd(X, W, y, -100, 0.1, "mean", grad_loss=g_loss, workspace_buf=ws,
                       err_word=err, stream=stream, **outs)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # eager warm-up: kernel attributes and occupancy are set here
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()

    for wl in wls[1:]:
        Xn, Wn, yn = to_device(wl)
        # replay on new inputs copied into the captured buffers
        X.copy_(Xn)
        W.copy_(Wn)
        y.copy_(yn)
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = {k: v.clone() for k, v in outs.items()}
        # eager on the same inputs
        call()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for k in outs:
            assert torch.equal(got[k], outs[k]), k
        assert np.isfinite(float(got["loss"].item()))
