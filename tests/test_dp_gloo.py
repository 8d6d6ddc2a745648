"""Token shards and vocabulary shards across two CPU ranks (gloo), no GPU.

Each rank holds half of the tokens.  The exchange a data-parallel trainer
performs around the fused op -- an all-reduce of (sum of losses, N_valid)
before the backward, so every rank scales by the global 1/N_valid, and an
all-reduce of the partial dW afterwards -- must reproduce the unsharded
result.  The per-rank arithmetic is the oracle's (sum reduction with the
global upstream gradient), which the GPU path matches in
test_gpu_parity.test_token_shards_compose_on_one_gpu.
"""
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_q):
    import torch
    import torch.distributed as dist
    from oracle import flce_oracle as O

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(0)
        N, H, V, eps = 40, 6, 23, 0.1
        X = rng.standard_normal((N, H))
        W = rng.standard_normal((V, H)) * 0.5
        y = rng.integers(0, V, N)
        y[rng.permutation(N)[:7]] = -100
        rows = np.array_split(np.arange(N), world)[rank]
        # forward on the shard, then exchange (sum of losses, N_valid)
        f = O.forward(X[rows], W, y[rows], -100, eps, "sum")
        t = torch.tensor([f.loss_sum, float(f.n_valid)], dtype=torch.float64)
        dist.all_reduce(t)
        loss_global = t[0].item() / t[1].item()
        nv_global = int(t[1].item())
        # backward with the global scale, then all-reduce dW
        b = O.backward(X[rows], W, y[rows], -100, eps, "sum", grad_loss=1.0 / nv_global)
        dW = torch.from_numpy(b.dW.copy())
        dist.all_reduce(dW)
        full_f, full_b = O.fwd_bwd(X, W, y, -100, eps, "mean")
        ok = (abs(loss_global - full_f.loss) < 1e-12
              and np.allclose(dW.numpy(), full_b.dW, atol=1e-14)
              and np.allclose(b.dX, full_b.dX[rows], atol=1e-14)
              and nv_global == full_f.n_valid)
        result_q.put((rank, bool(ok)))
    finally:
        dist.destroy_process_group()


def test_two_rank_token_shards_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: True, 1: True}


def _vocab_rank_main(rank, world, port, result_q):
    import torch
    import torch.distributed as dist
    from oracle import flce_oracle as O

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(1)
        N, H, V, eps, a = 30, 5, 37, 0.1, 0.01
        X = rng.standard_normal((N, H))
        W = rng.standard_normal((V, H)) * 0.5
        y = rng.integers(0, V, N)
        y[rng.permutation(N)[:6]] = -100
        bounds = [0, 20, 37]
        v0, v1 = bounds[rank], bounds[rank + 1]
        m, d, zy, zs = O.shard_partials(X, W[v0:v1], y, v0, V)
        mine = torch.from_numpy(np.stack([m, d, zy, zs]))
        gathered = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)  # the exchange of N x 4 statistics
        parts = [tuple(g.numpy()) for g in gathered]
        loss, lse, _, nv = O.combine_partials(parts, y, V, -100, eps, "mean", a)
        dx_p, dw_p = O.shard_backward(X, W[v0:v1], y, v0, V, lse, 1.0 / nv, -100, eps, a)
        dX = torch.from_numpy(dx_p.copy())
        dist.all_reduce(dX)  # partial dX summed over shards
        f, b = O.fwd_bwd(X, W, y, -100, eps, "mean", z_loss=a)
        ok = (abs(loss - f.loss) < 1e-12 and np.allclose(dX.numpy(), b.dX, atol=1e-14)
              and np.allclose(dw_p, b.dW[v0:v1], atol=1e-14))
        result_q.put((rank, bool(ok)))
    finally:
        dist.destroy_process_group()


def test_two_rank_vocab_shards_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_vocab_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: True, 1: True}
