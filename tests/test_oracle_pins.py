"""Pins for the fp64 oracle: checks against facts other than the oracle itself.

Each test targets a mistake that could plausibly hide in the oracle (a dropped
smoothing term, a wrong sign, the wrong normaliser, a transposed operand, a
missing max-subtraction) and checks a value fixed by the pages' equations or
by mathematics: closed forms, brute-force softmax written with scalar loops,
central finite differences, and PyTorch's own float64 cross_entropy (the call
the pages' chunked reference makes, "Cut Cross-Entropy: Memory-Efficient
Large-Vocab LLM Guide", "Pure PyTorch Chunked Cross-Entropy Implementation").
"""
import math

import numpy as np
import pytest

from oracle import flce_oracle as O

IGN = -100


def rand_case(N, H, V, seed, n_ignore=0, x_scale=1.0, w_scale=0.3):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, H)) * x_scale
    W = rng.standard_normal((V, H)) * w_scale
    y = rng.integers(0, V, size=N)
    if n_ignore:
        y[rng.permutation(N)[:n_ignore]] = IGN
    return X, W, y


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("eps", [0.0, 0.1, 0.5])
def test_zero_weight_closed_form(eps):
    """W = 0: every logit is 0, so lse = log V, loss = log V for any eps, dX = 0,
    dZ_ij = c (1/V - (1-eps) 1[j=y] - eps/V) and dW_j = sum_i dZ_ij x_i."""
    N, H, V = 9, 5, 13
    X, _, y = rand_case(N, H, V, 1, n_ignore=2)
    W = np.zeros((V, H))
    f = O.forward(X, W, y, IGN, eps)
    assert np.allclose(f.lse, math.log(V), atol=1e-14, rtol=0)
    assert f.loss == pytest.approx(math.log(V), abs=1e-13)
    b = O.backward(X, W, y, IGN, eps)
    assert np.all(b.dX == 0.0)
    nv = int((y != IGN).sum())
    c = 1.0 / nv
    dW = np.zeros((V, H))
    for i in range(N):
        if y[i] == IGN:
            continue
        for j in range(V):
            g = 1.0 / V - eps / V - ((1.0 - eps) if j == y[i] else 0.0)
            for k in range(H):
                dW[j, k] += c * g * X[i, k]
    assert np.allclose(b.dW, dW, atol=1e-14, rtol=0)


def test_uniform_logits_give_log_v():
    """Identical W rows make each row's logits equal: loss = log V, p = 1/V."""
    N, H, V = 7, 4, 10
    X, _, y = rand_case(N, H, V, 2)
    u = np.random.default_rng(3).standard_normal(H)
    W = np.tile(u, (V, 1))
    f = O.forward(X, W, y, IGN, 0.0)
    assert f.loss == pytest.approx(math.log(V), abs=1e-12)
    assert np.allclose(f.lse, X @ u + math.log(V), atol=1e-12)


def test_x_zero_closed_form():
    """X = 0: dW = 0 and dX_i = c (1-eps) (mean_j W_j - W_{y_i})."""
    N, H, V, eps = 6, 5, 9, 0.2
    _, W, y = rand_case(N, H, V, 4, n_ignore=1)
    X = np.zeros((N, H))
    b = O.backward(X, W, y, IGN, eps)
    assert np.all(b.dW == 0.0)
    nv = int((y != IGN).sum())
    wbar = W.mean(axis=0)
    for i in range(N):
        want = np.zeros(H) if y[i] == IGN else (1 - eps) / nv * (wbar - W[y[i]])
        assert np.allclose(b.dX[i], want, atol=1e-14)


def test_two_classes_softplus():
    """V = 2, eps = 0: l_i = softplus(z_other - z_y)."""
    N, H, V = 8, 6, 2
    X, W, y = rand_case(N, H, V, 5)
    f = O.forward(X, W, y, IGN, 0.0)
    for i in range(N):
        z = [sum(X[i, k] * W[j, k] for k in range(H)) for j in range(V)]
        d = z[1 - y[i]] - z[y[i]]
        sp = d + math.log1p(math.exp(-d)) if d > 0 else math.log1p(math.exp(d))
        assert f.row_loss[i] == pytest.approx(sp, abs=1e-13)


# --------------------------------------------------------------------------
# Brute force with scalar loops, no max-subtraction (|z| < 20 keeps exp finite)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("eps", [0.0, 0.15])
def test_bruteforce_softmax(eps):
    N, H, V = 6, 5, 7
    X, W, y = rand_case(N, H, V, 6, n_ignore=1)
    nv = sum(1 for t in y if t != IGN)
    c = 1.0 / nv
    lse = [0.0] * N
    total = 0.0
    dX = [[0.0] * H for _ in range(N)]
    dW = [[0.0] * H for _ in range(V)]
    for i in range(N):
        z = [sum(X[i, k] * W[j, k] for k in range(H)) for j in range(V)]
        assert max(abs(t) for t in z) < 20
        e = [math.exp(t) for t in z]
        s = sum(e)
        lse[i] = math.log(s)
        if y[i] == IGN:
            continue
        # cross-entropy against the smoothed target distribution q
        q = [eps / V + ((1.0 - eps) if j == y[i] else 0.0) for j in range(V)]
        total += -sum(q[j] * math.log(e[j] / s) for j in range(V))
        for j in range(V):
            g = c * (e[j] / s - q[j])
            for k in range(H):
                dX[i][k] += g * W[j, k]
                dW[j][k] += g * X[i, k]
    f = O.forward(X, W, y, IGN, eps)
    b = O.backward(X, W, y, IGN, eps)
    assert np.allclose(f.lse, lse, atol=1e-13, rtol=0)
    assert f.loss == pytest.approx(total / nv, abs=1e-13)
    assert np.allclose(b.dX, dX, atol=1e-14)
    assert np.allclose(b.dW, dW, atol=1e-14)


# --------------------------------------------------------------------------
# Finite differences (dX, dW) with an ignored row and smoothing
# --------------------------------------------------------------------------
def test_finite_differences():
    N, H, V, eps = 5, 7, 11, 0.1
    X, W, y = rand_case(N, H, V, 7, w_scale=0.5)
    y[3] = IGN
    h = 1e-6

    def L(Xa, Wa):
        return O.forward(Xa, Wa, y, IGN, eps).loss

    b = O.backward(X, W, y, IGN, eps)
    for i in range(N):
        for k in range(H):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, k] += h
            Xm[i, k] -= h
            fd = (L(Xp, W) - L(Xm, W)) / (2 * h)
            assert abs(fd - b.dX[i, k]) <= 1e-7, (i, k)
    for j in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, k] += h
            Wm[j, k] -= h
            fd = (L(X, Wp) - L(X, Wm)) / (2 * h)
            assert abs(fd - b.dW[j, k]) <= 1e-7, (j, k)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------
def test_shift_invariance():
    """W_j <- W_j + u for all j shifts lse_i by x_i.u and leaves the loss unchanged
    (also with smoothing: lse, z_y and mean_j z all shift by the same amount)."""
    N, H, V, eps = 10, 6, 17, 0.1
    X, W, y = rand_case(N, H, V, 8, n_ignore=2)
    u = np.random.default_rng(9).standard_normal(H)
    f0 = O.forward(X, W, y, IGN, eps)
    f1 = O.forward(X, W + u, y, IGN, eps)
    assert np.allclose(f1.lse, f0.lse + X @ u, atol=1e-12)
    assert f1.loss == pytest.approx(f0.loss, abs=1e-12)


def test_lse_bounds_and_row_sums():
    N, H, V, eps = 12, 8, 33, 0.3
    X, W, y = rand_case(N, H, V, 10, n_ignore=3)
    f = O.forward(X, W, y, IGN, eps)
    assert np.all(f.m <= f.lse + 1e-15)
    assert np.all(f.lse <= f.m + math.log(V) + 1e-12)
    Z = O.logits(X, W)
    valid = O.valid_mask(y, V, IGN)
    dZ = O.dlogits(Z, f.lse, y, valid, 1.0 / valid.sum(), eps)
    assert np.allclose(dZ.sum(axis=1), 0.0, atol=1e-15)
    b = O.backward(X, W, y, IGN, eps)
    # sum_j dW_j = sum_i (sum_j dZ_ij) x_i = 0
    assert np.allclose(b.dW.sum(axis=0), 0.0, atol=1e-14)


def test_vocab_permutation_equivariance():
    N, H, V, eps = 9, 6, 14, 0.05
    X, W, y = rand_case(N, H, V, 11, n_ignore=2)
    perm = np.random.default_rng(12).permutation(V)  # new class j is old class perm[j]
    inv = np.argsort(perm)
    y2 = np.where(y == IGN, IGN, inv[np.where(y == IGN, 0, y)])
    f0, b0 = O.fwd_bwd(X, W, y, IGN, eps)
    f1, b1 = O.fwd_bwd(X, W[perm], y2, IGN, eps)
    assert np.allclose(f0.lse, f1.lse, atol=1e-13)
    assert f0.loss == pytest.approx(f1.loss, abs=1e-13)
    assert np.allclose(b0.dX, b1.dX, atol=1e-14)
    assert np.allclose(b0.dW[perm], b1.dW, atol=1e-14)


def test_large_logits_no_overflow():
    """Max-subtraction ("Numerical traps": exp without max-subtraction overflows
    above ~88.7 in fp32): logits near 1000 give the shifted lse exactly."""
    N, H, V = 4, 3, 6
    X, W, y = rand_case(N, H, V, 13)
    f0 = O.forward(X, W, y, IGN)
    # add a constant 1000 to every logit through an extra hidden unit
    X2 = np.concatenate([X, np.full((N, 1), 1000.0)], axis=1)
    W2 = np.concatenate([W, np.ones((V, 1))], axis=1)
    f1 = O.forward(X2, W2, y, IGN)
    assert np.all(np.isfinite(f1.lse))
    assert np.allclose(f1.lse, f0.lse + 1000.0, atol=1e-10)
    assert f1.loss == pytest.approx(f0.loss, abs=1e-10)


# --------------------------------------------------------------------------
# Masking, normaliser, reductions, errors
# --------------------------------------------------------------------------
def test_masking():
    N, H, V, eps = 8, 5, 9, 0.1
    X, W, y = rand_case(N, H, V, 14)
    y[[1, 5]] = IGN
    f, b = O.fwd_bwd(X, W, y, IGN, eps)
    assert f.row_loss[1] == 0.0 and f.row_loss[5] == 0.0
    assert np.all(b.dX[1] == 0.0) and np.all(b.dX[5] == 0.0)
    assert f.n_valid == 6
    assert f.loss == pytest.approx(f.row_loss.sum() / 6, abs=1e-15)
    X2 = X.copy()
    X2[5] += 3.0
    f2, b2 = O.fwd_bwd(X2, W, y, IGN, eps)
    assert f2.loss == pytest.approx(f.loss, abs=1e-15)
    assert np.allclose(b2.dW, b.dW, atol=1e-15)
    # lse of an ignored row is still defined (R4)
    assert np.isfinite(f.lse[5])


def test_all_ignored():
    N, H, V = 4, 3, 5
    X, W, _ = rand_case(N, H, V, 15)
    y = np.full(N, IGN)
    f, b = O.fwd_bwd(X, W, y, IGN, 0.1)
    assert f.loss == 0.0 and f.n_valid == 0
    assert np.all(b.dX == 0.0) and np.all(b.dW == 0.0)
    acc = np.random.default_rng(16).standard_normal((V, H))
    b2 = O.backward(X, W, y, IGN, 0.1, dW_in=acc)
    assert np.array_equal(b2.dW, acc)


def test_sum_reduction_and_grad_scale():
    N, H, V, eps = 7, 4, 8, 0.2
    X, W, y = rand_case(N, H, V, 17, n_ignore=2)
    fm, bm = O.fwd_bwd(X, W, y, IGN, eps, "mean")
    fs, bs = O.fwd_bwd(X, W, y, IGN, eps, "sum", grad_loss=0.5)
    assert fs.loss == pytest.approx(fm.loss * 5, abs=1e-12)
    assert np.allclose(bs.dX, 0.5 * 5 * bm.dX, atol=1e-14)
    assert np.allclose(bs.dW, 0.5 * 5 * bm.dW, atol=1e-14)


def test_accumulate_dw():
    N, H, V = 5, 4, 6
    X, W, y = rand_case(N, H, V, 18)
    acc = np.random.default_rng(19).standard_normal((V, H))
    b0 = O.backward(X, W, y, IGN)
    b1 = O.backward(X, W, y, IGN, dW_in=acc)
    assert np.allclose(b1.dW, b0.dW + acc, atol=1e-15)


def test_bad_label_is_error():
    X, W, y = rand_case(3, 2, 4, 20)
    y[1] = 4
    with pytest.raises(ValueError):
        O.forward(X, W, y, IGN)
    y[1] = -1
    with pytest.raises(ValueError):
        O.forward(X, W, y, IGN)
    # a non-negative ignore_index masks that class as a label
    y[1] = 2
    f = O.forward(X, W, y, ignore_index=2)
    assert f.row_loss[1] == 0.0


def test_bf16_upcast_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F], dtype=np.uint16)
    want = [1.0, -1.0, 3.140625, 2.0 ** -133, 3.3895313892515355e38]
    assert list(O.upcast(bits)) == want


# --------------------------------------------------------------------------
# Sampled-output helpers agree with the full definition
# --------------------------------------------------------------------------
def test_sampled_helpers_match_full():
    N, H, V, eps = 20, 6, 31, 0.1
    X, W, y = rand_case(N, H, V, 21, n_ignore=4)
    f, b = O.fwd_bwd(X, W, y, IGN, eps)
    rows = [0, 3, 7, 19]
    lse, rl, _ = O.forward_rows(X, W, y, rows, IGN, eps)
    assert np.allclose(lse, f.lse[rows], atol=1e-14)
    assert np.allclose(rl, f.row_loss[rows], atol=1e-14)
    c = 1.0 / f.n_valid
    assert np.allclose(O.dx_rows(X, W, y, rows, c, IGN, eps), b.dX[rows], atol=1e-14)
    vr = [0, 5, 30]
    assert np.allclose(O.dw_rows(X, W, y, vr, f.lse, c, IGN, eps), b.dW[vr], atol=1e-14)


# --------------------------------------------------------------------------
# Library cross-check: PyTorch float64 cross_entropy + autograd on CPU
# --------------------------------------------------------------------------
@pytest.mark.parametrize("eps,reduction", [(0.0, "mean"), (0.1, "mean"), (0.1, "sum")])
def test_against_torch_cross_entropy(eps, reduction):
    torch = pytest.importorskip("torch")
    N, H, V = 37, 19, 53
    X, W, y = rand_case(N, H, V, 22, n_ignore=6)
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    yt = torch.tensor(y)
    loss = torch.nn.functional.cross_entropy(Xt @ Wt.T, yt, ignore_index=IGN,
                                             label_smoothing=eps, reduction=reduction)
    loss.backward()
    f, b = O.fwd_bwd(X, W, y, IGN, eps, reduction)
    lse_t = torch.logsumexp((Xt @ Wt.T).detach(), dim=1).numpy()
    assert f.loss == pytest.approx(loss.item(), abs=1e-12)
    assert np.allclose(f.lse, lse_t, atol=1e-12)
    assert np.allclose(b.dX, Xt.grad.numpy(), atol=1e-13)
    assert np.allclose(b.dW, Wt.grad.numpy(), atol=1e-13)


# --------------------------------------------------------------------------
# Data-parallel algebra: shards with the global valid count sum to the whole
# --------------------------------------------------------------------------
def test_token_shards_compose():
    N, H, V, eps = 24, 5, 12, 0.1
    X, W, y = rand_case(N, H, V, 23, n_ignore=5)
    f, b = O.fwd_bwd(X, W, y, IGN, eps, "mean")
    nv = f.n_valid
    parts = np.array_split(np.arange(N), 3)
    loss_sum, dW = 0.0, np.zeros((V, H))
    for p in parts:
        fs = O.forward(X[p], W, y[p], IGN, eps, "sum")
        bs = O.backward(X[p], W, y[p], IGN, eps, "sum", grad_loss=1.0 / nv)
        loss_sum += fs.loss
        dW += bs.dW
        assert np.allclose(bs.dX, b.dX[p], atol=1e-14)
    assert loss_sum / nv == pytest.approx(f.loss, abs=1e-13)
    assert np.allclose(dW, b.dW, atol=1e-14)


# --------------------------------------------------------------------------
# z-loss (R19): alpha * lse_i^2 per valid token
# --------------------------------------------------------------------------
@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_z_loss_zero_weight_closed_form(eps):
    """W = 0: lse = log V for every row, so loss = log V + alpha log^2 V and
    dZ_ij = c ((1 + 2 alpha log V)/V - (1-eps) 1[j=y] - eps/V)."""
    N, H, V, a = 7, 4, 9, 0.03
    X, _, y = rand_case(N, H, V, 30, n_ignore=2)
    W = np.zeros((V, H))
    f = O.forward(X, W, y, IGN, eps, z_loss=a)
    L = math.log(V)
    assert f.loss == pytest.approx(L + a * L * L, abs=1e-13)
    Z = O.logits(X, W)
    valid = O.valid_mask(y, V, IGN)
    c = 1.0 / valid.sum()
    dZ = O.dlogits(Z, f.lse, y, valid, c, eps, a)
    for i in range(N):
        for j in range(V):
            want = 0.0 if y[i] == IGN else c * ((1 + 2 * a * L) / V - eps / V
                                                - ((1 - eps) if j == y[i] else 0.0))
            assert dZ[i, j] == pytest.approx(want, abs=1e-15)


def test_z_loss_finite_differences():
    N, H, V, eps, a = 5, 6, 9, 0.1, 0.05
    X, W, y = rand_case(N, H, V, 31, w_scale=0.5)
    y[2] = IGN
    h = 1e-6

    def L(Xa, Wa):
        return O.forward(Xa, Wa, y, IGN, eps, z_loss=a).loss

    b = O.backward(X, W, y, IGN, eps, z_loss=a)
    for i in range(N):
        for k in range(H):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, k] += h
            Xm[i, k] -= h
            assert abs((L(Xp, W) - L(Xm, W)) / (2 * h) - b.dX[i, k]) <= 1e-7
    for j in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, k] += h
            Wm[j, k] -= h
            assert abs((L(X, Wp) - L(X, Wm)) / (2 * h) - b.dW[j, k]) <= 1e-7


def test_z_loss_against_torch():
    torch = pytest.importorskip("torch")
    N, H, V, eps, a = 29, 11, 41, 0.1, 0.02
    X, W, y = rand_case(N, H, V, 32, n_ignore=5)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    yt = torch.tensor(y)
    Z = Xt @ Wt.T
    valid = yt != IGN
    ce = torch.nn.functional.cross_entropy(Z, yt, ignore_index=IGN, label_smoothing=eps,
                                           reduction="sum")
    zl = (torch.logsumexp(Z, dim=1) ** 2)[valid].sum()
    loss = (ce + a * zl) / valid.sum()
    loss.backward()
    f, b = O.fwd_bwd(X, W, y, IGN, eps, "mean", z_loss=a)
    assert f.loss == pytest.approx(loss.item(), abs=1e-12)
    assert np.allclose(b.dX, Xt.grad.numpy(), atol=1e-13)
    assert np.allclose(b.dW, Wt.grad.numpy(), atol=1e-13)
    rows = [0, 4, 10]
    _, rl, _ = O.forward_rows(X, W, y, rows, IGN, eps, z_loss=a)
    assert np.allclose(rl, f.row_loss[rows], atol=1e-14)
    c = 1.0 / f.n_valid
    assert np.allclose(O.dx_rows(X, W, y, rows, c, IGN, eps, a), b.dX[rows], atol=1e-14)
    assert np.allclose(O.dw_rows(X, W, y, [1, 7], f.lse, c, IGN, eps, a), b.dW[[1, 7]],
                       atol=1e-14)


# --------------------------------------------------------------------------
# Vocabulary shards compose to the unsharded definition
# --------------------------------------------------------------------------
@pytest.mark.parametrize("bounds", [[0, 7, 19, 31], [0, 1, 30, 31]])
def test_vocab_shards_compose(bounds):
    N, H, V, eps, a = 11, 6, 31, 0.1, 0.01
    X, W, y = rand_case(N, H, V, 33, n_ignore=3)
    f, b = O.fwd_bwd(X, W, y, IGN, eps, "mean", z_loss=a)
    parts = [O.shard_partials(X, W[v0:v1], y, v0, V, IGN) for v0, v1 in zip(bounds, bounds[1:])]
    loss, lse, row, nv = O.combine_partials(parts, y, V, IGN, eps, "mean", a)
    assert loss == pytest.approx(f.loss, abs=1e-13)
    assert np.allclose(lse, f.lse, atol=1e-13) and np.allclose(row, f.row_loss, atol=1e-13)
    assert nv == f.n_valid
    c = 1.0 / nv
    dX = np.zeros_like(b.dX)
    dW = []
    for v0, v1 in zip(bounds, bounds[1:]):
        dx_p, dw_p = O.shard_backward(X, W[v0:v1], y, v0, V, lse, c, IGN, eps, a)
        dX += dx_p
        dW.append(dw_p)
    assert np.allclose(dX, b.dX, atol=1e-14)
    assert np.allclose(np.concatenate(dW), b.dW, atol=1e-14)


def test_shard_partial_closed_form():
    """A shard with W = 0 has m = 0, d = V_p, z_y = 0 and sum_z = 0."""
    X, _, y = rand_case(4, 3, 10, 34)
    m, d, zy, zs = O.shard_partials(X, np.zeros((4, 3)), y, 6, 10)
    assert np.all(m == 0) and np.all(d == 4) and np.all(zs == 0)
    assert np.all(zy == 0)
