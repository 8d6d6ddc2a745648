"""fp64 CPU oracle for the fused linear cross-entropy path.

TEST INFRASTRUCTURE.  This module is the plain definition the CUDA path is
checked against.  Only the tests, the smoke check and the benchmark's CPU
baseline / reference arm may import or call it; the library itself never
does, and this module imports nothing from the library.

Sources (page title, then section / equation):
  [CFCE] "Chunked and Fused Cross-Entropy: How Online Logit Tiling Slashes
         Large-Vocabulary VRAM Bottlenecks in LLM Training"
         - "The Vocabulary Memory Wall in Modern LLMs": the projection
           Z = X W^T and the loss equation l_i = -z_{i,y_i} + log sum_j exp(z_ij).
         - "Mathematical Mechanics of Chunked Online Cross-Entropy", steps 2
           (stable log-sum-exp m_i, d_i, LSE), 3 (gradient
           (exp(z-m)/d - 1[j=y]) / N) and 4 (dX = dZ W, dW += dZ^T X).
         - "Numerical Considerations ...", items 2 (label -100 masking) and 3
           (label smoothing folded into the same pass).
  [CCE]  "Cut Cross-Entropy: Memory-Efficient Large-Vocab LLM Guide"
         - "Online Log-Sum-Exp Accumulation in High-Speed SRAM" (LSE = m +
           log sum exp(z - m); l = LSE - z_y).
         - "Numerical Stability and Maximum Subtraction on Chip".
         - "Pure PyTorch Chunked Cross-Entropy Implementation": ignore_index
           rows are skipped, the sum of per-token losses is divided by
           max(valid_token_count, 1).
  [FCE]  "Fused cross-entropy -- the memory kernel"
         - "The gradient that makes fusion trivial": dlogits = (p - y) / N.
         - "Numerical traps" table: max-subtraction, fp32 accumulation,
           smoothing and ignore_index folded into the pass.

Readings where the pages are silent or garbled (R-numbers match the design
notes):
  R1 label smoothing eps: uniform eps/V mass over all V classes, target
     weight 1-eps+eps/V (the semantics of the F.cross_entropy call the pages'
     own code makes):  l_i = lse_i - (1-eps) z_{i,y_i} - (eps/V) sum_j z_ij.
  R2 the mean divides by the number of non-ignored tokens N_v.
  R3 N_v = 0 gives loss 0 and zero gradients (max(valid, 1)).
  R4 lse is defined and returned for every row, ignored rows included.
  R5 a label outside [0, V) that is not ignore_index is an error.
  R7 labels are 0-based.
  R8 dW is overwritten unless an accumulator is passed (then +=).
  R11 dlogits = c * (softmax - onehot), c = grad_loss / N_v (mean) or
      grad_loss (sum).
  R19 z-loss ([CFCE] "Numerical Considerations ...", item 3, gives
      L_z = alpha * log^2 sum_j exp(z_ij) per token without saying how it is
      averaged): each valid token adds alpha * lse_i^2 to its loss, averaged
      with the same normaliser as the cross-entropy; its gradient adds
      c * 2 alpha lse_i * softmax_ij to dZ_ij.

Rows are independent in every formula below.  ``forward`` therefore walks
the rows in groups only to bound memory; no value is computed differently
from the per-row definition.  The matrix product is numpy's float64 matmul,
used as a library primitive for the sums over H (forward) and over V or N
(backward).

Parity pins: tests/test_oracle_pins.py checks every function here against
closed forms, brute-force softmax, finite differences and PyTorch's own
cross_entropy on small cases.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

IGNORE_INDEX = -100


# ----------------------------------------------------------------------------
# Step 0: exact widening of the given bits to float64.
# ----------------------------------------------------------------------------
def upcast(a: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) or float32/float64 values -> float64, exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if a.dtype in (np.float32, np.float64):
        return a.astype(np.float64)
    raise TypeError(f"unsupported input dtype {a.dtype}")


# ----------------------------------------------------------------------------
# [CFCE] "The Vocabulary Memory Wall": Z = X W^T.
# ----------------------------------------------------------------------------
def logits(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z_ij = sum_k X_ik W_jk, float64."""
    return upcast(X) @ upcast(W).T


# ----------------------------------------------------------------------------
# [CFCE] step 2 / [CCE] "Online Log-Sum-Exp": m_i, d_i, LSE_i.
# ----------------------------------------------------------------------------
def row_logsumexp(Z: np.ndarray):
    """Return (m, d, lse): m_i = max_j z_ij, d_i = sum_j exp(z_ij - m_i),
    lse_i = m_i + log d_i."""
    m = Z.max(axis=1)
    d = np.exp(Z - m[:, None]).sum(axis=1)
    return m, d, m + np.log(d)


def valid_mask(labels: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    """R5/R7: labels are 0-based; ignore_index rows are masked; any other label
    outside [0, V) is an error."""
    labels = np.asarray(labels, dtype=np.int64)
    valid = labels != ignore_index
    bad = valid & ((labels < 0) | (labels >= V))
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise ValueError(f"label {int(labels[i])} at row {i} is outside [0, {V})")
    return valid


def grad_scale(n_valid: int, reduction: str, grad_loss: float = 1.0) -> float:
    """c = grad_loss / N_v for the mean (0 when N_v = 0, R3); grad_loss for sum."""
    if reduction == "mean":
        return 0.0 if n_valid == 0 else float(grad_loss) / float(n_valid)
    if reduction == "sum":
        return float(grad_loss)
    raise ValueError(f"unknown reduction {reduction!r}")


def row_losses(Z: np.ndarray, lse: np.ndarray, labels: np.ndarray,
               valid: np.ndarray, smoothing: float, z_loss: float = 0.0) -> np.ndarray:
    """l_i = valid_i * (lse_i - (1-eps) z_{i,y_i} - (eps/V) sum_j z_ij + alpha lse_i^2)
    (R1, R19).  With eps = alpha = 0 this is [CFCE] step 2's
    l_i = -z_{i,y_i} + m_i + log d_i."""
    V = Z.shape[1]
    y = np.where(valid, labels, 0)
    z_y = Z[np.arange(Z.shape[0]), y]
    loss = lse - (1.0 - smoothing) * z_y
    if smoothing != 0.0:
        loss = loss - (smoothing / V) * Z.sum(axis=1)
    if z_loss != 0.0:
        loss = loss + z_loss * lse * lse
    return np.where(valid, loss, 0.0)


@dataclasses.dataclass
class ForwardResult:
    loss: float            # mean over valid rows (or sum), R2/R3
    lse: np.ndarray        # N, every row (R4)
    row_loss: np.ndarray   # N, 0 on ignored rows
    n_valid: int
    m: np.ndarray          # N row maxima
    loss_sum: float


def forward(X, W, labels, ignore_index: int = IGNORE_INDEX,
            smoothing: float = 0.0, reduction: str = "mean",
            row_group: int = 512, z_loss: float = 0.0) -> ForwardResult:
    """Loss, per-row lse and per-row loss ([CFCE] steps 1-2, [CCE] loss)."""
    Xd, Wd = upcast(X), upcast(W)
    N, V = Xd.shape[0], Wd.shape[0]
    labels = np.asarray(labels, dtype=np.int64)
    valid = valid_mask(labels, V, ignore_index)
    lse = np.empty(N)
    m = np.empty(N)
    row_loss = np.empty(N)
    for r0 in range(0, N, row_group):
        r1 = min(N, r0 + row_group)
        Z = Xd[r0:r1] @ Wd.T
        m[r0:r1], _, lse[r0:r1] = row_logsumexp(Z)
        row_loss[r0:r1] = row_losses(Z, lse[r0:r1], labels[r0:r1], valid[r0:r1], smoothing,
                                     z_loss)
    n_valid = int(valid.sum())
    loss_sum = float(row_loss.sum())
    if reduction == "mean":
        loss = loss_sum / n_valid if n_valid else 0.0
    elif reduction == "sum":
        loss = loss_sum
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    return ForwardResult(loss, lse, row_loss, n_valid, m, loss_sum)


# ----------------------------------------------------------------------------
# [CFCE] step 3, [FCE] "The gradient that makes fusion trivial":
#   dZ_ij = c * valid_i * (exp(z_ij - lse_i) - (1-eps) 1[j=y_i] - eps/V)
# ----------------------------------------------------------------------------
def dlogits(Z: np.ndarray, lse: np.ndarray, labels: np.ndarray,
            valid: np.ndarray, c: float, smoothing: float,
            z_loss: float = 0.0) -> np.ndarray:
    """... + c * valid_i * 2 alpha lse_i * softmax_ij with z-loss (R19)."""
    V = Z.shape[1]
    P = np.exp(Z - lse[:, None])
    if z_loss != 0.0:
        P = P * (1.0 + 2.0 * z_loss * lse)[:, None]
    dZ = P - smoothing / V
    rows = np.flatnonzero(valid)
    dZ[rows, labels[rows]] -= (1.0 - smoothing)
    dZ[~valid] = 0.0
    return c * dZ


@dataclasses.dataclass
class BackwardResult:
    dX: np.ndarray  # N x H float64
    dW: np.ndarray  # V x H float64


def backward(X, W, labels, ignore_index: int = IGNORE_INDEX,
             smoothing: float = 0.0, reduction: str = "mean",
             grad_loss: float = 1.0, dW_in: Optional[np.ndarray] = None,
             n_valid: Optional[int] = None, z_loss: float = 0.0) -> BackwardResult:
    """[CFCE] step 4: dX = dZ W and dW = dZ^T X (+ dW_in when accumulating).

    ``n_valid`` overrides the local count of valid rows (a data-parallel shard
    scales by the global count)."""
    Xd, Wd = upcast(X), upcast(W)
    V = Wd.shape[0]
    labels = np.asarray(labels, dtype=np.int64)
    valid = valid_mask(labels, V, ignore_index)
    nv = int(valid.sum()) if n_valid is None else int(n_valid)
    c = grad_scale(nv, reduction, grad_loss)
    Z = Xd @ Wd.T
    _, _, lse = row_logsumexp(Z)
    dZ = dlogits(Z, lse, labels, valid, c, smoothing, z_loss)
    dX = dZ @ Wd
    dW = dZ.T @ Xd
    if dW_in is not None:
        dW = dW + upcast(dW_in)
    return BackwardResult(dX, dW)


# ----------------------------------------------------------------------------
# Sampled outputs for large workloads: the same per-row / per-vocab-row
# definitions evaluated only where asked.
# ----------------------------------------------------------------------------
def forward_rows(X, W, labels, rows: Sequence[int], ignore_index: int = IGNORE_INDEX,
                 smoothing: float = 0.0, z_loss: float = 0.0):
    """(lse, row_loss, m) of the selected token rows."""
    rows = np.asarray(rows, dtype=np.int64)
    Wd = upcast(W)
    V = Wd.shape[0]
    lab = np.asarray(labels, dtype=np.int64)[rows]
    valid = valid_mask(lab, V, ignore_index)
    Z = upcast(np.asarray(X)[rows]) @ Wd.T
    m, _, lse = row_logsumexp(Z)
    return lse, row_losses(Z, lse, lab, valid, smoothing, z_loss), m


def dx_rows(X, W, labels, rows: Sequence[int], c: float,
            ignore_index: int = IGNORE_INDEX, smoothing: float = 0.0,
            z_loss: float = 0.0) -> np.ndarray:
    """dX_i = sum_j dZ_ij W_j for the selected token rows."""
    rows = np.asarray(rows, dtype=np.int64)
    Wd = upcast(W)
    V = Wd.shape[0]
    lab = np.asarray(labels, dtype=np.int64)[rows]
    valid = valid_mask(lab, V, ignore_index)
    Z = upcast(np.asarray(X)[rows]) @ Wd.T
    _, _, lse = row_logsumexp(Z)
    return dlogits(Z, lse, lab, valid, c, smoothing, z_loss) @ Wd


def dw_rows(X, W, labels, vocab_rows: Sequence[int], lse: np.ndarray, c: float,
            ignore_index: int = IGNORE_INDEX, smoothing: float = 0.0,
            z_loss: float = 0.0) -> np.ndarray:
    """dW_j = sum_i dZ_ij X_i for the selected vocabulary rows j.

    ``lse`` must be the oracle's own lse of every token row (from ``forward``)."""
    vocab_rows = np.asarray(vocab_rows, dtype=np.int64)
    Xd = upcast(X)
    Wd = upcast(W)
    V = Wd.shape[0]
    labels = np.asarray(labels, dtype=np.int64)
    valid = valid_mask(labels, V, ignore_index)
    Zc = Xd @ Wd[vocab_rows].T                   # N x J columns of Z
    Pc = np.exp(Zc - lse[:, None])
    if z_loss != 0.0:
        Pc = Pc * (1.0 + 2.0 * z_loss * lse)[:, None]
    dZc = Pc - smoothing / V
    hit = valid[:, None] & (labels[:, None] == vocab_rows[None, :])
    dZc = dZc - (1.0 - smoothing) * hit
    dZc[~valid] = 0.0
    return c * (dZc.T @ Xd)


def fwd_bwd(X, W, labels, ignore_index: int = IGNORE_INDEX, smoothing: float = 0.0,
            reduction: str = "mean", grad_loss: float = 1.0,
            dW_in: Optional[np.ndarray] = None, z_loss: float = 0.0):
    """Forward and backward of one batch (what one fused call produces)."""
    f = forward(X, W, labels, ignore_index, smoothing, reduction, z_loss=z_loss)
    b = backward(X, W, labels, ignore_index, smoothing, reduction, grad_loss, dW_in,
                 z_loss=z_loss)
    return f, b


# ----------------------------------------------------------------------------
# Vocabulary-parallel decomposition ([CFCE] step 2's running (m, d) carried
# across vocabulary shards instead of tiles; [CFCE] comparison table:
# "Tiled vocabulary dot products").  Shard p holds W rows [v0, v0 + V_p) of a
# vocabulary of V_total; labels stay global.
# ----------------------------------------------------------------------------
def shard_partials(X, W_shard, labels, v0: int, V_total: int,
                   ignore_index: int = IGNORE_INDEX):
    """Per-row (m, d, z_y, sum_z) of this shard: m = max over the shard's
    logits, d = sum exp(z - m), z_y = the target logit if y_i lies in the
    shard (else 0), sum_z = the shard's row sum of logits."""
    Z = upcast(X) @ upcast(W_shard).T
    m = Z.max(axis=1)
    d = np.exp(Z - m[:, None]).sum(axis=1)
    labels = np.asarray(labels, dtype=np.int64)
    rel = labels - v0
    mine = (labels != ignore_index) & (rel >= 0) & (rel < Z.shape[1])
    z_y = np.zeros(Z.shape[0])
    rows = np.flatnonzero(mine)
    z_y[rows] = Z[rows, rel[rows]]
    return m, d, z_y, Z.sum(axis=1)


def combine_partials(parts, labels, V_total: int, ignore_index: int = IGNORE_INDEX,
                     smoothing: float = 0.0, reduction: str = "mean", z_loss: float = 0.0):
    """LSE-combine of the shards' (m, d, z_y, sum_z): M = max_p m_p,
    lse = M + log sum_p d_p exp(m_p - M); z_y and sum_z add up.  Returns
    (loss, lse, row_loss, n_valid) with the same loss as ``forward``."""
    m = np.stack([p[0] for p in parts])
    d = np.stack([p[1] for p in parts])
    M = m.max(axis=0)
    lse = M + np.log((d * np.exp(m - M)).sum(axis=0))
    z_y = sum(p[2] for p in parts)
    zs = sum(p[3] for p in parts)
    labels = np.asarray(labels, dtype=np.int64)
    valid = valid_mask(labels, V_total, ignore_index)
    row = lse - (1.0 - smoothing) * z_y - (smoothing / V_total) * zs + z_loss * lse * lse
    row = np.where(valid, row, 0.0)
    nv = int(valid.sum())
    total = float(row.sum())
    loss = total if reduction == "sum" else (total / nv if nv else 0.0)
    return loss, lse, row, nv


def shard_backward(X, W_shard, labels, v0: int, V_total: int, lse: np.ndarray, c: float,
                   ignore_index: int = IGNORE_INDEX, smoothing: float = 0.0,
                   z_loss: float = 0.0):
    """This shard's dZ columns (global lse, eps / V_total), its partial
    dX = dZ_p W_p (to be summed over shards) and its dW rows."""
    Xd, Wd = upcast(X), upcast(W_shard)
    Z = Xd @ Wd.T
    labels = np.asarray(labels, dtype=np.int64)
    valid = valid_mask(labels, V_total, ignore_index)
    P = np.exp(Z - lse[:, None])
    if z_loss != 0.0:
        P = P * (1.0 + 2.0 * z_loss * lse)[:, None]
    dZ = P - smoothing / V_total
    rel = labels - v0
    hit = valid & (rel >= 0) & (rel < Z.shape[1])
    rows = np.flatnonzero(hit)
    dZ[rows, rel[rows]] -= (1.0 - smoothing)
    dZ[~valid] = 0.0
    dZ *= c
    return dZ @ Wd, dZ.T @ Xd
