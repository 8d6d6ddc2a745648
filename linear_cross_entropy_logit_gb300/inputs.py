"""Seeded synthetic workloads for the fused linear cross-entropy path.

This module only draws numbers: it holds none of the loss or gradient
arithmetic, and it is the one piece shared by the CUDA path's tests and bench
and by the fp64 oracle's tests.  Both sides receive the very same bits.

Workload shapes follow the model families the pages discuss ("Chunked and
Fused Cross-Entropy ...", section "The Vocabulary Memory Wall in Modern LLMs"
and the "VRAM Footprint Across Model Families" table; "Fused cross-entropy --
the memory kernel", table "Why logits are the biggest tensor in the model"):
Llama-3 (H=4096, V=128256), Qwen-2.5 (H=3584, V=152064) and Gemma-2-2B
(H=2304, V=256000).  No dataset exists here; every tensor is synthetic.

Recipe (seed ``s``; tensor index ``k``: 0 X, 1 W, 2 labels, 3 ignore
positions, 4 Zipf rank-to-token permutation, 5 scaled W rows):
  * X, W: standard normals drawn in float32 with numpy's PCG64, in row blocks
    of ``BLOCK_ROWS`` rows, block ``b`` seeded by ``SeedSequence([s, k, b])``;
    multiplied by the stated standard deviation in float32, then rounded to
    nearest-even bfloat16 (bf16 configs) or kept as float32 (fp32 configs).
  * "RMS-normed rows": each X row divided by its float32 RMS before rounding.
  * labels: uniform integers in [0, V), or a finite Zipf law P(r) ~ r^-s over
    ranks r = 1..V drawn by inverse CDF, rank mapped to a token id through a
    seeded permutation of [0, V).
  * ignore positions: the first ``n_ignore`` entries of a seeded permutation
    of [0, N) get the label ``ignore_index``.
  * peaked logits (``x_align`` > 0): after the labels are drawn, each valid row
    x_i gets x_align * u_{y_i} added before rounding, u_j = W_j scaled to unit
    RMS, so the target's logit stands out as it does for a trained model.
  * instruction-tuning masks (``labels="sft"``): N tokens are sequences of
    ``seq_len``; sequence b ignores its first floor(u_b * seq_len) tokens (the
    prompt), u_b uniform in ``prompt_frac``, drawn from stream k = 6; the other
    labels are uniform.
  * scaled W rows: ``n_scaled`` distinct rows chosen by a seeded permutation,
    multiplied by ``row_scale`` before rounding.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

BLOCK_ROWS = 4096
IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    N: int
    H: int
    V: int
    dtype: str  # "bf16" or "fp32": storage type of X and W
    x_std: float = 1.0
    w_std: float = 0.02
    x_rms_rows: bool = False
    labels: str = "uniform"  # "uniform" or "zipf"
    zipf_s: float = 1.1
    n_ignore: int = 0
    smoothing: float = 0.0
    n_scaled_w_rows: int = 0
    w_row_scale: float = 1.0
    ignore_index: int = IGNORE_INDEX
    reduction: str = "mean"
    seq_len: int = 0                       # "sft" labels: tokens per sequence
    x_align: float = 0.0                   # pull each x_i towards its target's W row
    prompt_frac: tuple = (0.2, 0.8)        # "sft" labels: masked prompt share per sequence

    @property
    def flops_fwd_bwd(self) -> float:
        """Dense-GEMM work of one forward+backward: 4 GEMMs of 2*N*V*H."""
        return 8.0 * self.N * self.V * self.H


# The five workloads: a small fp32 case, then the three model families.
TINY = WorkloadSpec("tiny", N=256, H=256, V=4096, dtype="fp32")
LLAMA = WorkloadSpec("llama3_n8192", N=8192, H=4096, V=128256, dtype="bf16",
                     x_rms_rows=True, n_ignore=round(0.05 * 8192))
LLAMA_LONG = WorkloadSpec("llama3_long_n16384", N=16384, H=4096, V=128256,
                          dtype="bf16", labels="zipf",
                          n_ignore=int(0.10 * 16384))
QWEN = WorkloadSpec("qwen25_n16384", N=16384, H=3584, V=152064, dtype="bf16",
                    n_ignore=int(0.10 * 16384), smoothing=0.1)
GEMMA = WorkloadSpec("gemma2_n32768", N=32768, H=2304, V=256000, dtype="bf16",
                     labels="zipf", n_ignore=int(0.05 * 32768),
                     n_scaled_w_rows=2560, w_row_scale=8.0)

# Peaked logits on the Llama-3 shape (target logit ~ 15 above the rest's
# spread): the regime where gradient filtering drops most of dZ.
LLAMA_PEAKED = WorkloadSpec("llama3_peaked_n8192", N=8192, H=4096, V=128256, dtype="bf16",
                            n_ignore=round(0.05 * 8192), x_align=0.18)

# Instruction tuning on the Llama-3 shape: 4 sequences of 4096 tokens whose
# prompts (20-80% of each sequence) are masked ("Chunked and Fused
# Cross-Entropy ...", "Numerical Considerations ...", item 2).
LLAMA_SFT = WorkloadSpec("llama3_sft_n16384", N=16384, H=4096, V=128256, dtype="bf16",
                         labels="sft", seq_len=4096)

CONFIGS = {s.name: s for s in (TINY, LLAMA, LLAMA_LONG, QWEN, GEMMA, LLAMA_SFT, LLAMA_PEAKED)}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to nearest-even bfloat16; return the uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, k: int, b: Optional[int] = None) -> np.random.Generator:
    key = [seed, k] if b is None else [seed, k, b]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def _normal_matrix(seed: int, k: int, rows: int, cols: int, std: float,
                   rms_rows: bool, to_bf16: bool,
                   scale_rows: Optional[np.ndarray] = None,
                   row_scale: float = 1.0) -> np.ndarray:
    """rows x cols draws, returned as bf16 bits (uint16) or float32 values."""
    out = np.empty((rows, cols), dtype=np.uint16 if to_bf16 else np.float32)
    scale_mask = None
    if scale_rows is not None and len(scale_rows):
        scale_mask = np.zeros(rows, dtype=bool)
        scale_mask[scale_rows] = True
    nblk = (rows + BLOCK_ROWS - 1) // BLOCK_ROWS

    def one(b: int) -> None:
        r0, r1 = b * BLOCK_ROWS, min(rows, (b + 1) * BLOCK_ROWS)
        v = _rng(seed, k, b).standard_normal((r1 - r0, cols), dtype=np.float32)
        v *= np.float32(std)
        if rms_rows:
            rms = np.sqrt(np.mean(v.astype(np.float64) ** 2, axis=1)).astype(np.float32)
            v /= rms[:, None]
        if scale_mask is not None:
            m = scale_mask[r0:r1]
            if m.any():
                v[m] *= np.float32(row_scale)
        out[r0:r1] = f32_to_bf16_bits(v) if to_bf16 else v

    if nblk == 1:
        one(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(nblk)))
    return out


def zipf_labels(rng_u: np.random.Generator, rng_perm: np.random.Generator,
                n: int, V: int, s: float) -> np.ndarray:
    """Finite Zipf(s) over ranks 1..V by inverse CDF, ranks mapped to token ids."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng_u.random(n)
    rank = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)
    perm = rng_perm.permutation(V)
    return perm[rank].astype(np.int64)


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    x: np.ndarray       # N x H: uint16 bf16 bits or float32
    w: np.ndarray       # V x H: uint16 bf16 bits or float32
    labels: np.ndarray  # N int64, ignore_index marks ignored rows

    @property
    def N(self) -> int:
        return self.spec.N

    @property
    def H(self) -> int:
        return self.spec.H

    @property
    def V(self) -> int:
        return self.spec.V

    @property
    def dtype(self) -> str:
        return self.spec.dtype

    def x_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.x) if self.dtype == "bf16" else self.x

    def w_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.w) if self.dtype == "bf16" else self.w


def make_labels(spec: WorkloadSpec, seed: int, N: Optional[int] = None) -> np.ndarray:
    N = spec.N if N is None else N
    if spec.labels == "uniform":
        labels = _rng(seed, 2).integers(0, spec.V, size=N, dtype=np.int64)
    elif spec.labels == "zipf":
        labels = zipf_labels(_rng(seed, 2), _rng(seed, 4), N, spec.V, spec.zipf_s)
    elif spec.labels == "sft":
        labels = _rng(seed, 2).integers(0, spec.V, size=N, dtype=np.int64)
        S = spec.seq_len if spec.seq_len > 0 else N
        n_seq = (N + S - 1) // S
        u = _rng(seed, 6).uniform(spec.prompt_frac[0], spec.prompt_frac[1], size=n_seq)
        for b in range(n_seq):
            start = b * S
            labels[start:min(N, start + int(u[b] * S))] = spec.ignore_index
    else:
        raise ValueError(f"unknown label law {spec.labels!r}")
    n_ign = min(spec.n_ignore, N)
    if n_ign:
        pos = _rng(seed, 3).permutation(N)[:n_ign]
        labels[pos] = spec.ignore_index
    return labels


def make_workload(spec: WorkloadSpec | str, seed: int = 0) -> Workload:
    """Draw the workload ``spec`` with ``seed`` (same bits on every call)."""
    if isinstance(spec, str):
        spec = CONFIGS[spec]
    bf16 = spec.dtype == "bf16"
    if spec.dtype not in ("bf16", "fp32"):
        raise ValueError(f"unknown dtype {spec.dtype!r}")
    x = _normal_matrix(seed, 0, spec.N, spec.H, spec.x_std, spec.x_rms_rows,
                       bf16 and not spec.x_align)
    scaled = None
    if spec.n_scaled_w_rows:
        scaled = _rng(seed, 5).permutation(spec.V)[:spec.n_scaled_w_rows]
    w = _normal_matrix(seed, 1, spec.V, spec.H, spec.w_std, False, bf16,
                       scale_rows=scaled, row_scale=spec.w_row_scale)
    labels = make_labels(spec, seed)
    if spec.x_align:
        wf = bf16_bits_to_f32(w) if bf16 else w
        rows = np.flatnonzero(labels != spec.ignore_index)
        for r0 in range(0, len(rows), 4096):
            rr = rows[r0:r0 + 4096]
            u = wf[labels[rr]].astype(np.float32)
            u /= np.sqrt(np.mean(u.astype(np.float64) ** 2, axis=1)).astype(np.float32)[:, None]
            x[rr] += np.float32(spec.x_align) * u
        if bf16:
            x = f32_to_bf16_bits(x)
    return Workload(spec, seed, x, w, labels)


def custom_spec(name: str = "custom", **kw) -> WorkloadSpec:
    """A workload of arbitrary shape with the same recipe (used for parity cases)."""
    return WorkloadSpec(name=name, **kw)
