"""Thin ctypes binding of ``libflce.so`` (include/flce.h).

Argument marshalling only: every step of the forward and backward runs in the
library's CUDA kernels.  PyTorch provides device memory and the stream.  If the
library is missing, ``lib()`` raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libflce.so")
# The same library built with FLCE_DEBUG: index math range-checked on the
# device (an out-of-range index sets FLCE_ERR_BOUNDS instead of being used).
DEBUG_LIB_PATH = os.path.join(_HERE, "_lib", "libflce_debug.so")

FLCE_OK = 0
FLCE_ERR_ARG = 1
FLCE_ERR_UNSUPPORTED = 2
FLCE_ERR_WORKSPACE = 3
FLCE_ERR_LABEL = 4
FLCE_ERR_TIMEOUT = 5
FLCE_ERR_CUDA = 6
FLCE_ERR_BOUNDS = 7

FLCE_BF16 = 0
FLCE_FP32 = 1
FLCE_MEAN = 0
FLCE_SUM = 1
MODE_FWD = 1
MODE_BWD = 2
MODE_FWD_BWD = 3

EXPORTED = (
    "flce_workspace_size", "flce_set_vocab_chunk", "flce_vocab_chunk", "flce_forward",
    "flce_backward", "flce_fwd_bwd", "flce_status_string", "flce_last_cuda_error",
    "flce_last_launch_count", "flce_abi_version", "flce_debug_gemm", "flce_profile_enable",
    "flce_profile_read", "flce_profile_reset", "flce_forward_noalloc", "flce_noalloc_last_error",
    "flce_set_cta_pair", "flce_cta_pair", "flce_set_l2_hints", "flce_options_init",
    "flce_forward_ex", "flce_backward_ex", "flce_fwd_bwd_ex", "flce_forward_vocab_shard",
    "flce_combine_workspace_size", "flce_combine_vocab_shards", "flce_backward_vocab_shard",
    "flce_debug_wait_timeout", "flce_set_backward_merge", "flce_backward_merge",
    "flce_workspace_size_ex", "flce_vocab_chunk_ex", "flce_set_cluster_multicast",
    "flce_cluster_multicast", "flce_debug_last_multicast_launches",
)

PROFILE_KINDS = ("fwd_logits_lse", "bwd_dz_recompute", "bwd_dw_gemm", "bwd_dx_gemm",
                 "bwd_merged")

_lib = None


class FlceOptions(ctypes.Structure):
    """Mirror of ``flce_options`` in include/flce.h."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("ignore_index", ctypes.c_int64),
                ("smoothing", ctypes.c_float), ("z_loss", ctypes.c_float),
                ("reduction", ctypes.c_int), ("row_loss", ctypes.c_void_p),
                ("skip_ignored_blocks", ctypes.c_int), ("grad_filter", ctypes.c_float),
                ("cta_pair", ctypes.c_int), ("backward_merge", ctypes.c_int),
                ("l2_hints", ctypes.c_int), ("vocab_chunk", ctypes.c_int64),
                ("cluster_multicast", ctypes.c_int)]


class FlceError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == FLCE_ERR_CUDA:
            detail = " (" + lib().flce_last_cuda_error().decode() + ")"
        super().__init__(f"{what}: {lib().flce_status_string(status).decode()}{detail}")


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def use_library(L: Optional[ctypes.CDLL]) -> Optional[ctypes.CDLL]:
    """Make every wrapper below call ``L`` (e.g. ``load(DEBUG_LIB_PATH)``);
    returns the library used before.  ``None`` goes back to the default."""
    global _lib
    prev = _lib
    _lib = L
    return prev


def load(path: str) -> ctypes.CDLL:
    """Open a build of the library and declare its C signatures."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with "
            "`python -m linear_cross_entropy_logit_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    P, I64, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.flce_workspace_size.argtypes = [I64, I64, I64, I32, I32]
    L.flce_workspace_size.restype = SZ
    L.flce_set_vocab_chunk.argtypes = [I64]
    L.flce_set_vocab_chunk.restype = I32
    L.flce_vocab_chunk.argtypes = [I64, I64, I64]
    L.flce_vocab_chunk.restype = I64
    L.flce_forward.argtypes = [P, P, P, I64, I64, I64, I64, F32, I32, I32, P, P, P, P, SZ, P, P]
    L.flce_forward.restype = I32
    L.flce_backward.argtypes = [P, P, P, I64, I64, I64, I64, F32, I32, I32, P, P, P, P, P, I32,
                                P, SZ, P, P]
    L.flce_backward.restype = I32
    L.flce_fwd_bwd.argtypes = [P, P, P, I64, I64, I64, I64, F32, I32, I32, P, P, P, P, P, P, I32,
                               P, SZ, P, P]
    L.flce_fwd_bwd.restype = I32
    L.flce_status_string.argtypes = [I32]
    L.flce_status_string.restype = ctypes.c_char_p
    L.flce_last_cuda_error.argtypes = []
    L.flce_last_cuda_error.restype = ctypes.c_char_p
    L.flce_last_launch_count.argtypes = []
    L.flce_last_launch_count.restype = I32
    L.flce_abi_version.argtypes = []
    L.flce_abi_version.restype = I32
    L.flce_debug_gemm.argtypes = [P, P, P, I64, I64, I64, I32, I32, I32, P, P]
    L.flce_debug_gemm.restype = I32
    L.flce_profile_enable.argtypes = [I32]
    L.flce_profile_enable.restype = I32
    L.flce_profile_read.argtypes = [I32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I32)]
    L.flce_profile_read.restype = I32
    L.flce_profile_reset.argtypes = []
    L.flce_profile_reset.restype = None
    L.flce_forward_noalloc.argtypes = [P, P, P, I64, I64, I64, I64, F32, I32, P, P, P, P, P]
    L.flce_forward_noalloc.restype = I32
    L.flce_noalloc_last_error.argtypes = []
    L.flce_noalloc_last_error.restype = ctypes.c_char_p
    L.flce_set_cta_pair.argtypes = [I32]
    L.flce_set_cta_pair.restype = I32
    L.flce_cta_pair.argtypes = []
    L.flce_cta_pair.restype = I32
    L.flce_set_l2_hints.argtypes = [I32]
    L.flce_set_l2_hints.restype = I32
    L.flce_set_backward_merge.argtypes = [I32]
    L.flce_set_backward_merge.restype = I32
    L.flce_backward_merge.argtypes = []
    L.flce_backward_merge.restype = I32
    OPT = ctypes.POINTER(FlceOptions)
    L.flce_options_init.argtypes = [OPT]
    L.flce_options_init.restype = None
    L.flce_forward_ex.argtypes = [P, P, P, I64, I64, I64, I32, OPT, P, P, P, P, SZ, P, P]
    L.flce_forward_ex.restype = I32
    L.flce_backward_ex.argtypes = [P, P, P, I64, I64, I64, I32, OPT, P, P, P, P, P, I32, P, SZ,
                                   P, P]
    L.flce_backward_ex.restype = I32
    L.flce_fwd_bwd_ex.argtypes = [P, P, P, I64, I64, I64, I32, OPT, P, P, P, P, P, P, I32, P, SZ,
                                  P, P]
    L.flce_fwd_bwd_ex.restype = I32
    L.flce_forward_vocab_shard.argtypes = [P, P, P, I64, I64, I64, I64, I64, I32, OPT, P, P, SZ,
                                           P, P]
    L.flce_forward_vocab_shard.restype = I32
    L.flce_combine_workspace_size.argtypes = [I64]
    L.flce_combine_workspace_size.restype = SZ
    L.flce_combine_vocab_shards.argtypes = [P, I32, I64, P, I64, OPT, P, P, P, P, SZ, P, P]
    L.flce_combine_vocab_shards.restype = I32
    L.flce_backward_vocab_shard.argtypes = [P, P, P, I64, I64, I64, I64, I64, I32, OPT, P, P, P,
                                            P, P, I32, P, SZ, P, P]
    L.flce_backward_vocab_shard.restype = I32
    L.flce_debug_wait_timeout.argtypes = [P, ctypes.c_uint64, P, P]
    L.flce_debug_wait_timeout.restype = I32
    L.flce_workspace_size_ex.argtypes = [I64, I64, I64, I32, I32, OPT]
    L.flce_workspace_size_ex.restype = SZ
    L.flce_vocab_chunk_ex.argtypes = [I64, I64, I64, OPT]
    L.flce_vocab_chunk_ex.restype = I64
    L.flce_set_cluster_multicast.argtypes = [I32]
    L.flce_set_cluster_multicast.restype = I32
    L.flce_cluster_multicast.argtypes = []
    L.flce_cluster_multicast.restype = I32
    L.flce_debug_last_multicast_launches.argtypes = []
    L.flce_debug_last_multicast_launches.restype = I32
    return L


def _check(status: int, what: str) -> None:
    if status != FLCE_OK:
        raise FlceError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FLCE_BF16
    if t.dtype == torch.float32:
        return FLCE_FP32
    raise TypeError(f"X and W must be bfloat16 or float32, got {t.dtype}")


def _red_code(reduction: str) -> int:
    if reduction == "mean":
        return FLCE_MEAN
    if reduction == "sum":
        return FLCE_SUM
    raise ValueError(f"reduction must be 'mean' or 'sum', got {reduction!r}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_inputs(X, W, labels):
    for name, t in (("X", X), ("W", W), ("labels", labels)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if X.dtype != W.dtype:
        raise TypeError("X and W must have the same dtype")
    if labels.dtype != torch.int64:
        raise TypeError("labels must be int64")
    N, H = X.shape
    V, H2 = W.shape
    if H2 != H or labels.shape != (N,):
        raise ValueError(f"shape mismatch: X {tuple(X.shape)}, W {tuple(W.shape)}, labels {tuple(labels.shape)}")
    return N, H, V


def flce_workspace_size(N: int, H: int, V: int, dtype: int = FLCE_BF16, mode: int = MODE_FWD_BWD,
                        options: Optional["FlceOptions"] = None) -> int:
    """Workspace bytes; with ``options`` the launch settings are taken from them
    (flce_workspace_size_ex), else from the process-wide defaults."""
    if options is None:
        return int(lib().flce_workspace_size(N, H, V, dtype, mode))
    return int(lib().flce_workspace_size_ex(N, H, V, dtype, mode, ctypes.byref(options)))


def flce_set_vocab_chunk(cols: int) -> None:
    _check(lib().flce_set_vocab_chunk(cols), "flce_set_vocab_chunk")


def flce_set_cta_pair(on: bool) -> None:
    """1: 256 x 256 tiles on CTA pairs (default); 0: 128 x 256 tiles on single CTAs."""
    _check(lib().flce_set_cta_pair(int(bool(on))), "flce_set_cta_pair")


def flce_set_l2_hints(on: bool) -> None:
    _check(lib().flce_set_l2_hints(int(bool(on))), "flce_set_l2_hints")


def flce_cta_pair() -> bool:
    return bool(lib().flce_cta_pair())


def flce_set_cluster_multicast(on: bool) -> None:
    """1: pair launches whose tiles pair up take 4-CTA clusters with operand
    multicast (default); 0: plain CTA pairs.  Bit-identical results."""
    _check(lib().flce_set_cluster_multicast(int(bool(on))), "flce_set_cluster_multicast")


def flce_cluster_multicast() -> bool:
    return bool(lib().flce_cluster_multicast())


def flce_set_backward_merge(mode) -> None:
    """Backward layout: 0 three launches per chunk (default); 1 (or True) one
    merged dW(c) + dX(c) + dZ(c+1) launch per chunk (two dZ buffers); 2 the dZ
    recompute alone, then one merged dW(c) + dX(c) launch (one dZ buffer)."""
    _check(lib().flce_set_backward_merge(int(mode)), "flce_set_backward_merge")


def flce_backward_merge() -> int:
    return int(lib().flce_backward_merge())


def flce_vocab_chunk(N: int, H: int, V: int, options: Optional["FlceOptions"] = None) -> int:
    if options is None:
        return int(lib().flce_vocab_chunk(N, H, V))
    return int(lib().flce_vocab_chunk_ex(N, H, V, ctypes.byref(options)))


def workspace(N: int, H: int, V: int, dtype: int, mode: int, device,
              options: Optional["FlceOptions"] = None) -> torch.Tensor:
    """A workspace of the required size (torch-allocated, 256-byte aligned)."""
    n = flce_workspace_size(N, H, V, dtype, mode, options)
    if n == 0:
        raise ValueError(f"no workspace plan for N={N}, H={H}, V={V} with these options")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def new_err_word(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def make_options(ignore_index: int = -100, smoothing: float = 0.0, reduction: str = "mean",
                 z_loss: float = 0.0, row_loss=None, skip_ignored_blocks: bool = False,
                 grad_filter: float = 0.0, *, cta_pair: Optional[bool] = None,
                 backward_merge: Optional[int] = None, l2_hints: Optional[bool] = None,
                 vocab_chunk: Optional[int] = None,
                 cluster_multicast: Optional[bool] = None) -> FlceOptions:
    """An ``flce_options``; the launch settings left at None take the
    process-wide defaults at the time of each call."""
    o = FlceOptions()
    lib().flce_options_init(ctypes.byref(o))
    o.ignore_index = ignore_index
    o.smoothing = smoothing
    o.z_loss = z_loss
    o.reduction = _red_code(reduction)
    o.row_loss = _ptr(row_loss)
    o.skip_ignored_blocks = int(bool(skip_ignored_blocks))
    o.grad_filter = grad_filter
    if cta_pair is not None:
        o.cta_pair = int(bool(cta_pair))
    if backward_merge is not None:
        o.backward_merge = int(backward_merge)
    if l2_hints is not None:
        o.l2_hints = int(bool(l2_hints))
    if vocab_chunk is not None:
        o.vocab_chunk = int(vocab_chunk)
    if cluster_multicast is not None:
        o.cluster_multicast = int(bool(cluster_multicast))
    return o


def flce_forward(X, W, labels, ignore_index: int = -100, smoothing: float = 0.0,
                 reduction: str = "mean", *, loss=None, lse=None, valid_count=None,
                 workspace_buf=None, err_word=None, stream=None, z_loss: float = 0.0,
                 row_loss=None, skip_ignored_blocks: bool = False):
    """Returns (loss[1] fp32, lse[N] fp32, valid_count[1] int32, err_word[1] int32).
    With z_loss, row_loss or skip_ignored_blocks set it calls flce_forward_ex."""
    if z_loss or row_loss is not None or skip_ignored_blocks:
        return flce_forward_ex(X, W, labels, make_options(ignore_index, smoothing, reduction,
                                                          z_loss, row_loss, skip_ignored_blocks),
                               loss=loss, lse=lse, valid_count=valid_count,
                               workspace_buf=workspace_buf, err_word=err_word, stream=stream)
    N, H, V = _check_inputs(X, W, labels)
    dev = X.device
    dt = _dtype_code(X)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(N, dtype=torch.float32, device=dev) if lse is None else lse
    valid_count = torch.empty(1, dtype=torch.int32, device=dev) if valid_count is None else valid_count
    ws = workspace(N, H, V, dt, MODE_FWD, dev) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_forward(_ptr(X), _ptr(W), _ptr(labels), N, H, V, ignore_index, smoothing, dt,
                            _red_code(reduction), _ptr(loss), _ptr(lse), _ptr(valid_count),
                            _ptr(ws), ws.numel(), _ptr(err_word), _stream(stream))
    _check(st, "flce_forward")
    return loss, lse, valid_count, err_word


def flce_forward_ex(X, W, labels, options: FlceOptions, *, loss=None, lse=None,
                    valid_count=None, workspace_buf=None, err_word=None, stream=None):
    N, H, V = _check_inputs(X, W, labels)
    dev = X.device
    dt = _dtype_code(X)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(N, dtype=torch.float32, device=dev) if lse is None else lse
    valid_count = torch.empty(1, dtype=torch.int32, device=dev) if valid_count is None else valid_count
    ws = workspace(N, H, V, dt, MODE_FWD, dev, options) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_forward_ex(_ptr(X), _ptr(W), _ptr(labels), N, H, V, dt, ctypes.byref(options),
                               _ptr(loss), _ptr(lse), _ptr(valid_count), _ptr(ws), ws.numel(),
                               _ptr(err_word), _stream(stream))
    _check(st, "flce_forward_ex")
    return loss, lse, valid_count, err_word


def flce_backward(X, W, labels, lse, valid_count, ignore_index: int = -100,
                  smoothing: float = 0.0, reduction: str = "mean", *, grad_loss=None,
                  dX=None, dW=None, accumulate_dW: bool = False, workspace_buf=None,
                  err_word=None, stream=None, z_loss: float = 0.0,
                  skip_ignored_blocks: bool = False, grad_filter: float = 0.0):
    """Returns (dX [N, H] in X's dtype, dW [V, H] fp32, err_word).
    With z_loss, skip_ignored_blocks or grad_filter set it calls flce_backward_ex."""
    if z_loss or skip_ignored_blocks or grad_filter:
        return flce_backward_ex(X, W, labels, lse, valid_count,
                                make_options(ignore_index, smoothing, reduction, z_loss,
                                             skip_ignored_blocks=skip_ignored_blocks,
                                             grad_filter=grad_filter),
                                grad_loss=grad_loss, dX=dX, dW=dW, accumulate_dW=accumulate_dW,
                                workspace_buf=workspace_buf, err_word=err_word, stream=stream)
    N, H, V = _check_inputs(X, W, labels)
    dev = X.device
    dt = _dtype_code(X)
    dX = torch.empty_like(X) if dX is None else dX
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws = workspace(N, H, V, dt, MODE_BWD, dev) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_backward(_ptr(X), _ptr(W), _ptr(labels), N, H, V, ignore_index, smoothing, dt,
                             _red_code(reduction), _ptr(lse), _ptr(valid_count), _ptr(grad_loss),
                             _ptr(dX), _ptr(dW), int(bool(accumulate_dW)), _ptr(ws), ws.numel(),
                             _ptr(err_word), _stream(stream))
    _check(st, "flce_backward")
    return dX, dW, err_word


def flce_backward_ex(X, W, labels, lse, valid_count, options: FlceOptions, *, grad_loss=None,
                     dX=None, dW=None, accumulate_dW: bool = False, workspace_buf=None,
                     err_word=None, stream=None):
    N, H, V = _check_inputs(X, W, labels)
    dev = X.device
    dt = _dtype_code(X)
    dX = torch.empty_like(X) if dX is None else dX
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws = workspace(N, H, V, dt, MODE_BWD, dev, options) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_backward_ex(_ptr(X), _ptr(W), _ptr(labels), N, H, V, dt,
                                ctypes.byref(options), _ptr(lse), _ptr(valid_count),
                                _ptr(grad_loss), _ptr(dX), _ptr(dW), int(bool(accumulate_dW)),
                                _ptr(ws), ws.numel(), _ptr(err_word), _stream(stream))
    _check(st, "flce_backward_ex")
    return dX, dW, err_word


def flce_fwd_bwd(X, W, labels, ignore_index: int = -100, smoothing: float = 0.0,
                 reduction: str = "mean", *, grad_loss=None, loss=None, lse=None,
                 valid_count=None, dX=None, dW=None, accumulate_dW: bool = False,
                 workspace_buf=None, err_word=None, stream=None, z_loss: float = 0.0,
                 row_loss=None, skip_ignored_blocks: bool = False, grad_filter: float = 0.0):
    """Returns (loss, lse, valid_count, dX, dW, err_word).
    With z_loss, row_loss, skip_ignored_blocks or grad_filter set it calls flce_fwd_bwd_ex."""
    if z_loss or row_loss is not None or skip_ignored_blocks or grad_filter:
        return flce_fwd_bwd_ex(X, W, labels, make_options(ignore_index, smoothing, reduction,
                                                          z_loss, row_loss, skip_ignored_blocks,
                                                          grad_filter),
                               grad_loss=grad_loss, loss=loss, lse=lse, valid_count=valid_count,
                               dX=dX, dW=dW, accumulate_dW=accumulate_dW,
                               workspace_buf=workspace_buf, err_word=err_word, stream=stream)
    N, H, V = _check_inputs(X, W, labels)
    dev = X.device
    dt = _dtype_code(X)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(N, dtype=torch.float32, device=dev) if lse is None else lse
    valid_count = torch.empty(1, dtype=torch.int32, device=dev) if valid_count is None else valid_count
    dX = torch.empty_like(X) if dX is None else dX
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws = workspace(N, H, V, dt, MODE_FWD_BWD, dev) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_fwd_bwd(_ptr(X), _ptr(W), _ptr(labels), N, H, V, ignore_index, smoothing, dt,
                            _red_code(reduction), _ptr(grad_loss), _ptr(loss), _ptr(lse),
                            _ptr(valid_count), _ptr(dX), _ptr(dW), int(bool(accumulate_dW)),
                            _ptr(ws), ws.numel(), _ptr(err_word), _stream(stream))
    _check(st, "flce_fwd_bwd")
    return loss, lse, valid_count, dX, dW, err_word


def flce_fwd_bwd_ex(X, W, labels, options: FlceOptions, *, grad_loss=None, loss=None, lse=None,
                    valid_count=None, dX=None, dW=None, accumulate_dW: bool = False,
                    workspace_buf=None, err_word=None, stream=None):
    N, H, V = _check_inputs(X, W, labels)
    dev = X.device
    dt = _dtype_code(X)
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(N, dtype=torch.float32, device=dev) if lse is None else lse
    valid_count = torch.empty(1, dtype=torch.int32, device=dev) if valid_count is None else valid_count
    dX = torch.empty_like(X) if dX is None else dX
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws = workspace(N, H, V, dt, MODE_FWD_BWD, dev, options) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_fwd_bwd_ex(_ptr(X), _ptr(W), _ptr(labels), N, H, V, dt, ctypes.byref(options),
                               _ptr(grad_loss), _ptr(loss), _ptr(lse), _ptr(valid_count),
                               _ptr(dX), _ptr(dW), int(bool(accumulate_dW)), _ptr(ws),
                               ws.numel(), _ptr(err_word), _stream(stream))
    _check(st, "flce_fwd_bwd_ex")
    return loss, lse, valid_count, dX, dW, err_word


def flce_forward_vocab_shard(X, W_shard, labels, vocab_offset: int, vocab_total: int,
                             options: FlceOptions = None, *, partials=None, workspace_buf=None,
                             err_word=None, stream=None):
    """This shard's per-row partial statistics, a float32 [N, 4] tensor."""
    N, H, Vs = _check_inputs(X, W_shard, labels)
    dev = X.device
    dt = _dtype_code(X)
    options = make_options() if options is None else options
    partials = torch.empty(N, 4, dtype=torch.float32, device=dev) if partials is None else partials
    ws = workspace(N, H, Vs, dt, MODE_FWD, dev, options) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_forward_vocab_shard(_ptr(X), _ptr(W_shard), _ptr(labels), N, H, Vs,
                                        vocab_offset, vocab_total, dt, ctypes.byref(options),
                                        _ptr(partials), _ptr(ws), ws.numel(), _ptr(err_word),
                                        _stream(stream))
    _check(st, "flce_forward_vocab_shard")
    return partials, err_word


def flce_combine_vocab_shards(partials, labels, vocab_total: int, options: FlceOptions = None, *,
                              loss=None, lse=None, valid_count=None, err_word=None, stream=None):
    """LSE-combine of P shards' partials (float32 [P, N, 4]) -> (loss, lse, valid_count, err)."""
    n_shards, N = partials.shape[0], partials.shape[1]
    dev = partials.device
    options = make_options() if options is None else options
    loss = torch.empty(1, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(N, dtype=torch.float32, device=dev) if lse is None else lse
    valid_count = torch.empty(1, dtype=torch.int32, device=dev) if valid_count is None else valid_count
    n = max(int(lib().flce_combine_workspace_size(N)), 256)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_combine_vocab_shards(_ptr(partials.contiguous()), n_shards, N, _ptr(labels),
                                         vocab_total, ctypes.byref(options), _ptr(loss), _ptr(lse),
                                         _ptr(valid_count), _ptr(ws), ws.numel(), _ptr(err_word),
                                         _stream(stream))
    _check(st, "flce_combine_vocab_shards")
    return loss, lse, valid_count, err_word


def flce_backward_vocab_shard(X, W_shard, labels, vocab_offset: int, vocab_total: int, lse,
                              valid_count, options: FlceOptions = None, *, grad_loss=None,
                              dX_partial=None, dW_shard=None, accumulate_dW: bool = False,
                              workspace_buf=None, err_word=None, stream=None):
    """(fp32 partial dX [N, H], dW rows of this shard [V_shard, H] fp32, err)."""
    N, H, Vs = _check_inputs(X, W_shard, labels)
    dev = X.device
    dt = _dtype_code(X)
    options = make_options() if options is None else options
    dX_partial = torch.empty(N, H, dtype=torch.float32, device=dev) if dX_partial is None else dX_partial
    dW_shard = torch.empty(Vs, H, dtype=torch.float32, device=dev) if dW_shard is None else dW_shard
    ws = workspace(N, H, Vs, dt, MODE_BWD, dev, options) if workspace_buf is None else workspace_buf
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_backward_vocab_shard(_ptr(X), _ptr(W_shard), _ptr(labels), N, H, Vs,
                                         vocab_offset, vocab_total, dt, ctypes.byref(options),
                                         _ptr(lse), _ptr(valid_count), _ptr(grad_loss),
                                         _ptr(dX_partial), _ptr(dW_shard), int(bool(accumulate_dW)),
                                         _ptr(ws), ws.numel(), _ptr(err_word), _stream(stream))
    _check(st, "flce_backward_vocab_shard")
    return dX_partial, dW_shard, err_word


def flce_debug_gemm(A, B, M: int, Nn: int, K: int, a_mn: bool, b_mn: bool, D=None,
                    accumulate: bool = False, err_word=None, stream=None):
    """Test-only: D (M x Nn fp32) = A B^T through the tcgen05 GEMM core."""
    dev = A.device
    D = torch.empty(M, Nn, dtype=torch.float32, device=dev) if D is None else D
    err_word = new_err_word(dev) if err_word is None else err_word
    st = lib().flce_debug_gemm(_ptr(A), _ptr(B), _ptr(D), M, Nn, K, int(a_mn), int(b_mn),
                               int(accumulate), _ptr(err_word), _stream(stream))
    _check(st, "flce_debug_gemm")
    return D, err_word


def flce_forward_noalloc(X, W, labels, ignore_index: int = -100, smoothing: float = 0.0,
                         reduction: str = "mean", *, loss, lse, valid_count, err_word,
                         stream=None):
    """Forward for callers that cannot allocate: every output buffer is the
    caller's and no workspace is passed (the library uses its own fixed device
    scratch).  bf16 X and W only.  Returns (loss, lse, valid_count, err_word)."""
    N, H, V = _check_inputs(X, W, labels)
    if X.dtype != torch.bfloat16:
        raise TypeError("flce_forward_noalloc takes bf16 X and W")
    st = lib().flce_forward_noalloc(_ptr(X), _ptr(W), _ptr(labels), N, H, V, ignore_index,
                                    smoothing, _red_code(reduction), _ptr(loss), _ptr(lse),
                                    _ptr(valid_count), _ptr(err_word), _stream(stream))
    if st != FLCE_OK:
        raise RuntimeError(f"flce_forward_noalloc: {lib().flce_status_string(st).decode()} "
                           f"({lib().flce_noalloc_last_error().decode()})")
    return loss, lse, valid_count, err_word


def last_launch_count() -> int:
    return int(lib().flce_last_launch_count())


def last_multicast_launches() -> int:
    """Test-only: launches of the last call made with the operand-multicast walk."""
    return int(lib().flce_debug_last_multicast_launches())


def flce_profile_enable(on: bool) -> None:
    _check(lib().flce_profile_enable(int(bool(on))), "flce_profile_enable")


def flce_profile_reset() -> None:
    lib().flce_profile_reset()


def flce_profile_read() -> dict:
    """{kind: (total_ms, launches)} accumulated since the last reset."""
    out = {}
    for k, name in enumerate(PROFILE_KINDS):
        ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
        _check(lib().flce_profile_read(k, ctypes.byref(ms), ctypes.byref(n)), "flce_profile_read")
        out[name] = (ms.value, n.value)
    return out


class _LinearCrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, W, labels, ignore_index, smoothing, reduction, z_loss):
        loss, lse, nv, err = flce_forward(X, W, labels, ignore_index, smoothing, reduction,
                                          z_loss=z_loss)
        ctx.save_for_backward(X, W, labels, lse, nv, err)
        ctx.cfg = (ignore_index, smoothing, reduction, z_loss)
        return loss[0]

    @staticmethod
    def backward(ctx, g):
        X, W, labels, lse, nv, err = ctx.saved_tensors
        ii, eps, red, zl = ctx.cfg
        g1 = g.reshape(1).to(torch.float32).contiguous()
        dX, dW, _ = flce_backward(X, W, labels, lse, nv, ii, eps, red, grad_loss=g1, err_word=err,
                                  z_loss=zl)
        return dX, dW.to(W.dtype), None, None, None, None, None


def linear_cross_entropy(h, W, labels, ignore_index: int = -100, smoothing: float = 0.0,
                         reduction: str = "mean", z_loss: float = 0.0):
    """Autograd entry with the pages' call shape: linear_cross_entropy(h, W, labels,
    ignore_index=-100).  h may be [..., H]; labels [...] of the same leading shape."""
    H = h.shape[-1]
    return _LinearCrossEntropy.apply(h.reshape(-1, H).contiguous(), W.contiguous(),
                                     labels.reshape(-1).contiguous(), ignore_index, smoothing,
                                     reduction, z_loss)
