"""fp64 CPU oracle (test infrastructure only; see flce_oracle.py)."""
from .flce_oracle import (  # noqa: F401
    IGNORE_INDEX, upcast, logits, row_logsumexp, valid_mask, grad_scale,
    row_losses, forward, dlogits, backward, forward_rows, dx_rows, dw_rows,
    fwd_bwd, ForwardResult, BackwardResult,
)
