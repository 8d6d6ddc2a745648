"""Helpers shared by the GPU tests: device copies of seeded workloads and the
comparison metrics with the tolerances the parity bar states."""
import numpy as np

# Parity bar: loss relative error, lse absolute error, relative Frobenius
# error of dX and dW, all against the fp64 oracle on the same input bits.
LOSS_REL = 2e-3
LSE_ABS = 1e-2
GRAD_REL_FRO = 1e-2


def to_device(wl, device="cuda"):
    import torch
    if wl.dtype == "bf16":
        X = torch.from_numpy(np.ascontiguousarray(wl.x).view(np.int16)).view(torch.bfloat16)
        W = torch.from_numpy(np.ascontiguousarray(wl.w).view(np.int16)).view(torch.bfloat16)
    else:
        X = torch.from_numpy(np.ascontiguousarray(wl.x))
        W = torch.from_numpy(np.ascontiguousarray(wl.w))
    labels = torch.from_numpy(np.ascontiguousarray(wl.labels))
    return X.to(device), W.to(device), labels.to(device)


def tensor_f64(t):
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def rel_fro(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    if den == 0.0:
        return num
    return num / den


def rel_err(got, want):
    got, want = float(got), float(want)
    if want == 0.0:
        return abs(got)
    return abs(got - want) / abs(want)
