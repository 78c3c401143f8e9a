"""Shared helpers for the parity tests: error metrics and device plumbing.

The comparison metric is the relative L2 error in fp64 over a whole tensor,
||x - x_ref|| / ||x_ref||, taken separately for o and for the final state.
Tolerances are the stated contract: 1e-4 when q/k/v are fp32, 2e-2 when they
are bf16 (tensor-core path); integer indexing and varlen offsets bit-exact.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def tol_for(dtype):
    return TOL_F32 if dtype in ("f32", torch.float32) else TOL_BF16


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 \
        else t.detach().cpu().numpy().astype(np.float64)


def to_dev(d, device="cuda"):
    out = {}
    for key, val in d.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out


def worst_slice(x, ref, axis_names=("t", "h", "i")):
    """Relative L2 per value head for o [T, h, i]: returns (worst head, its error)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    errs = [rel_l2(x[:, h], ref[:, h]) for h in range(ref.shape[1])]
    h = int(np.argmax(errs))
    return h, errs[h]
