"""fp64 CPU oracle for the output RMS normalisation — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the CUDA library never calls it.

What it computes.  The page "Optimizing on-device inference for Apple
Silicon" (section "Reduce intermediate and state traffic") fuses the decode
step's recurrent update "with its normalization" without giving the form of
the normalisation.  Besides the q/k normalisation (GDN_OPT_QK_L2NORM), the
plainest reading of a normalisation of the layer's output is a root-mean-square
normalisation of each (token, value head)'s d_v output values, with a learned
per-channel weight w shared by the heads:

    o'_i = w_i * o_i / sqrt( (1 / d_v) * sum_j o_j^2 + eps )

written out here in fp64 on the exact input values (o widened from its
storage type; w and eps as given).  ``weight=None`` means w_i = 1.
"""
import numpy as np


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def output_rmsnorm(o, weight=None, eps=1e-6):
    """o [..., h_v, d_v] (any leading shape); weight [d_v] or None.  Returns the
    normalised values in fp64, same shape as o."""
    x = _f64(o)
    d_v = x.shape[-1]
    w = np.ones(d_v) if weight is None else _f64(weight).reshape(d_v)
    ms = (x * x).sum(axis=-1, keepdims=True) / d_v
    return x / np.sqrt(ms + float(eps)) * w
