"""fp64 CPU oracle for the Gated DeltaNet recurrence — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, token by token; see
its header for the definition and the citations).  This module only marshals
arguments through ctypes.  Inputs may be torch CPU tensors or numpy arrays in
bf16 / fp32 / fp64; they are passed in their storage type and widened exactly
inside the oracle.
"""
import ctypes

import numpy as np

from .build import build_oracle

F64, F32, BF16 = 0, 1, 2
_ERRORS = {1: "invalid argument", 2: "invalid cu_seqlens", 3: "out of memory",
           4: "thread creation failed"}
_libs = {}


def _lib(mutant=0):
    if mutant not in _libs:
        lib = ctypes.CDLL(build_oracle(mutant))
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.gdn_oracle_prefill.restype = ctypes.c_int
        lib.gdn_oracle_prefill.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                           vp, i32, i64, i32, i32, i32, i32, dbl, ctypes.c_int,
                                           vp, vp, i32]
        lib.gdn_oracle_rows.restype = ctypes.c_int
        lib.gdn_oracle_rows.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                        vp, i32, i64, i32, i32, i32, i32, dbl, ctypes.c_int,
                                        vp, i64, vp, vp, vp, i32]
        lib.gdn_oracle_default_threads.restype = ctypes.c_int
        _libs[mutant] = lib
    return _libs[mutant]


def default_threads():
    """Threads a call with threads=0 uses (all online cores)."""
    return int(_lib().gdn_oracle_default_threads())


def _as_np(x):
    """Return (contiguous numpy array in storage type, dtype code)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:  # raw bf16 bits
        return x, BF16
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _prep(q, k, v, g, beta, state_in, cu_seqlens):
    qa, qd = _as_np(q)
    ka, kd = _as_np(k)
    va, vd = _as_np(v)
    if not (qd == kd == vd):
        raise TypeError("q, k and v must share one dtype")
    ga, gd = _as_np(g)
    ba, bd = _as_np(beta)
    if gd != bd or gd == BF16:
        raise TypeError("g and beta must both be fp32 or both fp64")
    sa = None
    if state_in is not None:
        sa, sd = _as_np(state_in)
        if sd != gd:
            sa = sa.astype(np.float64 if gd == F64 else np.float32)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens), dtype=np.int32)
    return qa, ka, va, ga, ba, sa, cu, qd, gd


def prefill(q, k, v, g, beta, cu_seqlens, h_k, h_v, d_k, d_v, state_in=None, scale=1.0,
            threads=0, mutant=0, qk_l2norm=False):
    """Full evaluation.  Returns (o [T, h_v, d_v] fp64, state [N, h_v, d_v, d_k] fp64).

    Output rows of tokens that belong to no sequence stay NaN.  ``qk_l2norm``
    divides q and k of every (token, key head) by sqrt(|x|^2 + 1e-6) first.
    """
    qa, ka, va, ga, ba, sa, cu, qd, gd = _prep(q, k, v, g, beta, state_in, cu_seqlens)
    n = len(cu) - 1
    t = int(cu[-1]) if n >= 0 else 0
    total = qa.size // (h_k * d_k) if qa.size else 0
    o = np.full((total, h_v, d_v), np.nan)
    st = np.zeros((n, h_v, d_v, d_k))
    rc = _lib(mutant).gdn_oracle_prefill(qd, gd, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ga),
                                         _ptr(ba), _ptr(sa), _ptr(cu), n, total, h_k, h_v,
                                         d_k, d_v, float(scale), int(bool(qk_l2norm)), _ptr(o),
                                         _ptr(st), threads)
    if rc:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")
    del t
    return o, st


def rows(q, k, v, g, beta, cu_seqlens, h_k, h_v, d_k, d_v, tasks, state_in=None, scale=1.0,
         threads=0, mutant=0, qk_l2norm=False):
    """Sampled evaluation of value rows.

    ``tasks`` is a sequence of (seq, value_head, row).  Returns a list with, per
    task, (o [L_seq] fp64 — o[t, h, row] for the sequence's tokens in order,
    final state row [d_k] fp64).
    """
    qa, ka, va, ga, ba, sa, cu, qd, gd = _prep(q, k, v, g, beta, state_in, cu_seqlens)
    n = len(cu) - 1
    total = qa.size // (h_k * d_k) if qa.size else 0
    tk = np.ascontiguousarray(np.asarray(tasks, dtype=np.int64).reshape(-1, 3))
    lens = (cu[1:] - cu[:-1]).astype(np.int64)
    if len(tk) and (tk[:, 0].min() < 0 or tk[:, 0].max() >= n):
        raise ValueError("oracle: task sequence index out of range")
    per = lens[tk[:, 0]] if len(tk) else np.zeros(0, np.int64)
    off = np.ascontiguousarray(np.concatenate([[0], np.cumsum(per)[:-1]]).astype(np.int64)
                               if len(tk) else np.zeros(0, np.int64))
    o = np.zeros(max(int(per.sum()), 1))
    st = np.zeros((max(len(tk), 1), d_k))
    rc = _lib(mutant).gdn_oracle_rows(qd, gd, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba),
                                      _ptr(sa), _ptr(cu), n, total, h_k, h_v, d_k, d_v,
                                      float(scale), int(bool(qk_l2norm)), _ptr(tk), len(tk),
                                      _ptr(off), _ptr(o),
                                      _ptr(st), threads)
    if rc:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")
    return [(o[off[j]:off[j] + per[j]].copy(), st[j].copy()) for j in range(len(tk))]
