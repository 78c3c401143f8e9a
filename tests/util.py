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


def sample_tasks(num_seqs, h_v, d_v, per_seq, seed):
    """(seq, head, row) triples: per_seq rows per sequence, spread over heads."""
    rng = np.random.default_rng(seed)
    tasks = []
    for n in range(num_seqs):
        hs = rng.choice(h_v, size=per_seq, replace=per_seq > h_v)
        rs = rng.choice(d_v, size=per_seq, replace=True)
        tasks += [(n, int(h), int(r)) for h, r in zip(hs, rs)]
    return tasks


def sampled_errors(d, o_gpu, st_gpu, tasks, scale=1.0):
    """Relative L2 of the sampled o rows and state rows against the oracle's
    row evaluation (each row of the state evolves independently)."""
    import oracle

    res = oracle.rows(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["h_k"],
                      d["h_v"], d["d_k"], d["d_v"], tasks, state_in=d["state_in"], scale=scale)
    cu = d["cu_seqlens"].tolist()
    o_ref, o_got, s_ref, s_got = [], [], [], []
    for (n, h, i), (ro, rs) in zip(tasks, res):
        o_ref.append(ro)
        o_got.append(to_np(o_gpu[cu[n]:cu[n + 1], h, i]))
        s_ref.append(rs)
        s_got.append(to_np(st_gpu[n, h, i]))
    return (rel_l2(np.concatenate(o_got), np.concatenate(o_ref)),
            rel_l2(np.stack(s_got), np.stack(s_ref)))
