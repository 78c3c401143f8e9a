"""fp64 CPU oracle for grouped-query decode attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the CUDA library never calls it.

What it computes.  The page "Optimizing on-device inference for Apple
Silicon" (section "Read the attention cache efficiently") describes the decode
step of a full-attention layer: the new token's query heads read the keys and
values cached for every earlier token, eight query heads share one key/value
head ("Group query heads to reuse KV rows"), and at long context the cache is
split into equal fixed blocks processed in parallel ("Switch attention layouts
at long context", for heads of 256 values with eight query heads per KV head).
Every layout computes the same attention; this is its definition, per sequence
b and query head h (KV head j = h // (h_q / h_kv)), over the L_b cached keys:

    s_i = scale * (q_h . k_{b,j,i})          i = 0 .. L_b - 1
    o_h = sum_i softmax(s)_i v_{b,j,i}

written out in fp64 with the usual max subtraction inside the softmax (which
leaves its value unchanged).  Inputs are widened exactly from their storage
type (bf16 arrives as torch bfloat16, fp32 / fp64 as numpy or torch).
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


def gqa_decode(q, k_cache, v_cache, cache_len, scale):
    """q [B, h_q, D]; k_cache, v_cache [B, h_kv, capacity, D]; cache_len [B].
    Returns o [B, h_q, D] fp64.  A sequence with L_b = 0 gets o = 0."""
    q, k, v = _f64(q), _f64(k_cache), _f64(v_cache)
    lens = [int(x) for x in (cache_len.tolist() if hasattr(cache_len, "tolist") else cache_len)]
    B, h_q, D = q.shape
    h_kv = k.shape[1]
    G = h_q // h_kv
    o = np.zeros((B, h_q, D))
    for b in range(B):
        L = lens[b]
        if L == 0:
            continue
        for h in range(h_q):
            j = h // G
            s = scale * (k[b, j, :L] @ q[b, h])
            w = np.exp(s - s.max())
            o[b, h] = (w / w.sum()) @ v[b, j, :L]
    return o
