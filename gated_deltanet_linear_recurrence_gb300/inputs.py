"""Seeded synthetic inputs for the Gated DeltaNet recurrence.

This module only draws random numbers; it holds none of the recurrence's
arithmetic.  The same tensors feed the CUDA library and the CPU oracle.

Recipe (one value per token and head, drawn on the host in fp64 from a seeded
``torch.Generator`` and then rounded to nearest-even in the storage dtype):

* q, k ~ N(0, 1), then scaled to unit L2 norm per (token, key head);
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1)) and g = -softplus(N(0, 1)), kept fp32;
* initial state zeros, or N(0, std^2) fp32 (std = 0.02 where a workload asks
  for a drawn state).

Workload shapes follow the page "Optimizing on-device inference for Apple
Silicon": prompt and context lengths from 256 to 128K tokens, batch-1 decode,
30 Gated DeltaNet layers, 16 key heads and 32 value heads of dimension 128.
Large tensors are drawn in token blocks so peak host memory stays bounded.
"""
import torch

_BLOCK_TOKENS = 8192

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _unit_rows(x):
    """Scale each trailing-dimension vector to unit L2 norm (input preparation)."""
    return x / x.norm(dim=-1, keepdim=True)


def _draw_qk(gen, tokens, heads, dim, dtype, unit=True):
    out = torch.empty((tokens, heads, dim), dtype=dtype)
    for t0 in range(0, tokens, _BLOCK_TOKENS):
        t1 = min(tokens, t0 + _BLOCK_TOKENS)
        blk = torch.randn((t1 - t0, heads, dim), generator=gen, dtype=torch.float64)
        out[t0:t1] = (_unit_rows(blk) if unit else blk).to(dtype)
    return out


def _draw_normal(gen, shape, dtype, std=1.0):
    out = torch.empty(shape, dtype=dtype)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    for t0 in range(0, shape[0], _BLOCK_TOKENS):
        t1 = min(shape[0], t0 + _BLOCK_TOKENS)
        blk = torch.randn((t1 - t0, flat.shape[1]), generator=gen, dtype=torch.float64)
        flat[t0:t1] = (blk * std).to(dtype)
    return out


def _draw_gates(gen, tokens, heads):
    beta = torch.sigmoid(torch.randn((tokens, heads), generator=gen, dtype=torch.float64))
    g = -torch.nn.functional.softplus(
        torch.randn((tokens, heads), generator=gen, dtype=torch.float64))
    return g.to(torch.float32), beta.to(torch.float32)


def cu_from_lengths(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def make_prefill(lengths, h_k, h_v, d_k, d_v, dtype="bf16", seed=0, state_std=0.0,
                 unit_qk=True):
    """Packed varlen prefill inputs on the host.

    Returns a dict with q, k [T, h_k, d_k]; v [T, h_v, d_v] (dtype); g, beta
    [T, h_v] fp32; state_in [N, h_v, d_v, d_k] fp32 or None (zeros);
    cu_seqlens [N+1] int32.  ``unit_qk=False`` leaves q and k as drawn, N(0, 1)
    (inputs for the in-kernel normalisation option).
    """
    dt = DTYPES[dtype]
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    gen = _gen(seed)
    q = _draw_qk(gen, T, h_k, d_k, dt, unit_qk)
    k = _draw_qk(gen, T, h_k, d_k, dt, unit_qk)
    v = _draw_normal(gen, (T, h_v, d_v), dt)
    g, beta = _draw_gates(gen, T, h_v)
    state = None
    if state_std > 0:
        n = len(lengths)
        state = _draw_normal(gen, (max(n, 1), h_v, d_v, d_k), torch.float32, state_std)[:n]
    return dict(q=q, k=k, v=v, g=g, beta=beta, state_in=state, cu_seqlens=cu,
                h_k=h_k, h_v=h_v, d_k=d_k, d_v=d_v, dtype=dtype)


def make_decode(batch, h_k, h_v, d_k, d_v, dtype="bf16", seed=0, state_std=0.02):
    """One-token-per-sequence decode inputs: q, k [B, h_k, d_k], v [B, h_v, d_v],
    g, beta [B, h_v] fp32, state [B, h_v, d_v, d_k] fp32."""
    dt = DTYPES[dtype]
    gen = _gen(seed)
    q = _draw_qk(gen, batch, h_k, d_k, dt)
    k = _draw_qk(gen, batch, h_k, d_k, dt)
    v = _draw_normal(gen, (batch, h_v, d_v), dt)
    g, beta = _draw_gates(gen, batch, h_v)
    if state_std > 0:
        state = _draw_normal(gen, (batch, h_v, d_v, d_k), torch.float32, state_std)
    else:
        state = torch.zeros((batch, h_v, d_v, d_k), dtype=torch.float32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, state=state,
                h_k=h_k, h_v=h_v, d_k=d_k, d_v=d_v, dtype=dtype)


# The workloads, each named by what it is.  Seeds are 20261202 + index.
SEED_BASE = 20261202
WORKLOADS = {
    # tiny fp32 prefill: one sequence of 64 tokens, one head of dimension 16
    "prefill_t64_d16_f32": dict(kind="prefill", lengths=[64], h_k=1, h_v=1, d_k=16, d_v=16,
                                dtype="f32", state_std=0.0, seed=SEED_BASE + 0),
    # batch-1 decode through 30 layers, 16 key / 32 value heads of dimension 128
    "decode_b1_x30layers": dict(kind="decode", batch=1, layers=30, h_k=16, h_v=32, d_k=128,
                                d_v=128, dtype="bf16", state_std=0.02, seed=SEED_BASE + 1),
    # prefill of one 4096-token prompt
    "prefill_t4096": dict(kind="prefill", lengths=[4096], h_k=16, h_v=32, d_k=128, d_v=128,
                          dtype="bf16", state_std=0.0, seed=SEED_BASE + 2),
    # prefill of one 128K-token prompt with a drawn initial state
    "prefill_t131072": dict(kind="prefill", lengths=[131072], h_k=16, h_v=32, d_k=128,
                            d_v=128, dtype="bf16", state_std=0.02, seed=SEED_BASE + 3),
    # batched decode of 256 independent sequences
    "decode_b256": dict(kind="decode", batch=256, layers=1, h_k=16, h_v=32, d_k=128, d_v=128,
                        dtype="bf16", state_std=0.02, seed=SEED_BASE + 4),
    # packed varlen prefill of ten prompts, 256 ... 128K tokens
    "prefill_varlen10": dict(kind="prefill", lengths=[256 << m for m in range(10)], h_k=16,
                             h_v=32, d_k=128, d_v=128, dtype="bf16", state_std=0.0,
                             seed=SEED_BASE + 5),
    # decode attention of the hybrid model's full-attention layers (16 query heads on
    # 2 KV heads of 256): one sequence's new token over a 128K-key cache
    "attn_b1_l131072": dict(kind="attention", batch=1, h_q=16, h_kv=2, head_dim=256,
                            capacity=131072, lengths=[131072], dtype="bf16",
                            seed=SEED_BASE + 6),
    # the same layer for 64 sequences of 8K cached keys each
    "attn_b64_l8192": dict(kind="attention", batch=64, h_q=16, h_kv=2, head_dim=256,
                           capacity=8192, lengths=[8192] * 64, dtype="bf16",
                           seed=SEED_BASE + 7),
}


def make_attention(batch, h_q, h_kv, head_dim, capacity, lengths, dtype="bf16", seed=0,
                   poison_tail=True):
    """Decode-attention inputs on the host: q [B, h_q, D]; k_cache, v_cache
    [B, h_kv, capacity, D]; cache_len [B] int32; all N(0, 1) in `dtype`.
    ``poison_tail`` fills the cache slots past each sequence's length with NaN
    (they must never reach a result).  Drawn in blocks of cache rows."""
    dt = DTYPES[dtype]
    gen = _gen(seed)
    q = _draw_normal(gen, (batch, h_q, head_dim), dt)
    k = torch.empty((batch, h_kv, capacity, head_dim), dtype=dt)
    v = torch.empty((batch, h_kv, capacity, head_dim), dtype=dt)
    for b in range(batch):
        for j in range(h_kv):
            k[b, j] = _draw_normal(gen, (capacity, head_dim), dt)
            v[b, j] = _draw_normal(gen, (capacity, head_dim), dt)
    lens = torch.tensor([int(x) for x in lengths], dtype=torch.int32)
    if poison_tail:
        for b in range(batch):
            k[b, :, int(lens[b]):] = float("nan")
            v[b, :, int(lens[b]):] = float("nan")
    return dict(q=q, k_cache=k, v_cache=v, cache_len=lens, h_q=h_q, h_kv=h_kv,
                head_dim=head_dim, capacity=capacity, dtype=dtype)
