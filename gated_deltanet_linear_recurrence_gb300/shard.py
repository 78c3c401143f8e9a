"""Partition of the layer's work across ranks (one process per GPU).

The recurrence is independent per (sequence, value head): each value head
keeps its own state and reads key head h // (h_v // h_k).  Ranks therefore
split the work along value heads in whole key-head groups, so that no key
head is read by two ranks, or along sequences.  Neither split needs any
exchange between ranks: there is no collective on the data path.
(Splitting one sequence along its tokens would need a scan of state
transitions across ranks; it is not offered.)

Host-side index arithmetic only; the shards run through the same C ABI calls
as the whole problem.
"""

__all__ = ["head_shard", "seq_shard", "slice_heads", "slice_seqs"]


def head_shard(h_k, h_v, rank, world):
    """Key heads [kh0, kh1) and value heads [vh0, vh1) owned by `rank`.

    Key heads are dealt out in contiguous, near-equal blocks (the first
    h_k % world ranks get one more); a rank owns every value head that reads
    one of its key heads.  Ranks beyond h_k get empty ranges.
    """
    if not (0 <= rank < world) or h_k <= 0 or h_v % h_k:
        raise ValueError("bad rank/world or head counts")
    base, extra = divmod(h_k, world)
    kh0 = rank * base + min(rank, extra)
    kh1 = kh0 + base + (1 if rank < extra else 0)
    g = h_v // h_k
    return kh0, kh1, kh0 * g, kh1 * g


def seq_shard(cu_seqlens, rank, world):
    """Sequences [n0, n1) owned by `rank`: contiguous ranges whose token counts
    are balanced; rank r's range starts at the first sequence that begins at or
    after token r * T / world.
    """
    cu = [int(c) for c in cu_seqlens]
    N, T = len(cu) - 1, cu[-1]
    if not (0 <= rank < world) or N < 0:
        raise ValueError("bad rank/world or cu_seqlens")

    def start(r):
        if r >= world:
            return N
        target = r * T / world
        n = 0
        while n < N and cu[n] < target:
            n += 1
        return n

    return start(rank), start(rank + 1)


def slice_heads(d, kh0, kh1, vh0, vh1):
    """Inputs of a head shard (contiguous copies): q, k on key heads [kh0, kh1);
    v, g, beta and state_in on value heads [vh0, vh1)."""
    out = dict(d)
    for key in ("q", "k"):
        out[key] = d[key][:, kh0:kh1].contiguous()
    for key in ("v", "g", "beta"):
        out[key] = d[key][:, vh0:vh1].contiguous()
    if d.get("state_in") is not None:
        out["state_in"] = d["state_in"][:, vh0:vh1].contiguous()
    out["h_k"], out["h_v"] = kh1 - kh0, vh1 - vh0
    return out


def slice_seqs(d, n0, n1):
    """Inputs of a sequence shard: the tokens of sequences [n0, n1) and their
    initial states, with cu_seqlens rebased to start at 0."""
    cu = d["cu_seqlens"]
    t0, t1 = int(cu[n0]), int(cu[n1])
    out = dict(d)
    for key in ("q", "k", "v", "g", "beta"):
        out[key] = d[key][t0:t1].contiguous()
    out["cu_seqlens"] = (cu[n0:n1 + 1] - t0).contiguous()
    if d.get("state_in") is not None:
        out["state_in"] = d["state_in"][n0:n1].contiguous()
    return out
