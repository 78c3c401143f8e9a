"""The multi-GPU partition, exercised on one GPU: the shards of a head split
and of a sequence split, run one after another through the C ABI, reproduce
the unsharded call bit for bit (every kernel computes each (sequence, value
head) on its own, with no cross-head or cross-sequence reduction)."""
import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_step, gdn_prefill,
                                                    gdn_stream_status, inputs)
from gated_deltanet_linear_recurrence_gb300.shard import (head_shard, seq_shard, slice_heads,
                                                          slice_seqs)

pytestmark = pytest.mark.gpu


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run(d, algo):
    x = dev(d)
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], algo=algo)
    assert gdn_stream_status() == "GDN_OK"
    return o, st


# (Not "auto": it picks the fused or the two-kernel form from the average
# sequence length, which differs between a sequence shard and the whole.)
@pytest.mark.parametrize("algo", ["scan", "chunked_fused", "chunked_split"])
@pytest.mark.parametrize("world", [2, 4])
def test_head_and_sequence_shards_bitwise(algo, world):
    d = inputs.make_prefill([700, 3, 0, 130, 64], 4, 8, 128, 64, "bf16", seed=51,
                            state_std=0.05)
    o, st = run(d, algo)
    o_parts, st_parts = [], []
    for r in range(world):
        kh0, kh1, vh0, vh1 = head_shard(4, 8, r, world)
        o_r, st_r = run(slice_heads(d, kh0, kh1, vh0, vh1), algo)
        o_parts.append(o_r)
        st_parts.append(st_r)
    assert torch.equal(torch.cat(o_parts, dim=1), o) and torch.equal(torch.cat(st_parts, dim=1), st)
    o_parts, st_parts = [], []
    for r in range(world):
        n0, n1 = seq_shard(d["cu_seqlens"], r, world)
        if n1 == n0:
            continue
        o_r, st_r = run(slice_seqs(d, n0, n1), algo)
        o_parts.append(o_r)
        st_parts.append(st_r)
    assert torch.equal(torch.cat(o_parts), o) and torch.equal(torch.cat(st_parts), st)


def test_decode_batch_shards_bitwise():
    d = inputs.make_decode(6, 2, 4, 128, 128, "bf16", seed=52)
    x = dev(d)
    state = x["state"].clone()
    o = gdn_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state)
    outs, states = [], []
    for b0, b1 in ((0, 3), (3, 6)):
        s = x["state"][b0:b1].clone()
        outs.append(gdn_decode_step(x["q"][b0:b1], x["k"][b0:b1], x["v"][b0:b1],
                                    x["g"][b0:b1], x["beta"][b0:b1], s))
        states.append(s)
    assert torch.equal(torch.cat(outs), o) and torch.equal(torch.cat(states), state)
