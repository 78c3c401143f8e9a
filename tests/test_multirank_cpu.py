"""The multi-rank path on CPU: two gloo ranks (world size 2) split the layer by
key-head groups and by sequences, each runs the fp64 oracle on its shard, and
the shards gathered on rank 0 equal the unsharded run bit for bit; the bench's
max-over-ranks timing reduction is checked with gloo too.  The collective
here only gathers results for the check: the sharded work itself exchanges
nothing."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gated_deltanet_linear_recurrence_gb300 import inputs
from gated_deltanet_linear_recurrence_gb300.shard import (head_shard, seq_shard, slice_heads,
                                                          slice_seqs)

LENGTHS = [70, 5, 0, 130, 33]
H_K, H_V, D_K, D_V = 3, 6, 16, 8


def _make():
    return inputs.make_prefill(LENGTHS, H_K, H_V, D_K, D_V, "f32", seed=41, state_std=0.1)


def _run_oracle(d):
    return oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["h_k"],
                          d["h_v"], d["d_k"], d["d_v"], state_in=d["state_in"], scale=0.8)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = _make()
        kh0, kh1, vh0, vh1 = head_shard(H_K, H_V, rank, world)
        o_h, s_h = _run_oracle(slice_heads(d, kh0, kh1, vh0, vh1))
        n0, n1 = seq_shard(d["cu_seqlens"], rank, world)
        o_s, s_s = _run_oracle(slice_seqs(d, n0, n1))
        heads = [None] * world
        seqs = [None] * world
        dist.all_gather_object(heads, (vh0, vh1, o_h, s_h))
        dist.all_gather_object(seqs, (n0, n1, o_s, s_s))
        import bench
        worst = bench.max_over_ranks(10.0 + rank, torch.device("cpu"))
        assert worst == 10.0 + world - 1
        if rank == 0:
            o_ref, s_ref = _run_oracle(d)
            o_cat = np.concatenate([h[2] for h in heads], axis=1)
            s_cat = np.concatenate([h[3] for h in heads], axis=1)
            assert [h[:2] for h in heads] == [(0, 4), (4, 6)]
            assert np.array_equal(o_cat, o_ref) and np.array_equal(s_cat, s_ref)
            cu = d["cu_seqlens"].tolist()
            assert seqs[0][0] == 0 and seqs[-1][1] == len(LENGTHS)
            for (a0, a1, _, _), (b0, _, _, _) in zip(seqs, seqs[1:]):
                assert a1 == b0
            o_cat = np.concatenate([s[2] for s in seqs], axis=0)
            s_cat = np.concatenate([s[3] for s in seqs], axis=0)
            assert o_cat.shape[0] == cu[-1]
            assert np.array_equal(o_cat, o_ref) and np.array_equal(s_cat, s_ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shards_equal_unsharded():
    oracle.build_oracle()
    mp.start_processes(_rank_main, args=(2, _free_port()), nprocs=2, join=True,
                       start_method="spawn")


@pytest.mark.parametrize("h_k,h_v,world", [(16, 32, 1), (16, 32, 2), (16, 32, 8), (3, 6, 2),
                                           (2, 4, 4), (1, 1, 3)])
def test_head_shards_cover_key_head_groups(h_k, h_v, world):
    owner_k, owner_v = [None] * h_k, [None] * h_v
    for r in range(world):
        kh0, kh1, vh0, vh1 = head_shard(h_k, h_v, r, world)
        assert vh0 == kh0 * (h_v // h_k) and vh1 == kh1 * (h_v // h_k)
        for j in range(kh0, kh1):
            assert owner_k[j] is None
            owner_k[j] = r
        for h in range(vh0, vh1):
            assert owner_v[h] is None
            owner_v[h] = r
    assert None not in owner_k and None not in owner_v
    for h in range(h_v):  # each value head sits with the key head it reads
        assert owner_v[h] == owner_k[h // (h_v // h_k)]


@pytest.mark.parametrize("lengths,world", [([4096] * 8, 8), ([4096] * 2, 2), (LENGTHS, 2),
                                           ([1, 1, 1], 5), ([], 2), ([100, 0, 0, 7], 3)])
def test_seq_shards_are_contiguous_and_complete(lengths, world):
    cu = inputs.cu_from_lengths(lengths)
    spans = [seq_shard(cu, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == len(lengths)
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a0 <= a1 == b0 <= b1
    if lengths and len(set(lengths)) == 1 and len(lengths) == world:
        assert spans == [(r, r + 1) for r in range(world)]  # one prompt per rank
