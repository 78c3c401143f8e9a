"""Grouped-query decode attention on the GPU against the fp64 oracle.

Inputs: N(0, 1) bf16 queries and caches, the cache slots past every
sequence's length filled with NaN (they must never reach a result); shapes of
the pages' attention layers (head dimension 256, 16 query heads on 2 KV
heads), ragged lengths that end inside a tile, empty sequences, and both
layouts.

Tolerance, from the arithmetic: scores are exact bf16 products summed in
fp32; the softmax weights are rounded to bf16 (relative 2^-9 each) before
the weighted sum of V rows while the normaliser sums the unrounded weights,
and o is stored in bf16 (2^-9 |o|).  With A = sum_i w_i |v_i| (the oracle's
attention over |v|, which bounds |o|): |o - o_ref| <= 2^-9 A + 2^-9 |o| +
2^-9 |o| <= 2^-8 (A + |o_ref|), plus 1e-4 for the fp32 sums.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import gdn_attn_decode, gdn_stream_status
from gated_deltanet_linear_recurrence_gb300.inputs import make_attention
from oracle.attention import gqa_decode

pytestmark = pytest.mark.gpu
REL, ABS = 2.0 ** -8, 1e-4


def run_case(batch, h_q, h_kv, capacity, lengths, layout, block_keys=0, seed=0):
    x = make_attention(batch, h_q, h_kv, 256, capacity, lengths, seed=seed)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    scale = 256 ** -0.5
    o = gdn_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"], dev["cache_len"], scale=scale,
                        layout=layout, block_keys=block_keys)
    assert gdn_stream_status() == "GDN_OK"
    ref = gqa_decode(x["q"], x["k_cache"], x["v_cache"], x["cache_len"], scale)
    wabs = gqa_decode(x["q"], x["k_cache"], x["v_cache"].abs(), x["cache_len"], scale)
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    check(got, ref, wabs)
    return got, ref


def check(got, ref, wabs):
    err = np.abs(got - ref)
    bound = REL * (wabs + np.abs(ref)) + ABS
    worst = np.unravel_index((err - bound).argmax(), err.shape)
    assert (err <= bound).all(), f"err {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}"


@pytest.mark.parametrize("layout,block_keys", [("general", 0), ("fixed_block", 64),
                                               ("fixed_block", 256), ("fixed_block", 0),
                                               ("auto", 0)])
def test_ragged_lengths(layout, block_keys):
    """Lengths that end inside a tile, a full cache, one key and an empty cache."""
    run_case(4, 16, 2, 1000, [1000, 333, 1, 0], layout, block_keys)


@pytest.mark.parametrize("h_q,h_kv", [(16, 2), (8, 8), (6, 2), (8, 1), (3, 3)])
def test_group_sizes(h_q, h_kv):
    """Query heads per KV head from 1 to 8 (the padded heads contribute nothing)."""
    run_case(2, h_q, h_kv, 700, [700, 450], "general", seed=1)
    run_case(2, h_q, h_kv, 700, [700, 450], "fixed_block", 128, seed=1)


def test_layouts_at_4k():
    """Both layouts at a 4,096-key cache, each within the bound of the oracle."""
    run_case(2, 16, 2, 4096, [4096, 2500], "general", seed=2)
    run_case(2, 16, 2, 4096, [4096, 2500], "fixed_block", 512, seed=2)


def test_all_empty():
    """Every sequence empty: o = 0 in both layouts."""
    got, _ = run_case(3, 16, 2, 256, [0, 0, 0], "general")
    assert (got == 0).all()
    got, _ = run_case(3, 16, 2, 256, [0, 0, 0], "fixed_block", 64)
    assert (got == 0).all()


def test_long_context_128k():
    """One sequence at the pages' longest context (131,072 keys), in the layout
    and launch the benchmark times (fixed blocks chosen by the library)."""
    run_case(1, 16, 2, 131072, [131072], "auto", seed=3)
    run_case(1, 16, 2, 131072, [131071], "fixed_block", 2048, seed=4)


def test_bad_cache_len_is_reported():
    """A length beyond the capacity is recorded in the error word and that
    sequence gets o = 0; the other sequences are unaffected."""
    x = make_attention(2, 16, 2, 256, 128, [128, 100], seed=5, poison_tail=False)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    lens = torch.tensor([129, 100], dtype=torch.int32, device="cuda")
    o = gdn_attn_decode(dev["q"], dev["k_cache"], dev["v_cache"], lens, layout="general")
    assert gdn_stream_status() == "GDN_ERR_BAD_CACHE_LEN"
    assert gdn_stream_status() == "GDN_OK"
    got = o.float().cpu().numpy()
    assert (got[0] == 0).all()
    ref = gqa_decode(x["q"], x["k_cache"], x["v_cache"], [0, 100], 256 ** -0.5)
    wabs = gqa_decode(x["q"], x["k_cache"], x["v_cache"].abs(), [0, 100], 256 ** -0.5)
    check(got[1:], ref[1:], wabs[1:])
