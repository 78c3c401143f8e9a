"""Parity of the token-scan prefill (gdn_prefill, algo='scan') with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import gdn_prefill, gdn_stream_status, inputs
from tests.util import rel_l2, to_np, tol_for

pytestmark = pytest.mark.gpu


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run(d, algo="scan", scale=1.0, state_in=True):
    x = dev(d)
    s_in = x["state_in"] if state_in else None
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=s_in, scale=scale, algo=algo)
    assert gdn_stream_status() == "GDN_OK"
    return o, st


def oracle_full(d, scale=1.0):
    return oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["h_k"],
                          d["h_v"], d["d_k"], d["d_v"], state_in=d["state_in"], scale=scale)


def check(d, o, st, scale=1.0):
    o_ref, s_ref = oracle_full(d, scale)
    T = d["q"].shape[0]
    tol = tol_for(d["dtype"])
    if T:
        assert rel_l2(to_np(o), o_ref) < tol
    assert rel_l2(to_np(st), s_ref) < tol
    return o_ref, s_ref


def test_tiny_f32_workload():
    """One sequence of 64 tokens, one head of dimension 16, fp32, zero state."""
    w = inputs.WORKLOADS["prefill_t64_d16_f32"]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"])
    o, st = run(d)
    o_ref, s_ref = oracle_full(d)
    assert rel_l2(to_np(o), o_ref) < 1e-5 and rel_l2(to_np(st), s_ref) < 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lengths", [[1], [63], [64], [65], [127], [129], [0, 5], [3, 0, 70, 1]])
def test_lengths(dtype, lengths):
    d = inputs.make_prefill(lengths, 2, 4, 32, 64, dtype, seed=sum(lengths) + 1, state_std=0.1)
    o, st = run(d, scale=0.9)
    check(d, o, st, scale=0.9)


@pytest.mark.parametrize("d_k,d_v", [(16, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("h_k,h_v", [(1, 1), (2, 4), (2, 2)])
def test_shapes(d_k, d_v, h_k, h_v):
    d = inputs.make_prefill([37, 90], h_k, h_v, d_k, d_v, "bf16", seed=d_k + d_v + h_v,
                            state_std=0.02)
    o, st = run(d)
    check(d, o, st)


def test_null_state_in_is_zero():
    d = inputs.make_prefill([50], 1, 2, 32, 32, "f32", seed=2)
    o, st = run(d, state_in=False)
    check(d, o, st)


def test_state_aliasing_in_place():
    d = inputs.make_prefill([20, 44], 1, 2, 64, 64, "f32", seed=3, state_std=0.1)
    x = dev(d)
    st = x["state_in"].clone()
    o, st2 = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                         state_in=st, state_out=st, algo="scan")
    assert st2.data_ptr() == st.data_ptr()
    check(d, o, st)


def test_varlen_bitwise_equals_single_sequence():
    lengths = [5, 64, 0, 130, 1]
    d = inputs.make_prefill(lengths, 2, 4, 64, 64, "bf16", seed=4, state_std=0.05)
    o, st = run(d)
    cu = d["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        sub = dict(d, q=d["q"][a:b], k=d["k"][a:b], v=d["v"][a:b], g=d["g"][a:b],
                   beta=d["beta"][a:b], state_in=d["state_in"][n:n + 1],
                   cu_seqlens=torch.tensor([0, b - a], dtype=torch.int32))
        o1, s1 = run(sub)
        assert torch.equal(o1, o[a:b]) and torch.equal(s1[0], st[n])


def test_empty_sequence_copies_state_and_writes_nothing():
    d = inputs.make_prefill([0, 4], 1, 1, 16, 16, "f32", seed=5, state_std=0.3)
    x = dev(d)
    o = torch.full((4, 1, 16), 7.0, device="cuda")
    _, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], o=o, algo="scan")
    assert torch.equal(st[0], x["state_in"][0])


def test_bad_cu_seqlens_reported_and_nothing_written():
    d = inputs.make_prefill([10, 10], 1, 1, 16, 16, "f32", seed=6)
    x = dev(d)
    cu = torch.tensor([0, 12, 10], dtype=torch.int32, device="cuda")  # decreasing
    o = torch.full((20, 1, 16), 3.0, device="cuda")
    st = torch.full((2, 1, 16, 16), 5.0, device="cuda")
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, state_out=st, o=o, algo="scan")
    assert gdn_stream_status() == "GDN_ERR_BAD_CU_SEQLENS"
    assert gdn_stream_status() == "GDN_OK"  # cleared by the read
    # sequence 1 is invalid and untouched; sequence 0 ([0, 12)) is valid and computed
    assert torch.all(st[1] == 5.0)
    cu = torch.tensor([0, 10, 25], dtype=torch.int32, device="cuda")  # cu[N] != T
    st.fill_(5.0)
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, state_out=st, o=o, algo="scan")
    assert gdn_stream_status() == "GDN_ERR_BAD_CU_SEQLENS"
    assert torch.all(st[1] == 5.0)


def test_split_prefill_equals_one_shot():
    d = inputs.make_prefill([300], 2, 4, 64, 64, "bf16", seed=7, state_std=0.02)
    o, st = run(d)
    x = dev(d)
    T1 = 113
    o1, s1 = gdn_prefill(x["q"][:T1], x["k"][:T1], x["v"][:T1], x["g"][:T1], x["beta"][:T1],
                         torch.tensor([0, T1], dtype=torch.int32, device="cuda"),
                         state_in=x["state_in"], algo="scan")
    o2, s2 = gdn_prefill(x["q"][T1:], x["k"][T1:], x["v"][T1:], x["g"][T1:], x["beta"][T1:],
                         torch.tensor([0, 300 - T1], dtype=torch.int32, device="cuda"),
                         state_in=s1, algo="scan")
    assert torch.equal(torch.cat([o1, o2]), o) and torch.equal(s2, st)


def test_prefill_t4096_full_heads_scan():
    """The 4096-token prompt, 16 key / 32 value heads of 128, bf16: the scan
    path against the full oracle."""
    w = inputs.WORKLOADS["prefill_t4096"]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"])
    o, st = run(d)
    o_ref, s_ref = check(d, o, st)
    assert rel_l2(to_np(o), o_ref) < 5e-3
