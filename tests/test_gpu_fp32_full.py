"""fp32 variants of the full-size workloads against the fp64 oracle, at the
contract's 1e-4 relative L2 bar for fp32 inputs.

The workloads keep their shapes, distributions and seeds (16 key / 32 value
heads of 128; the 4096-token prompt, the 128K-token prompt with a drawn state,
the ten packed prompts of 256 ... 128K tokens, and the 256-sequence decode
step); only q, k, v (and o) are fp32.  The library's own choice runs (the token
scan: the chunked forms take bf16 operands), and the tests check that it is
that choice.  The 4096-token prompt and the decode step are compared in full;
the long workloads on sampled value rows (every output of a row and its final
state row: a state row evolves on its own, so the oracle computes rows one by
one)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_step, gdn_prefill,
                                                    gdn_prefill_form, gdn_stream_status, inputs)
from tests.util import TOL_F32, rel_l2, sample_tasks, sampled_errors, to_np

pytestmark = pytest.mark.gpu


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def workload_f32(name):
    w = inputs.WORKLOADS[name]
    return w, inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], "f32",
                                  seed=w["seed"], state_std=w["state_std"])


def run_auto(d):
    x = dev(d)
    T, N = x["q"].shape[0], x["cu_seqlens"].numel() - 1
    form = gdn_prefill_form(N, T, d["h_k"], d["h_v"], d["d_k"], d["d_v"], torch.float32, "auto")
    assert form == "scan"
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], algo="auto")
    assert gdn_stream_status() == "GDN_OK"
    assert o.dtype == torch.float32
    return o, st


def test_f32_prefill_t4096_full_oracle():
    _, d = workload_f32("prefill_t4096")
    o, st = run_auto(d)
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                  d["h_k"], d["h_v"], d["d_k"], d["d_v"], state_in=None)
    eo, es = rel_l2(to_np(o), o_ref), rel_l2(to_np(st), s_ref)
    assert eo < TOL_F32 and es < TOL_F32, (eo, es)


def test_f32_prefill_t131072_carried_state_sampled():
    _, d = workload_f32("prefill_t131072")
    o, st = run_auto(d)
    eo, es = sampled_errors(d, o, st, sample_tasks(1, 32, 128, 32, seed=11))
    assert eo < TOL_F32 and es < TOL_F32, (eo, es)


def test_f32_varlen_ten_sequences_sampled():
    _, d = workload_f32("prefill_varlen10")
    o, st = run_auto(d)
    eo, es = sampled_errors(d, o, st, sample_tasks(10, 32, 128, 4, seed=12))
    assert eo < TOL_F32 and es < TOL_F32, (eo, es)


def test_f32_decode_b256_full_oracle():
    w = inputs.WORKLOADS["decode_b256"]
    d = inputs.make_decode(w["batch"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], dtype="f32",
                           seed=w["seed"], state_std=w["state_std"])
    x = dev(d)
    state = x["state"].clone()
    o = gdn_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state)
    assert gdn_stream_status() == "GDN_OK"
    cu = np.arange(w["batch"] + 1, dtype=np.int32)
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, d["h_k"],
                                  d["h_v"], d["d_k"], d["d_v"], state_in=d["state"])
    eo, es = rel_l2(to_np(o), o_ref), rel_l2(to_np(state), s_ref)
    assert eo < TOL_F32 and es < 1e-5, (eo, es)
