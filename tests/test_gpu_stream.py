"""gdn_prefill_streamed: a sequence prefilled as fixed-size pieces with the state
carried between them equals, bit for bit, the whole-sequence call with the same
evaluation, and the oracle within the bf16 / fp32 tolerances."""
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill, gdn_prefill_streamed,
                                                    gdn_prefill_streamed_workspace_size,
                                                    gdn_stream_status, inputs)
from tests.util import rel_l2, sample_tasks, sampled_errors, to_np

pytestmark = pytest.mark.gpu

TIGHT = 8e-3


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def whole(x, algo):
    return gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                       state_in=x["state_in"], algo=algo)


def streamed(x, piece, **kw):
    o, st = gdn_prefill_streamed(x["q"], x["k"], x["v"], x["g"], x["beta"], piece,
                                 state_in=x["state_in"], **kw)
    assert gdn_stream_status() == "GDN_OK"
    return o, st


@pytest.mark.parametrize("T,piece", [(1000, 256), (320, 64), (17, 64), (4096, 1024),
                                     (4100, 4096), (64, 64)])
def test_streamed_equals_whole_bitwise(T, piece):
    d = inputs.make_prefill([T], 2, 4, 128, 64, "bf16", seed=T + piece, state_std=0.05)
    x = dev(d)
    o_ref, s_ref = whole(x, "chunked_split")
    o, st = streamed(x, piece)
    assert torch.equal(o, o_ref) and torch.equal(st, s_ref)
    o_or, s_or = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], 2, 4,
                                128, 64, state_in=d["state_in"])
    assert rel_l2(to_np(o), o_or) < TIGHT and rel_l2(to_np(st), s_or) < TIGHT


def test_streamed_fp32_runs_the_scan_bitwise():
    d = inputs.make_prefill([200], 1, 2, 32, 16, "f32", seed=61, state_std=0.1)
    x = dev(d)
    o_ref, s_ref = whole(x, "scan")
    o, st = streamed(x, 64)
    assert torch.equal(o, o_ref) and torch.equal(st, s_ref)


def test_streamed_in_place_state_and_empty_prompt():
    d = inputs.make_prefill([300], 2, 4, 128, 32, "bf16", seed=62, state_std=0.1)
    x = dev(d)
    o_ref, s_ref = whole(x, "chunked_split")
    st = x["state_in"].clone()
    o, _ = gdn_prefill_streamed(x["q"], x["k"], x["v"], x["g"], x["beta"], 128, state_in=st,
                                state_out=st)
    assert torch.equal(o, o_ref) and torch.equal(st, s_ref)
    e = dev(inputs.make_prefill([0], 2, 4, 128, 32, "bf16", seed=63, state_std=0.1))
    o, st = gdn_prefill_streamed(e["q"], e["k"], e["v"], e["g"], e["beta"], 64,
                                 state_in=e["state_in"])
    assert gdn_stream_status() == "GDN_OK" and torch.equal(st, e["state_in"])


def test_streamed_128k_prompt_bounded_workspace():
    """The 128K-token prompt with a drawn state, in pieces of 8192 tokens: the
    workspace is that of one piece, the result the whole call's bit for bit."""
    w = inputs.WORKLOADS["prefill_t131072"]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"], state_std=w["state_std"])
    x = dev(d)
    need = gdn_prefill_streamed_workspace_size(8192, 16, 32, 128, 128)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, st = streamed(x, 8192, workspace=ws)
    o_ref, s_ref = whole(x, "chunked_split")
    assert torch.equal(o, o_ref) and torch.equal(st, s_ref)
    eo, es = sampled_errors(d, o, st, sample_tasks(1, 32, 128, 16, seed=3))
    assert eo < TIGHT and es < TIGHT, (eo, es)
