"""gdn_prefill_host (inputs and outputs in host memory, copies overlapped with
the prefill) against gdn_prefill_streamed on the device with the same piece
size: the two must agree bit for bit (the streamed prefill is itself checked
against the fp64 oracle in test_gpu_stream.py), for whole and ragged prompts,
an empty prompt, a carried-in state, page-locked and pageable host memory,
fp32 inputs (the token scan) and the q/k normalisation option."""
import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill_host, gdn_prefill_streamed,
                                                    gdn_stream_status, inputs)

pytestmark = pytest.mark.gpu


def run_pair(T, piece, h_k=16, h_v=32, d=128, dtype="bf16", state_std=0.0, pin=True, qk=False,
             seed=11):
    x = inputs.make_prefill([T], h_k, h_v, d, d, dtype, seed=seed, state_std=state_std,
                            unit_qk=not qk)
    host = {k: x[k] for k in ("q", "k", "v", "g", "beta")}
    if pin:
        host = {k: t.pin_memory() for k, t in host.items()}
    si = x["state_in"]
    si_host = None if si is None else (si.pin_memory() if pin else si)
    o_h, s_h = gdn_prefill_host(host["q"], host["k"], host["v"], host["g"], host["beta"], piece,
                                state_in=si_host, qk_l2norm=qk)
    torch.cuda.synchronize()
    assert gdn_stream_status() == "GDN_OK"
    dev = {k: t.cuda() for k, t in host.items()}
    o_d, s_d = gdn_prefill_streamed(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], piece,
                                    state_in=None if si is None else si.cuda(), qk_l2norm=qk)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()), "outputs differ"
    assert torch.equal(s_h, s_d.cpu()), "final states differ"


@pytest.mark.parametrize("T,piece", [(4096, 1024), (1000, 256), (64, 64), (4096, 4096)])
def test_equals_streamed(T, piece):
    run_pair(T, piece)


def test_carried_state_and_pageable_memory():
    run_pair(700, 128, state_std=0.02, pin=True)
    run_pair(700, 128, state_std=0.02, pin=False)


def test_empty_prompt_copies_the_state():
    run_pair(0, 64, state_std=0.02)


def test_fp32_inputs_take_the_token_scan():
    run_pair(300, 128, h_k=2, h_v=4, d=32, dtype="f32")


def test_qk_normalisation():
    run_pair(520, 128, qk=True)
