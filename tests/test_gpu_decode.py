"""Parity of gdn_decode_step (CUDA) with the fp64 oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import gdn_decode_step, inputs
from tests.util import rel_l2, to_np, tol_for

pytestmark = pytest.mark.gpu


def run_case(d, scale=1.0):
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    state = dev["state"].clone()
    o = gdn_decode_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], state, scale=scale)
    torch.cuda.synchronize()
    B = d["q"].shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, d["h_k"],
                                  d["h_v"], d["d_k"], d["d_v"], state_in=d["state"], scale=scale)
    return to_np(o), to_np(state), o_ref, s_ref


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d_k,d_v", [(16, 16), (32, 64), (64, 32), (128, 128), (128, 16)])
@pytest.mark.parametrize("h_k,h_v", [(1, 1), (2, 4), (4, 4)])
def test_decode_shapes(dtype, d_k, d_v, h_k, h_v):
    d = inputs.make_decode(3, h_k, h_v, d_k, d_v, dtype=dtype, seed=d_k * 7 + d_v + h_v,
                           state_std=0.3)
    o, s, o_ref, s_ref = run_case(d, scale=0.8)
    assert rel_l2(o, o_ref) < tol_for(dtype)
    assert rel_l2(s, s_ref) < 1e-5  # fp32 state arithmetic on exact inputs


@pytest.mark.parametrize("batch", [1, 5, 256])
def test_decode_full_heads(batch):
    """16 key heads, 32 value heads of 128, at batch 1 and the batched 256."""
    d = inputs.make_decode(batch, 16, 32, 128, 128, dtype="bf16", seed=20261206 + batch)
    o, s, o_ref, s_ref = run_case(d)
    assert rel_l2(o, o_ref) < 2e-2
    assert rel_l2(s, s_ref) < 1e-5
    # internal check: o is bf16-rounded only
    assert rel_l2(o, o_ref) < 5e-3


def test_decode_30_layers():
    """Batch-1 decode through 30 layers, each with its own state, in place."""
    wl = inputs.WORKLOADS["decode_b1_x30layers"]
    for layer in range(30):
        d = inputs.make_decode(1, 16, 32, 128, 128, dtype="bf16", seed=wl["seed"] * 100 + layer)
        o, s, o_ref, s_ref = run_case(d)
        assert rel_l2(o, o_ref) < 2e-2 and rel_l2(s, s_ref) < 1e-5, f"layer {layer}"


def test_batched_row_equals_single_call_bitwise():
    d = inputs.make_decode(7, 2, 4, 64, 32, dtype="bf16", seed=3)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    st = dev["state"].clone()
    o = gdn_decode_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], st)
    for b in range(7):
        st1 = dev["state"][b:b + 1].clone()
        o1 = gdn_decode_step(dev["q"][b:b + 1].contiguous(), dev["k"][b:b + 1].contiguous(),
                             dev["v"][b:b + 1].contiguous(), dev["g"][b:b + 1].contiguous(),
                             dev["beta"][b:b + 1].contiguous(), st1)
        assert torch.equal(o1[0], o[b]) and torch.equal(st1[0], st[b])


def test_decode_deterministic():
    d = inputs.make_decode(4, 16, 32, 128, 128, dtype="bf16", seed=9)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    outs = []
    for _ in range(2):
        st = dev["state"].clone()
        o = gdn_decode_step(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], st)
        outs.append((o, st))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_decode_special_cases():
    """beta = 0, g = 0 leaves the state unchanged; g = -200 (alpha underflows to
    exactly 0 in fp32) resets it to beta v k^T."""
    d = inputs.make_decode(2, 1, 2, 32, 32, dtype="f32", seed=4, state_std=0.5)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    st = dev["state"].clone()
    gdn_decode_step(dev["q"], dev["k"], dev["v"], torch.zeros_like(dev["g"]),
                    torch.zeros_like(dev["beta"]), st)
    assert torch.equal(st, dev["state"])
    st = dev["state"].clone()
    gdn_decode_step(dev["q"], dev["k"], dev["v"], torch.full_like(dev["g"], -200.0),
                    dev["beta"], st)
    k = dev["k"][:, 0]  # one key head
    expect = dev["beta"][:, :, None, None] * dev["v"][:, :, :, None] * k[:, None, None, :]
    torch.testing.assert_close(st, expect, rtol=1e-6, atol=1e-7)
