"""Out-of-bounds writes: every output buffer is a view into a larger allocation
whose first and last 256 bytes hold random canary bytes; after each call the
canaries must be unchanged, bit for bit (a kernel writing past its output, or
before it, changes them without faulting).  Covers the scan, the fused,
two-kernel and cooperative chunked forms on ragged varlen input, the decode
step and multi-token step (state updated in place) and both decode-attention
layouts."""
import math

import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (gdn_attn_decode, gdn_decode_multi,
                                                    gdn_decode_step, gdn_decode_step_rmsnorm,
                                                    gdn_output_rmsnorm, gdn_prefill,
                                                    gdn_stream_status, inputs)

pytestmark = pytest.mark.gpu

PAD_BYTES = 256


class Canaried:
    """A device tensor of `shape` inside an allocation padded by canary bytes."""

    def __init__(self, shape, dtype, seed):
        esize = torch.empty((), dtype=dtype).element_size()
        self.pad = PAD_BYTES // esize
        self.n = math.prod(shape)
        self.buf = torch.empty(2 * self.pad + self.n, dtype=dtype, device="cuda")
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.buf.view(torch.uint8).random_(0, 256, generator=gen)
        self.t = self.buf[self.pad:self.pad + self.n].view(shape)
        self.edges0 = self.edges()

    def edges(self):
        b = self.buf.view(torch.uint8)
        e = PAD_BYTES
        return torch.cat([b[:e], b[b.numel() - e:]]).clone()

    def intact(self):
        return torch.equal(self.edges(), self.edges0)


def dev(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


@pytest.mark.parametrize("algo", ["scan", "chunked_fused", "chunked_split", "chunked_coop"])
def test_prefill_writes_stay_inside_o_and_state(algo):
    lengths = [300, 77]
    h_k, h_v, d_k, d_v = 2, 4, 128, 64
    x = dev(inputs.make_prefill(lengths, h_k, h_v, d_k, d_v, "bf16", seed=211, state_std=0.02))
    T, N = sum(lengths), len(lengths)
    o = Canaried((T, h_v, d_v), torch.bfloat16, seed=1)
    st = Canaried((N, h_v, d_v, d_k), torch.float32, seed=2)
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                state_in=x["state_in"], state_out=st.t, o=o.t, algo=algo)
    assert gdn_stream_status() == "GDN_OK"
    assert o.intact(), "a write landed outside o"
    assert st.intact(), "a write landed outside state_out"
    assert torch.isfinite(o.t.float()).all() and torch.isfinite(st.t).all()


def test_decode_step_writes_stay_inside_state_and_o():
    B, h_k, h_v, d_k, d_v = 3, 2, 4, 128, 64
    x = dev(inputs.make_decode(B, h_k, h_v, d_k, d_v, "bf16", seed=212))
    st = Canaried((B, h_v, d_v, d_k), torch.float32, seed=3)
    st.t.copy_(x["state"])
    o = Canaried((B, h_v, d_v), torch.bfloat16, seed=4)
    gdn_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], st.t, o=o.t)
    assert gdn_stream_status() == "GDN_OK"
    assert st.intact() and o.intact()


def test_normalised_decode_and_norm_pass_write_inside_their_buffers():
    B, h_k, h_v, d_k, d_v = 3, 2, 4, 128, 64
    x = dev(inputs.make_decode(B, h_k, h_v, d_k, d_v, "bf16", seed=215))
    st = Canaried((B, h_v, d_v, d_k), torch.float32, seed=8)
    st.t.copy_(x["state"])
    o = Canaried((B, h_v, d_v), torch.bfloat16, seed=9)
    w = torch.ones(d_v, dtype=torch.float32, device="cuda")
    gdn_decode_step_rmsnorm(x["q"], x["k"], x["v"], x["g"], x["beta"], st.t, norm_weight=w,
                            o=o.t)
    assert gdn_stream_status() == "GDN_OK"
    assert st.intact() and o.intact()
    gdn_output_rmsnorm(o.t, norm_weight=w)
    assert gdn_stream_status() == "GDN_OK"
    assert o.intact()


def test_decode_multi_writes_stay_inside_state_and_o():
    B, n, h_k, h_v, d_k, d_v = 3, 4, 2, 4, 128, 64
    d = dev(inputs.make_prefill([n] * B, h_k, h_v, d_k, d_v, "bf16", seed=213, state_std=0.05))
    shp = lambda t, *tail: t.reshape(B, n, *tail).contiguous()
    st = Canaried((B, h_v, d_v, d_k), torch.float32, seed=5)
    st.t.copy_(d["state_in"])
    o = Canaried((B, n, h_v, d_v), torch.bfloat16, seed=6)
    gdn_decode_multi(shp(d["q"], h_k, d_k), shp(d["k"], h_k, d_k), shp(d["v"], h_v, d_v),
                     shp(d["g"], h_v), shp(d["beta"], h_v), st.t, o=o.t)
    assert gdn_stream_status() == "GDN_OK"
    assert st.intact() and o.intact()


@pytest.mark.parametrize("layout", ["general", "fixed_block"])
def test_attention_writes_stay_inside_o(layout):
    x = dev(inputs.make_attention(2, 16, 2, 256, 512, [512, 100], seed=214))
    o = Canaried((2, 16, 256), torch.bfloat16, seed=7)
    gdn_attn_decode(x["q"], x["k_cache"], x["v_cache"], x["cache_len"], o=o.t, layout=layout)
    assert gdn_stream_status() == "GDN_OK"
    assert o.intact()
    assert torch.isfinite(o.t.float()).all()
