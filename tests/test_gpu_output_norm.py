"""The output RMS normalisation: fused into the decode step
(gdn_decode_step_rmsnorm: the CTAs of a (sequence, head) exchange their partial
sums of squares in a thread-block cluster) and as a pass of its own
(gdn_output_rmsnorm), against the fp64 oracle (the recurrence, then the
normalisation).  The fused step's state equals the plain step's bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_step, gdn_decode_step_rmsnorm,
                                                    gdn_output_rmsnorm, gdn_prefill,
                                                    gdn_stream_status, inputs)
from oracle.output_norm import output_rmsnorm
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def ref_decode_norm(d, w, eps, scale=1.0):
    B = d["q"].shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, d["h_k"],
                                  d["h_v"], d["d_k"], d["d_v"], state_in=d["state"], scale=scale)
    return output_rmsnorm(o_ref, None if w is None else w.cpu(), eps), s_ref


# (batch, d_k, d_v): batch 1 uses 16 rows per CTA (clusters of d_v / 16 CTAs),
# batch 256 at 32 heads x 128 uses 64 rows per CTA (clusters of 2)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("batch,d_k,d_v", [(1, 128, 128), (1, 128, 64), (3, 64, 32), (2, 16, 16),
                                           (1, 32, 128), (256, 128, 128)])
def test_fused_decode_norm(dtype, batch, d_k, d_v):
    h_k, h_v = (16, 32) if batch == 256 else (2, 4)
    d = inputs.make_decode(batch, h_k, h_v, d_k, d_v, dtype=dtype, seed=batch * 7 + d_v + d_k,
                           state_std=0.3)
    x = dev(d)
    w = torch.linspace(0.5, 1.5, d_v, dtype=torch.float32, device="cuda")
    eps = 1e-5
    st_plain = x["state"].clone()
    gdn_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], st_plain, scale=0.8)
    st = x["state"].clone()
    o = gdn_decode_step_rmsnorm(x["q"], x["k"], x["v"], x["g"], x["beta"], st, norm_weight=w,
                                norm_eps=eps, scale=0.8)
    assert gdn_stream_status() == "GDN_OK"
    assert torch.equal(st, st_plain)
    o_ref, s_ref = ref_decode_norm(d, w, eps, scale=0.8)
    tol = 1e-4 if dtype == "f32" else 5e-3  # fp32 arithmetic; bf16: the output's rounding
    assert rel_l2(to_np(o), o_ref) < tol
    assert rel_l2(to_np(st), s_ref) < 1e-5


def test_fused_decode_norm_unit_weight_and_qk_option():
    d = inputs.make_decode(4, 2, 4, 128, 128, dtype="bf16", seed=91, state_std=0.1)
    x = dev(d)
    st = x["state"].clone()
    o = gdn_decode_step_rmsnorm(x["q"], x["k"], x["v"], x["g"], x["beta"], st, norm_weight=None,
                                norm_eps=0.0, qk_l2norm=True)
    assert gdn_stream_status() == "GDN_OK"
    # unit weight, eps = 0: every (sequence, head) row has RMS 1 (up to bf16 rounding)
    rms = o.float().pow(2).mean(-1).sqrt()
    assert torch.allclose(rms, torch.ones_like(rms), atol=5e-3)
    B = d["q"].shape[0]
    o_ref, _ = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"],
                              np.arange(B + 1, dtype=np.int32), 2, 4, 128, 128,
                              state_in=d["state"], qk_l2norm=True)
    assert rel_l2(to_np(o), output_rmsnorm(o_ref, None, 0.0)) < 5e-3


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d_v", [16, 32, 64, 128])
def test_standalone_norm_on_prefill_output(dtype, d_v):
    d = inputs.make_prefill([70, 0, 130], 2, 4, 64, d_v, dtype, seed=d_v + 3, state_std=0.05)
    x = dev(d)
    o, _ = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                       state_in=x["state_in"], algo="scan")
    assert gdn_stream_status() == "GDN_OK"
    before = o.clone()
    w = torch.randn(d_v, dtype=torch.float32, device="cuda")
    gdn_output_rmsnorm(o, norm_weight=w, norm_eps=1e-6)
    assert gdn_stream_status() == "GDN_OK"
    want = output_rmsnorm(before.cpu(), w.cpu(), 1e-6)  # of the stored values
    tol = 1e-6 if dtype == "f32" else 5e-3
    assert rel_l2(to_np(o), want) < tol
