"""The in-kernel q/k L2 normalisation option (GDN_OPT_QK_L2NORM) on every path:
raw N(0, 1) q and k, against the fp64 oracle with the same option; the decode
forms bit-exact against each other; the streamed prefill bit-exact against the
whole call."""
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_multi, gdn_decode_step,
                                                    gdn_prefill, gdn_prefill_streamed,
                                                    gdn_stream_status, inputs)
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu

TIGHT = 8e-3  # bf16 tensor-core and bf16-input paths
F32 = 1e-4


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def oracle_run(d, scale):
    return oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["h_k"],
                          d["h_v"], d["d_k"], d["d_v"], state_in=d["state_in"], scale=scale,
                          qk_l2norm=True)


@pytest.mark.parametrize("algo,dtype,d_k,d_v", [("scan", "f32", 64, 32), ("scan", "bf16", 128, 64),
                                                ("chunked", "bf16", 128, 64),
                                                ("chunked_split", "bf16", 128, 64),
                                                ("chunked_split", "bf16", 128, 128),
                                                ("auto", "bf16", 128, 32)])
def test_prefill_qk_l2norm_against_oracle(algo, dtype, d_k, d_v):
    d = inputs.make_prefill([77, 300, 1, 0, 64], 2, 4, d_k, d_v, dtype, seed=91 + d_v,
                            state_std=0.05, unit_qk=False)
    x = dev(d)
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], scale=0.7, algo=algo, qk_l2norm=True)
    assert gdn_stream_status() == "GDN_OK"
    o_ref, s_ref = oracle_run(d, 0.7)
    tol = F32 if dtype == "f32" else TIGHT
    eo, es = rel_l2(to_np(o), o_ref), rel_l2(to_np(st), s_ref)
    assert eo < tol and es < tol, (eo, es)
    # the option is not a no-op on these inputs (without it the raw |k|^2 ~ d_k
    # makes the delta rule blow up)
    o0, _ = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], scale=0.7, algo=algo)
    assert not torch.equal(o0, o)


def test_fused_form_refuses_the_option():
    from gated_deltanet_linear_recurrence_gb300 import GdnError
    d = inputs.make_prefill([100], 1, 2, 128, 32, "bf16", seed=95, unit_qk=False)
    x = dev(d)
    with pytest.raises(GdnError, match="INVALID_ARG"):
        gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                    algo="chunked_fused", qk_l2norm=True)


def test_prefill_t4096_qk_l2norm():
    d = inputs.make_prefill([4096], 16, 32, 128, 128, "bf16", seed=92, unit_qk=False)
    x = dev(d)
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        qk_l2norm=True)
    o_ref, s_ref = oracle_run(d, 1.0)
    eo, es = rel_l2(to_np(o), o_ref), rel_l2(to_np(st), s_ref)
    assert eo < TIGHT and es < TIGHT, (eo, es)


def test_streamed_qk_l2norm_bitwise():
    d = inputs.make_prefill([1000], 2, 4, 128, 64, "bf16", seed=93, state_std=0.05,
                            unit_qk=False)
    x = dev(d)
    o_ref, s_ref = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                               state_in=x["state_in"], algo="chunked_split", qk_l2norm=True)
    o, st = gdn_prefill_streamed(x["q"], x["k"], x["v"], x["g"], x["beta"], 256,
                                 state_in=x["state_in"], qk_l2norm=True)
    assert torch.equal(o, o_ref) and torch.equal(st, s_ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_qk_l2norm(dtype):
    B, n, h_k, h_v, d_k, d_v = 3, 4, 2, 4, 128, 64
    d = inputs.make_prefill([n] * B, h_k, h_v, d_k, d_v, dtype, seed=94, state_std=0.05,
                            unit_qk=False)
    x = dev(d)
    shp = lambda t, *tail: t.reshape(B, n, *tail).contiguous()
    y = dict(q=shp(x["q"], h_k, d_k), k=shp(x["k"], h_k, d_k), v=shp(x["v"], h_v, d_v),
             g=shp(x["g"], h_v), beta=shp(x["beta"], h_v))
    state = x["state_in"].clone()
    o_m = gdn_decode_multi(y["q"], y["k"], y["v"], y["g"], y["beta"], state, scale=0.5,
                           qk_l2norm=True)
    s_steps = x["state_in"].clone()
    o_s = torch.stack([gdn_decode_step(y["q"][:, t].contiguous(), y["k"][:, t].contiguous(),
                                       y["v"][:, t].contiguous(), y["g"][:, t].contiguous(),
                                       y["beta"][:, t].contiguous(), s_steps, scale=0.5,
                                       qk_l2norm=True) for t in range(n)], 1)
    assert gdn_stream_status() == "GDN_OK"
    assert torch.equal(o_m, o_s) and torch.equal(state, s_steps)
    o_ref, s_ref = oracle_run(d, 0.5)
    tol = F32 if dtype == "f32" else 2e-2
    assert rel_l2(to_np(o_m).reshape(o_ref.shape), o_ref) < tol
    assert rel_l2(to_np(state), s_ref) < 1e-5
