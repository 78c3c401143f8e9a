"""gdn_decode_multi (several tokens per sequence in one launch, optional
per-token state snapshots): bit-exact against successive gdn_decode_step calls,
and against the fp64 oracle within the fp32 / bf16 tolerances."""
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_multi, gdn_decode_step,
                                                    gdn_stream_status, inputs)
from tests.util import rel_l2, to_np, tol_for

pytestmark = pytest.mark.gpu


def make(B, n, h_k, h_v, d_k, d_v, dtype, seed):
    d = inputs.make_prefill([n] * B, h_k, h_v, d_k, d_v, dtype, seed=seed, state_std=0.05)
    x = {key: (val.cuda() if isinstance(val, torch.Tensor) else val) for key, val in d.items()}
    shp = lambda t, *tail: t.reshape(B, n, *tail).contiguous()
    y = dict(q=shp(x["q"], h_k, d_k), k=shp(x["k"], h_k, d_k), v=shp(x["v"], h_v, d_v),
             g=shp(x["g"], h_v), beta=shp(x["beta"], h_v), state=x["state_in"].clone())
    return d, y


def successive_steps(y):
    state = y["state"].clone()
    outs, snaps = [], []
    for t in range(y["q"].shape[1]):
        outs.append(gdn_decode_step(y["q"][:, t].contiguous(), y["k"][:, t].contiguous(),
                                    y["v"][:, t].contiguous(), y["g"][:, t].contiguous(),
                                    y["beta"][:, t].contiguous(), state))
        snaps.append(state.clone())
    return torch.stack(outs, 1), state, torch.stack(snaps, 1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [1, 2, 5])
@pytest.mark.parametrize("h_k,h_v,d_k,d_v", [(2, 4, 128, 128), (1, 2, 64, 32), (2, 2, 16, 16),
                                             (1, 1, 32, 64)])
def test_multi_equals_successive_steps_bitwise(n, h_k, h_v, d_k, d_v, dtype):
    d, y = make(3, n, h_k, h_v, d_k, d_v, dtype, seed=71 + n + d_k)
    o_ref, s_ref, snap_ref = successive_steps(y)
    state = y["state"].clone()
    o, snap = gdn_decode_multi(y["q"], y["k"], y["v"], y["g"], y["beta"], state, snapshots=True)
    assert gdn_stream_status() == "GDN_OK"
    assert torch.equal(o, o_ref) and torch.equal(state, s_ref) and torch.equal(snap, snap_ref)
    state2 = y["state"].clone()  # without snapshots: same outputs and final state
    o2 = gdn_decode_multi(y["q"], y["k"], y["v"], y["g"], y["beta"], state2)
    assert torch.equal(o2, o_ref) and torch.equal(state2, s_ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_multi_against_oracle_with_snapshots(dtype):
    B, n, h_k, h_v, d_k, d_v = 4, 5, 2, 4, 128, 64
    d, y = make(B, n, h_k, h_v, d_k, d_v, dtype, seed=81)
    state = y["state"].clone()
    o, snap = gdn_decode_multi(y["q"], y["k"], y["v"], y["g"], y["beta"], state, snapshots=True,
                               scale=0.5)
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                  h_k, h_v, d_k, d_v, state_in=d["state_in"], scale=0.5)
    tol = tol_for(dtype)
    assert rel_l2(to_np(o).reshape(o_ref.shape), o_ref) < tol
    assert rel_l2(to_np(state), s_ref) < 1e-5
    for t in range(n):  # snapshot t: the state after the first t + 1 tokens of every sequence
        sub = {key: d[key].reshape(B, n, *d[key].shape[1:])[:, :t + 1].reshape(
            B * (t + 1), *d[key].shape[1:]) for key in ("q", "k", "v", "g", "beta")}
        cu = torch.arange(0, B + 1, dtype=torch.int32) * (t + 1)
        _, s_t = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], cu, h_k, h_v,
                                d_k, d_v, state_in=d["state_in"], scale=0.5)
        assert rel_l2(to_np(snap[:, t]), s_t) < 1e-5, t


def test_multi_batched_decode_shape():
    """256 sequences x 4 tokens x 32 value heads of 128: bit-exact against four steps."""
    d, y = make(256, 4, 16, 32, 128, 128, "bf16", seed=82)
    o_ref, s_ref, _ = successive_steps(y)
    state = y["state"].clone()
    o = gdn_decode_multi(y["q"], y["k"], y["v"], y["g"], y["beta"], state)
    assert torch.equal(o, o_ref) and torch.equal(state, s_ref)
