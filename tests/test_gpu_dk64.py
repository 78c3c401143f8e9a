"""The chunked evaluation at key dimension 64: the two-kernel and cooperative
forms read Q and K as 3-D tiles whose columns past d_k arrive as zeros, so the
tensor-core products run at 128 columns on zero-padded operands and the state
keeps 64 real key columns.  Parity with the fp64 oracle (partial chunks,
varlen with an empty sequence, carried state), bit-exact varlen offsets, the
cooperative form equal to the two kernels bit for bit, and AUTO's choice."""
import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill, gdn_prefill_form,
                                                    gdn_prefill_workspace_size,
                                                    gdn_stream_status, inputs)
from tests.test_gpu_chunked import TIGHT, dev, full_errors, run

pytestmark = pytest.mark.gpu

FORMS = ["chunked_split", "chunked_coop"]


@pytest.mark.parametrize("algo", FORMS)
@pytest.mark.parametrize("lengths", [[1], [63], [64], [65], [130], [0, 5], [3, 0, 70, 1],
                                     [200, 64, 130]])
def test_lengths_dk64(lengths, algo):
    d = inputs.make_prefill(lengths, 2, 4, 64, 64, "bf16", seed=sum(lengths) + 70,
                            state_std=0.05)
    o, st = run(d, algo=algo, scale=0.9)
    eo, es = full_errors(d, o, st, scale=0.9)
    assert eo < TIGHT and es < TIGHT, (eo, es)


@pytest.mark.parametrize("d_v", [32, 64, 128])
@pytest.mark.parametrize("h_k,h_v", [(1, 1), (2, 4), (4, 4)])
def test_shapes_dk64(d_v, h_k, h_v):
    d = inputs.make_prefill([77, 300], h_k, h_v, 64, d_v, "bf16", seed=d_v + 5 * h_v,
                            state_std=0.02)
    o, st = run(d, algo="chunked_split")
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)


def test_full_heads_t4096_dk64():
    """16 key / 32 value heads, d_k = 64, d_v = 128, a 4096-token prompt with a
    drawn initial state: AUTO (the cooperative form) against the full oracle and
    bit for bit against the two kernels."""
    d = inputs.make_prefill([4096], 16, 32, 64, 128, "bf16", seed=64, state_std=0.02)
    o, st = run(d, algo="auto")
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)
    o2, st2 = run(d, algo="chunked_split")
    assert torch.equal(o2, o) and torch.equal(st2, st)


def test_varlen_bitwise_equals_single_sequence_dk64():
    lengths = [5, 64, 0, 130, 1, 257]
    d = inputs.make_prefill(lengths, 2, 4, 64, 64, "bf16", seed=81, state_std=0.05)
    o, st = run(d, algo="chunked_split")
    cu = d["cu_seqlens"].tolist()
    x = dev(d)
    for n in range(len(lengths)):
        t0, t1 = cu[n], cu[n + 1]
        if t1 == t0:
            assert torch.equal(st[n], x["state_in"][n])
            continue
        on, sn = gdn_prefill(x["q"][t0:t1], x["k"][t0:t1], x["v"][t0:t1], x["g"][t0:t1],
                             x["beta"][t0:t1],
                             torch.tensor([0, t1 - t0], dtype=torch.int32, device="cuda"),
                             state_in=x["state_in"][n:n + 1].contiguous(), algo="chunked_split")
        assert gdn_stream_status() == "GDN_OK"
        assert torch.equal(on, o[t0:t1]) and torch.equal(sn[0], st[n])


def test_auto_without_workspace_scans_dk64():
    """No fused kernel at d_k = 64: AUTO given no workspace runs the token scan,
    and the result is the oracle's."""
    d = inputs.make_prefill([150], 1, 2, 64, 32, "bf16", seed=82)
    x = dev(d)
    T = 150
    assert gdn_prefill_workspace_size(1, T, 1, 2, 64, 32, torch.bfloat16) > 0
    assert gdn_prefill_form(1, T, 1, 2, 64, 32, torch.bfloat16, "auto", 0) == "scan"
    o = torch.empty((T, 2, 32), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((1, 2, 32, 64), dtype=torch.float32, device="cuda")
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], state_out=st, o=o,
                algo="auto", workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert gdn_stream_status() == "GDN_OK"
    eo, es = full_errors(d, o, st)
    assert eo < 5e-3 and es < 1e-4, (eo, es)
