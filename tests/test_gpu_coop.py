"""The cooperative chunked prefill (GDN_ALGO_CHUNKED_COOP: prepare slots and
64-row chains in one resident grid, chained by per-item ready flags) against the
two-kernel form: the same packages and the same per-element arithmetic (the
chain's products are per output element independent of how many rows one CTA
owns), so the two agree bit for bit; the two-kernel form is itself checked
against the fp64 oracle in test_gpu_chunked.py."""
import pytest
import torch

from gated_deltanet_linear_recurrence_gb300 import (GdnError, gdn_prefill, gdn_stream_status,
                                                    inputs)

pytestmark = pytest.mark.gpu


def both(lengths, h_k=16, h_v=32, state_std=0.0, qk=False, seed=5):
    x = inputs.make_prefill(lengths, h_k, h_v, 128, 128, "bf16", seed=seed, state_std=state_std,
                            unit_qk=not qk)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    out = {}
    for algo in ("chunked_split", "chunked_coop"):
        o, s = gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                           state_in=d["state_in"], algo=algo, qk_l2norm=qk)
        torch.cuda.synchronize()
        assert gdn_stream_status() == "GDN_OK"
        out[algo] = (o, s)
    assert torch.equal(out["chunked_split"][0], out["chunked_coop"][0]), "outputs differ"
    assert torch.equal(out["chunked_split"][1], out["chunked_coop"][1]), "states differ"


@pytest.mark.parametrize("T", [64, 1000, 4096, 16384])
def test_one_sequence(T):
    both([T])


def test_carried_state_and_qk_normalisation():
    both([2500], state_std=0.02)
    both([777], qk=True)


def test_few_sequences():
    both([3000, 40, 700], h_k=4, h_v=8)


def test_too_many_chains_is_refused():
    """More 64-row chains than two thirds of the SMs: the cooperative form is refused."""
    x = inputs.make_prefill([64] * 8, 16, 32, 128, 128, "bf16", seed=1)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    with pytest.raises(GdnError, match="UNSUPPORTED_SHAPE"):
        gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                    algo="chunked_coop")


def test_library_choice_takes_the_cooperative_form():
    """algo='auto' on a sequence above the measured crossover (4,096 tokens) runs
    the cooperative form through the workspace the size query reports."""
    x = inputs.make_prefill([9000], 2, 4, 128, 64, "bf16", seed=9, state_std=0.02)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    outs = []
    for algo in ("auto", "chunked", "chunked_coop", "chunked_split"):
        o, s = gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                           state_in=d["state_in"], algo=algo)
        torch.cuda.synchronize()
        assert gdn_stream_status() == "GDN_OK"
        outs.append((o, s))
    for o, s in outs[1:]:
        assert torch.equal(outs[0][0], o) and torch.equal(outs[0][1], s)


def test_auto_mixes_the_cooperative_form_and_the_scan():
    """AUTO on a batch averaging more than 4,096 tokens with one sequence below the
    scan crossover: the long sequence runs the cooperative form, the short one the
    token scan, in the same call; both against the fp64 oracle."""
    import numpy as np
    import oracle

    x = inputs.make_prefill([16500, 9], 2, 4, 128, 64, "bf16", seed=21, state_std=0.02)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    o, s = gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                       state_in=d["state_in"], algo="auto")
    torch.cuda.synchronize()
    assert gdn_stream_status() == "GDN_OK"
    o_ref, s_ref = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                                  2, 4, 128, 64, state_in=x["state_in"])

    def rel(a, b):
        a = np.asarray(a, np.float64)
        return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))

    assert rel(o.float().cpu().numpy(), o_ref) < 8e-3
    assert rel(s.cpu().numpy(), s_ref) < 8e-3
    # the short sequence alone through the scan: bitwise the same rows
    t0 = 16500
    o9, s9 = gdn_prefill(d["q"][t0:], d["k"][t0:], d["v"][t0:], d["g"][t0:], d["beta"][t0:],
                         torch.tensor([0, 9], dtype=torch.int32, device="cuda"),
                         state_in=d["state_in"][1:].contiguous(), algo="scan")
    torch.cuda.synchronize()
    assert torch.equal(o9, o[t0:]) and torch.equal(s9[0], s[1])
