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
    """algo='auto' on a sequence above the measured crossover (8,192 tokens) runs
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
