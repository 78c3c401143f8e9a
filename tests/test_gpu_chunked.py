"""Parity of the chunked tcgen05 prefill with the fp64 oracle, and its bit-exact
invariants (varlen offsets, split prefill).  Edge cases run both forms: the
fused kernel (algo='chunked_fused') and the two kernels that meet in a
workspace (algo='chunked_split'); algo='chunked' lets the library choose."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import gdn_prefill, gdn_stream_status, inputs
from tests.util import rel_l2, sample_tasks, sampled_errors, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-2      # contract for the bf16 tensor-core path
TIGHT = 8e-3    # what the bf16 operand roundings leave in practice
KERNELS = ["chunked_fused", "chunked_split"]


def dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run(d, algo="chunked", scale=1.0):
    x = dev(d)
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], scale=scale, algo=algo)
    assert gdn_stream_status() == "GDN_OK"
    return o, st


def full_errors(d, o, st, scale=1.0):
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                  d["h_k"], d["h_v"], d["d_k"], d["d_v"],
                                  state_in=d["state_in"], scale=scale)
    eo = rel_l2(to_np(o), o_ref) if d["q"].shape[0] else 0.0
    return eo, rel_l2(to_np(st), s_ref)


@pytest.mark.parametrize("algo", KERNELS)
@pytest.mark.parametrize("lengths", [[1], [63], [64], [65], [127], [129], [0, 5], [3, 0, 70, 1],
                                     [200, 64, 130]])
def test_lengths(lengths, algo):
    d = inputs.make_prefill(lengths, 2, 4, 128, 64, "bf16", seed=sum(lengths) + 7,
                            state_std=0.05)
    o, st = run(d, algo=algo, scale=0.9)
    eo, es = full_errors(d, o, st, scale=0.9)
    assert eo < TIGHT and es < TIGHT, (eo, es)


@pytest.mark.parametrize("algo", KERNELS)
@pytest.mark.parametrize("d_v", [32, 64, 128])
@pytest.mark.parametrize("h_k,h_v", [(1, 1), (2, 4), (2, 2)])
def test_shapes(d_v, h_k, h_v, algo):
    d = inputs.make_prefill([77, 300], h_k, h_v, 128, d_v, "bf16", seed=d_v + 3 * h_v,
                            state_std=0.02)
    o, st = run(d, algo=algo)
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)


@pytest.mark.parametrize("algo", KERNELS)
def test_null_state_is_zero(algo):
    d = inputs.make_prefill([150], 1, 2, 128, 32, "bf16", seed=9)
    x = dev(d)
    o, st = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        algo=algo)
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT


@pytest.mark.parametrize("algo", KERNELS)
def test_state_aliasing_in_place(algo):
    d = inputs.make_prefill([100, 64], 1, 2, 128, 64, "bf16", seed=10, state_std=0.1)
    x = dev(d)
    st = x["state_in"].clone()
    o, _ = gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                       state_in=st, state_out=st, algo=algo)
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT


def test_prefill_t4096_full_oracle():
    """The 4096-token prompt, 16 key / 32 value heads of 128, bf16, zero state."""
    w = inputs.WORKLOADS["prefill_t4096"]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"])
    o, st = run(d, algo="chunked_split")
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)
    o2, st2 = run(d, algo="auto")  # AUTO takes the cooperative form at this length
    assert torch.equal(o2, o) and torch.equal(st2, st)


@pytest.mark.parametrize("algo", KERNELS)
def test_varlen_bitwise_equals_single_sequence(algo):
    lengths = [5, 64, 0, 130, 1, 257]
    d = inputs.make_prefill(lengths, 2, 4, 128, 64, "bf16", seed=11, state_std=0.05)
    o, st = run(d, algo=algo)
    cu = d["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        sub = dict(d, q=d["q"][a:b], k=d["k"][a:b], v=d["v"][a:b], g=d["g"][a:b],
                   beta=d["beta"][a:b], state_in=d["state_in"][n:n + 1],
                   cu_seqlens=torch.tensor([0, b - a], dtype=torch.int32))
        o1, s1 = run(sub, algo=algo)
        assert torch.equal(o1, o[a:b]) and torch.equal(s1[0], st[n]), n


@pytest.mark.parametrize("algo", KERNELS)
def test_split_at_chunk_boundary_bitwise(algo):
    """prefill(T1) -> state -> prefill(T2) equals prefill(T1 + T2) bit for bit
    when T1 is a multiple of the chunk length."""
    d = inputs.make_prefill([320], 2, 4, 128, 64, "bf16", seed=12, state_std=0.02)
    o, st = run(d, algo=algo)
    x = dev(d)
    T1 = 128
    cu1 = torch.tensor([0, T1], dtype=torch.int32, device="cuda")
    cu2 = torch.tensor([0, 320 - T1], dtype=torch.int32, device="cuda")
    o1, s1 = gdn_prefill(x["q"][:T1], x["k"][:T1], x["v"][:T1], x["g"][:T1], x["beta"][:T1],
                         cu1, state_in=x["state_in"], algo=algo)
    o2, s2 = gdn_prefill(x["q"][T1:], x["k"][T1:], x["v"][T1:], x["g"][T1:], x["beta"][T1:],
                         cu2, state_in=s1, algo=algo)
    assert torch.equal(torch.cat([o1, o2]), o) and torch.equal(s2, st)


@pytest.mark.parametrize("algo", KERNELS)
def test_deterministic(algo):
    d = inputs.make_prefill([500, 33], 2, 4, 128, 128, "bf16", seed=13, state_std=0.02)
    o1, s1 = run(d, algo=algo)
    o2, s2 = run(d, algo=algo)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_auto_mixed_lengths_runs_both_paths():
    """AUTO sends short sequences to the scan and long ones to the chunked kernel."""
    d = inputs.make_prefill([3, 400, 17, 90], 2, 4, 128, 64, "bf16", seed=14, state_std=0.05)
    o, st = run(d, algo="auto")
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT


@pytest.mark.parametrize("algo", KERNELS)
def test_reset_gate_and_no_write(algo):
    """g = -200 everywhere (alpha underflows to 0 in fp32) and beta = 0: the
    state decays to exactly 0 and o = 0; with g = 0, beta = 0 the state is kept."""
    d = inputs.make_prefill([130], 1, 2, 128, 32, "bf16", seed=15, state_std=0.3)
    x = dev(d)
    zero_b = torch.zeros_like(x["beta"])
    o, st = gdn_prefill(x["q"], x["k"], x["v"], torch.zeros_like(x["g"]), zero_b,
                        x["cu_seqlens"], state_in=x["state_in"], algo=algo)
    assert torch.equal(st, x["state_in"])  # alpha = 1, beta = 0: identity
    o, st = gdn_prefill(x["q"], x["k"], x["v"], torch.full_like(x["g"], -200.0), zero_b,
                        x["cu_seqlens"], state_in=x["state_in"], algo=algo)
    assert torch.count_nonzero(st) == 0 and torch.count_nonzero(o.float()) == 0


@pytest.mark.parametrize("algo", KERNELS)
def test_bad_cu_seqlens_reported(algo):
    d = inputs.make_prefill([70, 70], 1, 1, 128, 32, "bf16", seed=16)
    x = dev(d)
    cu = torch.tensor([0, 100, 90], dtype=torch.int32, device="cuda")
    st = torch.full((2, 1, 32, 128), 5.0, device="cuda")
    o = torch.zeros((140, 1, 32), dtype=torch.bfloat16, device="cuda")
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, state_out=st, o=o,
                algo=algo)
    assert gdn_stream_status() == "GDN_ERR_BAD_CU_SEQLENS"
    assert torch.all(st[1] == 5.0)


@pytest.mark.parametrize("algo", ["chunked_split", "chunked_coop"])
def test_bad_cu_seqlens_one_sequence(algo):
    """One sequence (no chunk-table kernel: the kernels check the range
    themselves) whose cu_seqlens ends past total_tokens: reported, and neither
    the output nor the state is touched."""
    d = inputs.make_prefill([130], 1, 2, 128, 64, "bf16", seed=17)
    x = dev(d)
    cu = torch.tensor([0, 200], dtype=torch.int32, device="cuda")
    st = torch.full((1, 2, 64, 128), 5.0, device="cuda")
    o = torch.zeros((130, 2, 64), dtype=torch.bfloat16, device="cuda")
    gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, state_out=st, o=o, algo=algo)
    assert gdn_stream_status() == "GDN_ERR_BAD_CU_SEQLENS"
    assert torch.all(st == 5.0) and torch.count_nonzero(o.float()) == 0


@pytest.fixture(scope="module")
def long_prefill():
    w = inputs.WORKLOADS["prefill_t131072"]
    return inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"],
                               w["dtype"], seed=w["seed"], state_std=w["state_std"])


def test_prefill_t131072_sampled(long_prefill):
    """One 128K-token prompt with a drawn initial state: 48 sampled value rows
    (all their outputs and final state rows) against the oracle."""
    d = long_prefill
    o, st = run(d)  # the library's choice: the two kernels at this length
    eo, es = sampled_errors(d, o, st, sample_tasks(1, 32, 128, 48, seed=1))
    assert eo < TIGHT and es < TIGHT, (eo, es)


def test_varlen_ten_sequences_sampled():
    """Ten packed prompts of 256 ... 128K tokens, zero initial states."""
    w = inputs.WORKLOADS["prefill_varlen10"]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"])
    o, st = run(d, algo="auto")
    eo, es = sampled_errors(d, o, st, sample_tasks(10, 32, 128, 6, seed=2))
    assert eo < TIGHT and es < TIGHT, (eo, es)


@pytest.mark.parametrize("lengths", [[200, 64, 130], [1], [4096]])
def test_fused_and_two_kernel_forms_agree(lengths):
    """The fused kernel and the two-kernel form agree within rounding."""
    d = inputs.make_prefill(lengths, 2, 4, 128, 64, "bf16", seed=len(lengths) + 21,
                            state_std=0.05)
    o, st = run(d, algo="chunked_fused")
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)
    o2, st2 = run(d, algo="chunked_split")
    assert rel_l2(to_np(o2), to_np(o)) < 5e-3 and rel_l2(to_np(st2), to_np(st)) < 5e-3


def test_library_choice_of_chunked_form():
    """algo='chunked' takes the two kernels (bitwise) only for sequences averaging
    256 tokens or more; shorter ones take the fused kernel and need no workspace."""
    from gated_deltanet_linear_recurrence_gb300 import gdn_prefill_workspace_size as wss
    assert wss(2, 500, 2, 4, 128, 64, algo="chunked") == 0
    assert wss(2, 500, 2, 4, 128, 64, algo="chunked_split") > 0
    assert wss(2, 512, 2, 4, 128, 64, algo="chunked") > 0
    assert wss(1, 4096, 2, 4, 128, 64, algo="chunked_fused") == 0
    for lengths, form in (([250, 250], "chunked_fused"), ([300, 212], "chunked_split")):
        d = inputs.make_prefill(lengths, 2, 4, 128, 64, "bf16", seed=23, state_std=0.05)
        o, st = run(d, algo="chunked")
        o2, st2 = run(d, algo=form)
        assert torch.equal(o, o2) and torch.equal(st, st2), form


def test_two_kernel_form_needs_workspace():
    from gated_deltanet_linear_recurrence_gb300 import GdnError
    d = inputs.make_prefill([100], 1, 2, 128, 32, "bf16", seed=24)
    x = dev(d)
    with pytest.raises(GdnError, match="WORKSPACE_TOO_SMALL"):
        gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                    algo="chunked_split", workspace=torch.empty(256, dtype=torch.uint8,
                                                                device="cuda"))


def test_workspace_size_covers_worst_case():
    """Many short sequences (each a partial chunk) stay within the reported bound."""
    lengths = [1, 65, 63, 2, 129, 0, 64]
    d = inputs.make_prefill(lengths, 1, 2, 128, 32, "bf16", seed=22, state_std=0.05)
    o, st = run(d, algo="chunked_split")
    eo, es = full_errors(d, o, st)
    assert eo < TIGHT and es < TIGHT, (eo, es)
