"""CPU pins of the fp64 oracle (no GPU needed)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_recurrence_gb300 import inputs
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(mutant=0)


# Each planted mistake in the oracle (gate not exponentiated, dropped or
# sign-flipped delta correction, unscaled write, readout with k, readout before
# the update, wrong head map, gate ignored, gate on the write, transposed state,
# scale ignored, q left unnormalised, scale applied before the normalisation)
# must make at least one pin fail.
MUTANTS = list(range(1, 14))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_planted_mistake(mutant):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant=mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught planted mistake #{mutant}"


def test_oracle_rejects_bad_cu_seqlens():
    q = np.zeros((4, 1, 4))
    g = np.zeros((4, 1))
    for cu in ([1, 4], [0, 3], [0, 3, 2, 4]):
        with pytest.raises(ValueError):
            oracle.prefill(q, q, q, g, g, np.array(cu, np.int32), 1, 1, 4, 4)


def test_oracle_bf16_widening_is_exact():
    """bf16 inputs are widened exactly: same result as passing the widened fp64."""
    d = inputs.make_prefill([19], 1, 2, 8, 8, dtype="bf16", seed=1, state_std=0.1)
    args = (d["cu_seqlens"], 1, 2, 8, 8)
    o1, s1 = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], *args,
                            state_in=d["state_in"])
    o2, s2 = oracle.prefill(d["q"].double(), d["k"].double(), d["v"].double(),
                            d["g"].double(), d["beta"].double(), *args,
                            state_in=d["state_in"].double())
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_generator_sanity():
    """q and k are unit-norm before rounding, beta in (0, 1), g < 0; seeded."""
    d = inputs.make_prefill([100, 28], 2, 4, 16, 8, dtype="f32", seed=5, state_std=0.02)
    nq = d["q"].double().norm(dim=-1)
    nk = d["k"].double().norm(dim=-1)
    assert torch.allclose(nq, torch.ones_like(nq), atol=1e-6)
    assert torch.allclose(nk, torch.ones_like(nk), atol=1e-6)
    assert (d["beta"] > 0).all() and (d["beta"] < 1).all()
    assert (d["g"] < 0).all()
    assert d["cu_seqlens"].tolist() == [0, 100, 128]
    e = inputs.make_prefill([100, 28], 2, 4, 16, 8, dtype="f32", seed=5, state_std=0.02)
    for key in ("q", "k", "v", "g", "beta", "state_in"):
        assert torch.equal(d[key], e[key])
    s = d["state_in"].double()
    assert abs(s.std().item() - 0.02) < 0.002
    b = inputs.make_prefill([100, 28], 2, 4, 16, 8, dtype="bf16", seed=5)
    assert b["q"].dtype == torch.bfloat16 and b["g"].dtype == torch.float32
