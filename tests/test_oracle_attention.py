"""Pins for the fp64 decode-attention oracle: values the definition fixes,
computed by routes other than its own (closed forms, invariances, a brute
force over each query head separately).  Each pin takes the attention function
as an argument, so that the same pins are also run against copies of the oracle
with one planted mistake each, every one of which must fail at least one pin."""
import numpy as np
import pytest

from oracle.attention import gqa_decode


def case(seed, B=2, h_q=8, h_kv=2, D=16, cap=12, lens=(12, 5)):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, h_q, D))
    k = r.standard_normal((B, h_kv, cap, D))
    v = r.standard_normal((B, h_kv, cap, D))
    return q, k, v, np.array(lens)


def pin_single_key_returns_its_value(att):
    q, k, v, _ = case(1, lens=(1, 1))
    o = att(q, k, v, [1, 1], 0.3)
    for b in range(2):
        for h in range(8):
            assert np.allclose(o[b, h], v[b, h // 4, 0], atol=1e-15)


def pin_zero_query_averages_the_values(att):
    q, k, v, lens = case(2)
    o = att(np.zeros_like(q), k, v, lens, 1.0)
    for b in range(2):
        for h in range(8):
            assert np.allclose(o[b, h], v[b, h // 4, :lens[b]].mean(0), atol=1e-13)


def pin_dominant_key_and_shift_invariance(att):
    q, k, v, lens = case(3)
    # a key aligned with q and a large scale: the output is that key's value
    k2 = k.copy()
    k2[0, 0, 3] = q[0, 1] * 10
    o = att(q, k2, v, lens, 50.0)
    assert np.allclose(o[0, 1], v[0, 0, 3], atol=1e-9)
    # shifting every key by a vector orthogonal to q leaves that head unchanged
    o_ref = att(q, k, v, lens, 0.7)
    qh = q[1, 5]
    d = np.random.default_rng(4).standard_normal(16)
    d -= qh * (d @ qh) / (qh @ qh)
    k3 = k.copy()
    k3[1, 1, :lens[1]] += d
    o3 = att(q, k3, v, lens, 0.7)
    assert np.allclose(o3[1, 5], o_ref[1, 5], atol=1e-13)


def pin_permutation_of_cached_tokens(att):
    q, k, v, lens = case(5)
    p = np.random.default_rng(6).permutation(lens[0])
    k2, v2 = k.copy(), v.copy()
    k2[0, :, :lens[0]] = k[0][:, p]
    v2[0, :, :lens[0]] = v[0][:, p]
    assert np.allclose(att(q, k2, v2, lens, 0.5), att(q, k, v, lens, 0.5), atol=1e-13)


def pin_brute_force_per_head_and_head_map(att):
    """Each head by an explicit loop over keys, including the grouped head map and
    the cache slots past the sequence length (which must not be read)."""
    q, k, v, lens = case(7, h_q=6, h_kv=3)
    k[:, :, 6:] = np.nan  # never read for sequence 1 (L = 5)
    k[0] = np.nan_to_num(k[0])
    o = att(q, k, v, lens, 0.9)
    for b in range(2):
        for h in range(6):
            j = h // 2
            num, den = np.zeros(16), 0.0
            smax = max(0.9 * float(np.dot(q[b, h], k[b, j, i])) for i in range(lens[b]))
            for i in range(lens[b]):
                w = np.exp(0.9 * float(np.dot(q[b, h], k[b, j, i])) - smax)
                num += w * v[b, j, i]
                den += w
            assert np.allclose(o[b, h], num / den, atol=1e-13)


PINS = [pin_single_key_returns_its_value, pin_zero_query_averages_the_values,
        pin_dominant_key_and_shift_invariance, pin_permutation_of_cached_tokens,
        pin_brute_force_per_head_and_head_map]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(gqa_decode)


# ------------------------------------------------------------ planted mistakes
def _mutant(kind):
    """A copy of the oracle's loop with one mistake of the given kind."""
    def att(q, k, v, cache_len, scale):
        q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
        B, h_q, D = q.shape
        h_kv = k.shape[1]
        G = h_q // h_kv
        o = np.zeros((B, h_q, D))
        for b in range(B):
            L = int(cache_len[b])
            if kind == "whole_capacity":
                L = k.shape[2]
            if L == 0:
                continue
            for h in range(h_q):
                j = h % h_kv if kind == "head_map" else h // G
                sc = 1.0 if kind == "no_scale" else scale
                s = sc * (k[b, j, :L] @ q[b, h])
                w = np.exp(s - s.max())
                if kind != "unnormalised":
                    w = w / w.sum()
                vals = k if kind == "keys_as_values" else v
                o[b, h] = w @ vals[b, j, :L]
                if kind == "scaled_output":
                    o[b, h] *= scale
        return o
    return att


MUTANTS = ["no_scale", "head_map", "unnormalised", "whole_capacity", "keys_as_values",
           "scaled_output"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind):
    att = _mutant(kind)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(att)
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake {kind!r}"


def test_unmutated_copy_passes_every_pin():
    """The mutant template with no mistake planted passes all pins (so a failing
    pin above is caused by the planted mistake alone)."""
    att = _mutant("none")
    for pin in PINS:
        pin(att)
