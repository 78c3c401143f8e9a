"""Pins for the fp64 decode-attention oracle: values the definition fixes,
computed by routes other than its own (closed forms, invariances, a brute
force over each query head separately)."""
import numpy as np
import pytest

from oracle.attention import gqa_decode


def case(seed, B=2, h_q=8, h_kv=2, D=16, cap=12, lens=(12, 5)):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, h_q, D))
    k = r.standard_normal((B, h_kv, cap, D))
    v = r.standard_normal((B, h_kv, cap, D))
    return q, k, v, np.array(lens)


def test_single_key_returns_its_value():
    q, k, v, _ = case(1, lens=(1, 1))
    o = gqa_decode(q, k, v, [1, 1], 0.3)
    for b in range(2):
        for h in range(8):
            assert np.allclose(o[b, h], v[b, h // 4, 0], atol=1e-15)


def test_zero_query_averages_the_values():
    q, k, v, lens = case(2)
    o = gqa_decode(np.zeros_like(q), k, v, lens, 1.0)
    for b in range(2):
        for h in range(8):
            assert np.allclose(o[b, h], v[b, h // 4, :lens[b]].mean(0), atol=1e-13)


def test_dominant_key_and_shift_invariance():
    q, k, v, lens = case(3)
    # a key aligned with q and a large scale: the output is that key's value
    k2 = k.copy()
    k2[0, 0, 3] = q[0, 1] * 10
    o = gqa_decode(q, k2, v, lens, 50.0)
    assert np.allclose(o[0, 1], v[0, 0, 3], atol=1e-9)
    # adding the same vector to every key leaves each head's weights unchanged
    # only if q . vector is constant per head: shift keys by a vector orthogonal to q
    o_ref = gqa_decode(q, k, v, lens, 0.7)
    qh = q[1, 5]
    d = np.random.default_rng(4).standard_normal(16)
    d -= qh * (d @ qh) / (qh @ qh)
    k3 = k.copy()
    k3[1, 1, :lens[1]] += d
    o3 = gqa_decode(q, k3, v, lens, 0.7)
    assert np.allclose(o3[1, 5], o_ref[1, 5], atol=1e-13)


def test_permutation_of_cached_tokens():
    q, k, v, lens = case(5)
    p = np.random.default_rng(6).permutation(lens[0])
    k2, v2 = k.copy(), v.copy()
    k2[0, :, :lens[0]] = k[0][:, p]
    v2[0, :, :lens[0]] = v[0][:, p]
    assert np.allclose(gqa_decode(q, k2, v2, lens, 0.5), gqa_decode(q, k, v, lens, 0.5),
                       atol=1e-13)


def test_brute_force_per_head_and_head_map():
    """Each head by an explicit loop over keys, including the grouped head map and
    the cache slots past the sequence length (which must not be read)."""
    q, k, v, lens = case(7, h_q=6, h_kv=3)
    k[:, :, 6:] = np.nan  # never read for sequence 1 (L = 5)
    k[0] = np.nan_to_num(k[0])
    o = gqa_decode(q, k, v, lens, 0.9)
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
