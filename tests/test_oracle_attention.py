"""Pins for the oracle's grouped-query causal attention (CPU only)."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.default_rng(11)


def _qkv(T, hq, hkv, d):
    return (RNG.standard_normal((T, hq, d)), RNG.standard_normal((T, hkv, d)),
            RNG.standard_normal((T, hkv, d)))


def _sdpa(q, k, v, cu):
    """torch fp64 SDPA per sequence, causal, GQA through enable_gqa."""
    out = np.zeros_like(q)
    for a, b in zip(cu[:-1], cu[1:]):
        t = lambda z: torch.from_numpy(z[a:b]).transpose(0, 1)[None]
        o = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True,
                                           enable_gqa=True)
        out[a:b] = o[0].transpose(0, 1).numpy()
    return out


def pin_attention_library(attn_fn):
    for hq, hkv, d, cu in ((4, 4, 16, [0, 9]), (8, 2, 32, [0, 5, 6, 19]),
                           (6, 3, 8, [0, 1, 2, 40])):
        q, k, v = _qkv(cu[-1], hq, hkv, d)
        np.testing.assert_allclose(attn_fn(q, k, v, np.array(cu)),
                                   _sdpa(q, k, v, cu), rtol=1e-11, atol=1e-12)


def test_attention_matches_torch_sdpa():
    pin_attention_library(oracle.causal_attention)


def test_attention_catches_wrong_group_mapping():
    def mutant(q, k, v, cu):
        n_rep = q.shape[1] // k.shape[1]
        # head h reads kv head h % Hkv instead of h // n_rep
        idx = np.arange(q.shape[1]) % k.shape[1]
        return oracle.causal_attention(q, k[:, idx], v[:, idx], cu) if n_rep \
            else None
    with pytest.raises(AssertionError):
        pin_attention_library(mutant)


def test_attention_catches_missing_scale():
    def mutant(q, k, v, cu):
        return oracle.causal_attention(q * math.sqrt(q.shape[-1]), k, v, cu)
    with pytest.raises(AssertionError):
        pin_attention_library(mutant)


def test_attention_brute_force_loops():
    T, hq, hkv, d = 7, 4, 2, 4
    q, k, v = _qkv(T, hq, hkv, d)
    cu = np.array([0, 3, 7])
    got = oracle.causal_attention(q, k, v, cu)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        for t in range(a, b):
            for h in range(hq):
                g = h // (hq // hkv)
                w = [math.exp(sum(q[t, h, i] * k[u, g, i] for i in range(d))
                              / math.sqrt(d)) for u in range(a, t + 1)]
                z = sum(w)
                for i in range(d):
                    o = sum(w[u - a] * v[u, g, i] for u in range(a, t + 1)) / z
                    assert abs(got[t, h, i] - o) < 1e-12


def test_zero_query_gives_running_mean():
    q, k, v = _qkv(12, 4, 2, 8)
    q[:] = 0.0
    cu = np.array([0, 5, 12])
    got = oracle.causal_attention(q, k, v, cu)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            want = v[a:t + 1].mean(axis=0)
            np.testing.assert_allclose(got[t, 0::2], want, rtol=1e-13)
            np.testing.assert_allclose(got[t, 1::2], want, rtol=1e-13)


def test_single_token_context_returns_value():
    q, k, v = _qkv(4, 4, 2, 8)
    got = oracle.causal_attention(q, k, v, np.array([0, 1, 2, 3, 4]))
    np.testing.assert_array_equal(got, oracle.repeat_kv(v, 2))


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v = _qkv(10, 8, 2, 8)
    cu = np.array([0, 10])
    gqa = oracle.causal_attention(q, k, v, cu)
    kk, vv = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    mha = oracle.causal_attention(q, kk, vv, cu)
    np.testing.assert_array_equal(gqa, mha)
    # and MHA itself against torch without enable_gqa
    t = lambda z: torch.from_numpy(z).transpose(0, 1)[None]
    ref = F.scaled_dot_product_attention(t(q), t(kk), t(vv), is_causal=True)
    np.testing.assert_allclose(mha, ref[0].transpose(0, 1).numpy(), rtol=1e-11,
                               atol=1e-12)


def test_causality_future_token_does_not_leak():
    q, k, v = _qkv(9, 4, 2, 8)
    cu = np.array([0, 9])
    base = oracle.causal_attention(q, k, v, cu)
    for t in range(8):
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[t + 1:] += 5.0
        k2[t + 1:] -= 3.0
        v2[t + 1:] *= -2.0
        got = oracle.causal_attention(q2, k2, v2, cu)
        np.testing.assert_array_equal(got[: t + 1], base[: t + 1])
        assert not np.array_equal(got[t + 1], base[t + 1])


def test_packed_sequences_are_independent():
    q, k, v = _qkv(15, 4, 1, 8)
    cu = np.array([0, 4, 11, 15])
    packed = oracle.causal_attention(q, k, v, cu)
    for a, b in zip(cu[:-1], cu[1:]):
        alone = oracle.causal_attention(q[a:b], k[a:b], v[a:b],
                                        np.array([0, b - a]))
        np.testing.assert_array_equal(packed[a:b], alone)
