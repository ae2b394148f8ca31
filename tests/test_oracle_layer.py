"""Pins for the oracle's MLP, the whole layer, varlen and decode (CPU only)."""

import os
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from llama_decoder_layer_prologue_b300 import synth

RNG = np.random.default_rng(3)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

SMALL = synth.LayerShape(hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                         intermediate=96, rms_eps=1e-5, rope_base=10000.0,
                         rope_scaling=0, max_position=64, dtype="fp32")
SMALL_L3 = synth.LayerShape(hidden=64, n_heads=8, n_kv_heads=2, head_dim=16,
                            intermediate=80, rms_eps=1e-5, rope_base=5e5,
                            rope_scaling=1, rope_factor=8.0, max_position=64,
                            dtype="fp32")


def weights(cfg, scale=0.1):
    r = lambda *s: RNG.standard_normal(s) * scale
    return types.SimpleNamespace(
        w_qkv=r(cfg.n_qkv, cfg.hidden), w_o=r(cfg.hidden, cfg.q_size),
        w_gate_up=r(2 * cfg.intermediate, cfg.hidden),
        w_down=r(cfg.hidden, cfg.intermediate),
        g_in=1 + r(cfg.hidden), g_post=1 + r(cfg.hidden))


def padded(B, S):
    return (np.tile(np.arange(S), B), np.arange(0, B * S + 1, S))


# ----------------------------------------------------------------- MLP
def pin_swiglu(mlp_fn):
    hn = RNG.standard_normal((5, 12))
    wg, wu = RNG.standard_normal((7, 12)), RNG.standard_normal((7, 12))
    wd = RNG.standard_normal((12, 7))
    act, out = mlp_fn(hn, np.concatenate([wg, wu]), wd)
    t = torch.from_numpy
    # the HF module's separate gate_proj / up_proj / down_proj linears
    ref = F.linear(F.silu(F.linear(t(hn), t(wg))) * F.linear(t(hn), t(wu)),
                   t(wd))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_swiglu_matches_separate_linears():
    pin_swiglu(oracle.swiglu_mlp)


def test_swiglu_catches_swapped_halves():
    def mutant(hn, w, wd):
        n = w.shape[0] // 2
        return oracle.swiglu_mlp(hn, np.concatenate([w[n:], w[:n]]), wd)
    with pytest.raises(AssertionError):
        pin_swiglu(mutant)


def test_silu():
    x = np.linspace(-30, 30, 1001)
    assert oracle.silu(np.zeros(1))[0] == 0.0
    np.testing.assert_allclose(oracle.silu(x), F.silu(torch.from_numpy(x)),
                               rtol=1e-14, atol=1e-300)


# ----------------------------------------------------------------- layer
def torch_layer(x, w, cfg, pos, cu):
    """The layer composed from torch fp64 library routines; RoPE in the
    complex (polar) form on interleaved pairs."""
    t = torch.from_numpy
    d, hq, hkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    xt = t(x)
    xn = F.rms_norm(xt, (cfg.hidden,), t(w.g_in), cfg.rms_eps)
    qkv = F.linear(xn, t(w.w_qkv))
    q = qkv[:, : hq * d].reshape(-1, hq, d)
    k = qkv[:, hq * d:(hq + hkv) * d].reshape(-1, hkv, d)
    v = qkv[:, (hq + hkv) * d:].reshape(-1, hkv, d)
    f = t(oracle.layer_inv_freq(cfg))
    cis = torch.polar(torch.ones(len(pos), d // 2, dtype=torch.float64),
                      torch.outer(t(pos.astype(np.float64)), f))[:, None]

    def rot(z):
        zc = torch.complex(z[..., : d // 2], z[..., d // 2:]) * cis
        return torch.cat([zc.real, zc.imag], dim=-1)

    q, k = rot(q), rot(k)
    o = torch.zeros_like(q)
    for a, b in zip(cu[:-1], cu[1:]):
        tr = lambda z: z[a:b].transpose(0, 1)[None]
        o[a:b] = F.scaled_dot_product_attention(
            tr(q), tr(k), tr(v), is_causal=True,
            enable_gqa=True)[0].transpose(0, 1)
    h = xt + F.linear(o.reshape(len(x), -1), t(w.w_o))
    hn = F.rms_norm(h, (cfg.hidden,), t(w.g_post), cfg.rms_eps)
    g, u = F.linear(hn, t(w.w_gate_up)).chunk(2, dim=-1)
    return (h + F.linear(F.silu(g) * u, t(w.w_down))).numpy()


@pytest.mark.parametrize("cfg", [SMALL, SMALL_L3])
def test_layer_matches_torch_composition(cfg):
    w = weights(cfg)
    x = RNG.standard_normal((3 * 9, cfg.hidden))
    pos, cu = padded(3, 9)
    got = oracle.decoder_layer(x, w, cfg, pos, cu)["out"]
    np.testing.assert_allclose(got, torch_layer(x, w, cfg, pos, cu),
                               rtol=1e-11, atol=1e-12)


def test_zero_projections_give_identity():
    w = weights(SMALL)
    w.w_o[:] = 0.0
    w.w_down[:] = 0.0
    x = RNG.standard_normal((8, SMALL.hidden))
    pos, cu = padded(1, 8)
    np.testing.assert_array_equal(
        oracle.decoder_layer(x, w, SMALL, pos, cu)["out"], x)


def test_varlen_equals_separate_padded_runs():
    w = weights(SMALL_L3)
    lens = [5, 1, 12, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    x = RNG.standard_normal((cu[-1], SMALL_L3.hidden))
    packed = oracle.decoder_layer(x, w, SMALL_L3, pos, cu)["out"]
    for a, b in zip(cu[:-1], cu[1:]):
        alone = oracle.decoder_layer(x[a:b], w, SMALL_L3, np.arange(b - a),
                                     np.array([0, b - a]))["out"]
        np.testing.assert_allclose(packed[a:b], alone, rtol=1e-13, atol=1e-13)


def test_selected_rows_equal_full_layer():
    w = weights(SMALL_L3)
    lens = [7, 1, 10]
    cu = np.concatenate([[0], np.cumsum(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    x = RNG.standard_normal((cu[-1], SMALL_L3.hidden))
    full = oracle.decoder_layer(x, w, SMALL_L3, pos, cu)
    rows = np.array([17, 0, 7, 6, 9, 3])
    part = oracle.decoder_layer_rows(x, w, SMALL_L3, pos, cu, rows)
    for key in ("attn", "h", "act", "out"):
        np.testing.assert_allclose(part[key], full[key][rows], rtol=1e-12,
                                   atol=1e-13)


def test_decode_equals_last_row_of_prefill():
    """Cache rows built from the prefill's own rotated k and v; the decoded
    token must reproduce the prefill's output row at that position."""
    cfg = SMALL_L3
    w = weights(cfg)
    lens = [9, 4, 1]
    B = len(lens)
    seqs = [RNG.standard_normal((L + 1, cfg.hidden)) for L in lens]
    pre = [oracle.decoder_layer(s, w, cfg, np.arange(len(s)),
                                np.array([0, len(s)])) for s in seqs]
    cache = lambda b, n: (pre[b]["k"][:n], pre[b]["v"][:n])
    x_new = np.stack([s[-1] for s in seqs])
    dec = oracle.decoder_layer_decode(x_new, w, cfg, cache, np.array(lens))
    for b in range(B):
        np.testing.assert_allclose(dec["out"][b], pre[b]["out"][-1],
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dec["k_new"][b], pre[b]["k"][-1],
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dec["v_new"][b], pre[b]["v"][-1],
                                   rtol=1e-12, atol=1e-13)


def test_cached_chunk_equals_the_rest_of_a_prefill():
    """A sequence split into a cached prefix (rotated k / v from the prefill
    of the whole sequence) and a chunk of S new tokens: the chunk must
    reproduce the prefill's rows and new cache rows after the prefix."""
    cfg = SMALL_L3
    w = weights(cfg)
    S = 5
    prefix = [9, 0, 3, 14]
    seqs = [RNG.standard_normal((p + S, cfg.hidden)) for p in prefix]
    pre = [oracle.decoder_layer(s, w, cfg, np.arange(len(s)),
                                np.array([0, len(s)])) for s in seqs]
    cache = lambda b, n: (pre[b]["k"][:n], pre[b]["v"][:n])
    x_new = np.concatenate([s[-S:] for s in seqs])
    got = oracle.decoder_layer_cached(x_new, w, cfg, cache, np.array(prefix), S)
    for b, p in enumerate(prefix):
        rows = slice(b * S, (b + 1) * S)
        np.testing.assert_allclose(got["out"][rows], pre[b]["out"][p:],
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got["k_new"][rows], pre[b]["k"][p:],
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(got["v_new"][rows], pre[b]["v"][p:],
                                   rtol=1e-12, atol=1e-13)


def test_cached_chunk_of_one_token_is_decode():
    cfg = SMALL_L3
    w = weights(cfg)
    sp = np.array([3, 0, 11])
    cache_k = [RNG.standard_normal((n, cfg.n_kv_heads, cfg.head_dim)) for n in sp]
    cache_v = [RNG.standard_normal((n, cfg.n_kv_heads, cfg.head_dim)) for n in sp]
    cache = lambda b, n: (cache_k[b][:n], cache_v[b][:n])
    x = RNG.standard_normal((len(sp), cfg.hidden))
    a = oracle.decoder_layer_cached(x, w, cfg, cache, sp, 1)
    b = oracle.decoder_layer_decode(x, w, cfg, cache, sp)
    for key in ("out", "attn", "k_new", "v_new"):
        np.testing.assert_allclose(a[key], b[key], rtol=1e-13, atol=1e-14)


def test_cached_chunk_with_empty_cache_is_prefill():
    cfg = SMALL
    w = weights(cfg)
    B, S = 3, 6
    x = RNG.standard_normal((B * S, cfg.hidden))
    empty = lambda b, n: (np.zeros((0, cfg.n_kv_heads, cfg.head_dim)),) * 2
    a = oracle.decoder_layer_cached(x, w, cfg, empty, np.zeros(B, np.int64), S)
    pos = np.tile(np.arange(S), B)
    ref = oracle.decoder_layer(x, w, cfg, pos, np.arange(0, B * S + 1, S))
    np.testing.assert_allclose(a["out"], ref["out"], rtol=1e-12, atol=1e-12)


def test_cached_chunk_is_causal_within_the_chunk():
    # changing the last new token leaves every earlier token's output exactly
    # as it was (row i sees the prefix and new rows 0 .. i only)
    cfg = SMALL_L3
    w = weights(cfg)
    S, sp = 4, np.array([6])
    ck = RNG.standard_normal((6, cfg.n_kv_heads, cfg.head_dim))
    cv = RNG.standard_normal((6, cfg.n_kv_heads, cfg.head_dim))
    cache = lambda b, n: (ck[:n], cv[:n])
    x = RNG.standard_normal((S, cfg.hidden))
    y = x.copy()
    y[-1] += 1.0
    a = oracle.decoder_layer_cached(x, w, cfg, cache, sp, S)["out"]
    b = oracle.decoder_layer_cached(y, w, cfg, cache, sp, S)["out"]
    np.testing.assert_array_equal(a[:-1], b[:-1])
    assert not np.allclose(a[-1], b[-1])


def test_model_stack_hands_each_layer_the_previous_output():
    """A layer with zero o_proj and down_proj weights returns its input
    exactly (both residual branches add zero), so inserting one before or
    after a real layer must leave the logits unchanged bit for bit."""
    import types
    cfg = SMALL_L3
    w = weights(cfg)
    ident = types.SimpleNamespace(**vars(w))
    ident.w_o = np.zeros_like(w.w_o)
    ident.w_down = np.zeros_like(w.w_down)
    lens = [6, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    x = RNG.standard_normal((cu[-1], cfg.hidden))
    g = 1.0 + 0.1 * RNG.standard_normal(cfg.hidden)
    w_lm = 0.02 * RNG.standard_normal((64, cfg.hidden))
    one = oracle.model_forward(x, [w], cfg, pos, cu, g, w_lm)
    for stack in ([ident, w], [w, ident], [ident, w, ident]):
        got = oracle.model_forward(x, stack, cfg, pos, cu, g, w_lm)
        np.testing.assert_array_equal(got["logits"], one["logits"])
    np.testing.assert_array_equal(
        one["hidden"], oracle.decoder_layer(x, w, cfg, pos, cu)["out"])
    two = oracle.model_forward(x, [w, w], cfg, pos, cu, g, w_lm)
    assert not np.allclose(two["logits"], one["logits"])


# ----------------------------------------------------------------- shapes
def test_1b_shapes_match_page_printout():
    rows = {}
    with open(os.path.join(GOLDEN, "llama32_1b_decoder_layer.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, i, o = line.split()
                rows[name] = (int(i), int(o))
    s = synth.WORKLOADS["1b"].shape
    H, qs, kvs, I = s.hidden, s.q_size, s.kv_size, s.intermediate
    assert rows["q_proj"] == (H, qs)
    assert rows["k_proj"] == (H, kvs) and rows["v_proj"] == (H, kvs)
    assert rows["o_proj"] == (qs, H)
    assert rows["gate_proj"] == (H, I) and rows["up_proj"] == (H, I)
    assert rows["down_proj"] == (I, H)
    assert rows["input_layernorm"][0] == H
    n_linear = sum(i * o for k, (i, o) in rows.items() if k.endswith("proj"))
    fused = s.n_qkv * H + H * qs + 2 * I * H + I * H
    assert n_linear == fused == 60_817_408


def test_workload_inputs_are_reproducible():
    a = synth.make_inputs("tiny")
    b = synth.make_inputs("tiny")
    np.testing.assert_array_equal(a.x, b.x)
    np.testing.assert_array_equal(a.weights.w_down, b.weights.w_down)
    assert a.x.dtype == np.float32 and a.x.shape == (64, 256)
    v = synth.make_inputs(synth.custom_workload(
        "v", synth.WORKLOADS["varlen"].shape, "varlen", total_tokens=5000),
        x_only=True)
    lens = np.diff(v.cu_seqlens)
    assert v.cu_seqlens[-1] == 5000 and np.all(lens[:-1] >= 128)
    assert np.all(lens <= 1024) and lens[-1] >= 1
    assert np.all(v.positions == np.concatenate([np.arange(L) for L in lens]))
