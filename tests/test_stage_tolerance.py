"""Where the intermediate-stage tolerance of the GPU parity tests comes from
(parity.BF16_STAGE_MAX_ABS_REL_RMS = 8e-2), reproduced on the CPU.

A numpy emulation of every rounding point of the bf16 layer's kernels (the
fp16 intermediates and packed weights, fp32 accumulation, the softmax
exponent and probabilities in fp16 with their sum in fp32 (the kernel's
fp16 partial sums of eight values are taken exactly here), the scaled fp16
copies of h and act,
the bf16 output) runs on the same seeded inputs as the fp64 oracle.  Its
stage errors are what a correct implementation of that rounding scheme
shows: the attention output's largest error is a few percent of its RMS
(it inherits the softmax's sensitivity to the rounding of q and k), above
the 2e-2 bound of the layer output, while its mean relative error stays far
below 5e-3.  The test asserts that the emulated maxima sit at least a
factor 1.5 under the stage bound, and that the emulated layer output meets
the layer bounds (so the emulation is a faithful stand-in for the kernels).
"""

import math

import numpy as np
import pytest

import oracle
from llama_decoder_layer_prologue_b300 import synth

from parity import BF16_MAX_ABS_REL_RMS, BF16_MEAN_REL, BF16_STAGE_MAX_ABS_REL_RMS, weights_f64


def f16(a):
    return np.asarray(a, dtype=np.float32).astype(np.float16).astype(np.float64)


def f32(a):
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def bf16(a):
    return synth.to_f64(synth.bf16_round_bits(np.asarray(a, dtype=np.float32)))


def emulate(inp):
    """The bf16 layer with the kernels' rounding points (see the module
    docstring); returns the stages the GPU tests compare."""
    s = inp.workload.shape
    x = synth.to_f64(inp.x)
    w = weights_f64(inp.weights)
    T, H, d = x.shape[0], s.hidden, s.head_dim
    n_rep = s.n_heads // s.n_kv_heads
    r1 = f32(1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + s.rms_eps))
    xn = f16(x * r1)
    qkv = f32(xn @ f16(w.w_qkv * w.g_in).T)
    qs, ks = s.q_size, s.kv_size
    q = qkv[:, :qs].reshape(T, s.n_heads, d)
    k = qkv[:, qs:qs + ks].reshape(T, s.n_kv_heads, d)
    v = f16(qkv[:, qs + ks:].reshape(T, s.n_kv_heads, d))
    inv = oracle.layer_inv_freq(s)
    ang = np.outer(inp.positions.astype(np.float64), inv)
    c, sn = f32(np.cos(ang))[:, None, :], f32(np.sin(ang))[:, None, :]

    def rope(a):
        a1, a2 = a[..., : d // 2], a[..., d // 2:]
        return f16(np.concatenate([f32(a1 * c - a2 * sn), f32(a2 * c + a1 * sn)], axis=-1))

    q, k = rope(q), rope(k)
    scale = math.log2(math.e) / math.sqrt(d)
    attn = np.zeros((T, s.n_heads, d))
    for a0, a1 in zip(inp.cu_seqlens[:-1], inp.cu_seqlens[1:]):
        L = a1 - a0
        mask = np.triu(np.full((L, L), -np.inf), k=1)
        for hh in range(s.n_heads):
            kv = hh // n_rep
            sc = f32(q[a0:a1, hh] @ k[a0:a1, kv].T) * scale + mask
            # the packed exp2: exponent and result in fp16, the row sum
            # taken from the same fp16 values
            p16 = f16(np.exp2(f16(sc - sc.max(axis=1, keepdims=True))))
            l = p16.sum(axis=1, keepdims=True)
            attn[a0:a1, hh] = f32(p16 @ v[a0:a1, kv]) / l
    attn = f16(attn.reshape(T, -1))
    h = x + f32(attn @ f16(w.w_o).T)
    hg = f16(h / 256.0) * 256.0
    r2 = f32(1.0 / np.sqrt(np.sum(h * h, axis=1, keepdims=True) / H + s.rms_eps))
    gu = r2 * f32(hg @ f16(w.w_gate_up * w.g_post).T)
    I = s.intermediate
    g, u = gu[:, :I], gu[:, I:]
    act = f16(g / (1.0 + np.exp(-g)) * u / 16.0) * 16.0
    out = bf16(hg + f32(act @ f16(w.w_down).T))
    qkv_r = np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], axis=1)
    return dict(qkv=qkv_r, attn=attn, h=hg, act=act, out=out)


def err(got, ref):
    diff = np.abs(got - ref)
    rms = math.sqrt(float(np.mean(ref * ref)))
    return float(diff.max()) / rms, float(diff.sum() / np.abs(ref).sum())


@pytest.mark.parametrize("name,s,kw", [
    ("d64_gqa4", synth.LayerShape(hidden=512, n_heads=8, n_kv_heads=2, head_dim=64,
                                  intermediate=1024, rms_eps=1e-5, rope_base=500000.0,
                                  rope_scaling=1, rope_factor=32.0, max_position=4096),
     dict(batch=2, seq=384)),
    ("d128_gqa4", synth.LayerShape(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128,
                                   intermediate=1024, rms_eps=1e-5, rope_base=500000.0,
                                   rope_scaling=1, rope_factor=8.0, max_position=4096),
     dict(batch=1, seq=512)),
])
def test_emulated_rounding_sits_inside_the_stage_bound(name, s, kw):
    inp = synth.make_inputs(synth.custom_workload(name, s, "padded", index=400, **kw))
    em = emulate(inp)
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights), s,
                               inp.positions, inp.cu_seqlens)
    T = inp.tokens
    refs = dict(qkv=np.concatenate([ref["q"].reshape(T, -1), ref["k"].reshape(T, -1),
                                    ref["v"].reshape(T, -1)], axis=1),
                attn=ref["attn"], h=ref["h"], act=ref["act"], out=ref["out"])
    found = {k: err(em[k], refs[k]) for k in refs}
    for k, (mx, mean) in found.items():
        print(f"[emulated] {name} {k}: max_abs/rms={mx:.4g} mean_rel={mean:.4g}")
    mx, mean = found["out"]
    assert mx <= BF16_MAX_ABS_REL_RMS and mean <= BF16_MEAN_REL
    for k in ("qkv", "attn", "h", "act"):
        mx, mean = found[k]
        assert mx * 1.5 <= BF16_STAGE_MAX_ABS_REL_RMS, (k, mx)
        assert mean <= BF16_MEAN_REL, (k, mean)


def test_long_sequences_push_attention_past_the_layer_bound():
    """With 4096-token sequences (head_dim 128, 16 / 4 heads) the emulated
    attention output's largest error passes the layer output's 2e-2 * RMS
    (the GPU shows the same on the 8B-shaped workloads: 2.6 % for 2 x 4096,
    3.7 % for the varlen pack), while its mean relative error stays at
    5e-4: the stage bound has to sit above 2e-2, and 8e-2 keeps a margin of
    more than 1.5 over what the rounding scheme itself produces."""
    s = synth.LayerShape(hidden=1024, n_heads=16, n_kv_heads=4, head_dim=128,
                         intermediate=1024, rms_eps=1e-5, rope_base=500000.0,
                         rope_scaling=1, rope_factor=8.0, max_position=8192)
    inp = synth.make_inputs(synth.custom_workload("long", s, "padded", index=401,
                                                  batch=1, seq=4096))
    em = emulate(inp)
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights), s,
                               inp.positions, inp.cu_seqlens)
    mx, mean = err(em["attn"], ref["attn"])
    print(f"[emulated] long attn: max_abs/rms={mx:.4g} mean_rel={mean:.4g}")
    assert mx > BF16_MAX_ABS_REL_RMS
    assert mx * 1.5 <= BF16_STAGE_MAX_ABS_REL_RMS
    assert mean <= BF16_MEAN_REL
    omx, omean = err(em["out"], ref["out"])
    assert omx <= BF16_MAX_ABS_REL_RMS and omean <= BF16_MEAN_REL
