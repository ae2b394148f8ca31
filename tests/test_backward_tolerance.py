"""Where the backward pass's tolerance comes from (tests/test_backward_gpu.py:
the bf16 layer output's bounds, max |gpu - oracle| <= 2e-2 * RMS and
sum|gpu - oracle| / sum|oracle| <= 5e-3, for every gradient, with dx allowed
its own rounding to bf16 on top), reproduced on the CPU.

A numpy emulation of every rounding point of llama_layer_backward (the
forward's fp16 recomputation, the fp16 copies of dL/d(out), d gate | d up,
dh, d attn, dz, P and dq | dk | dv, the softmax exponent in fp16, fp32
accumulation, the bf16 dx) runs on the inputs of the GPU test's 8B-shaped
case (2 x 256 tokens) next to the fp64 oracle; it reproduces the GPU's
figures (dx: 2.34 % of RMS at most, about 0.18 % mean relative).  Computed without any fp16 rounding, dx still shows the same
largest error: it is the bf16 rounding of one element seven RMS large (half
a bf16 spacing there is 2.3 % of RMS), which no implementation can avoid.
With that rounding allowed for (2^-8 |oracle| per element) every emulated
gradient sits well inside the bounds.
"""

import math

import numpy as np

import oracle
from oracle.backward import decoder_layer_backward
from llama_decoder_layer_prologue_b300 import synth

from parity import weights_f64
from test_stage_tolerance import bf16, err, f16, f32

GRADS = ("dx", "dw_qkv", "dw_o", "dw_gate_up", "dw_down", "dg_in", "dg_post")


def emulate_backward(inp, dout):
    """The gradients with the kernels' rounding points (see the module
    docstring)."""
    s = inp.workload.shape
    x = synth.to_f64(inp.x)
    w = weights_f64(inp.weights)
    T, H, d, I = x.shape[0], s.hidden, s.head_dim, s.intermediate
    Hq, Hkv = s.n_heads, s.n_kv_heads
    n_rep = Hq // Hkv
    qs, ks = s.q_size, s.kv_size
    # ---- forward recomputation
    r1 = f32(1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + s.rms_eps))
    xn = f16(x * r1)
    wqkv = f16(w.w_qkv * w.g_in)
    qkv = f32(xn @ wqkv.T)
    q = qkv[:, :qs].reshape(T, Hq, d)
    k = qkv[:, qs:qs + ks].reshape(T, Hkv, d)
    v = f16(qkv[:, qs + ks:].reshape(T, Hkv, d))
    ang = np.outer(inp.positions.astype(np.float64), oracle.layer_inv_freq(s))
    c, sn = f32(np.cos(ang))[:, None, :], f32(np.sin(ang))[:, None, :]
    half = d // 2

    def rope(a):
        a1, a2 = a[..., :half], a[..., half:]
        return f16(np.concatenate([f32(a1 * c - a2 * sn), f32(a2 * c + a1 * sn)], axis=-1))

    def rope_t(g):
        g1, g2 = g[..., :half], g[..., half:]
        return f16(np.concatenate([g1 * c + g2 * sn, g2 * c - g1 * sn], axis=-1))

    q, k = rope(q), rope(k)
    scale = math.log2(math.e) / math.sqrt(d)
    attn = np.zeros((T, Hq, d))
    lse = np.zeros((T, Hq))
    seqs = list(zip(inp.cu_seqlens[:-1], inp.cu_seqlens[1:]))
    for a0, a1 in seqs:
        L = a1 - a0
        mask = np.triu(np.full((L, L), -np.inf), k=1)
        for hh in range(Hq):
            sc = f32(q[a0:a1, hh] @ k[a0:a1, hh // n_rep].T) * scale + mask
            m = sc.max(axis=1, keepdims=True)
            p16 = f16(np.exp2(f16(sc - m)))
            l = p16.sum(axis=1, keepdims=True)
            attn[a0:a1, hh] = f32(p16 @ v[a0:a1, hh // n_rep]) / l
            lse[a0:a1, hh] = (m + np.log2(l))[:, 0]
    attn = f16(attn.reshape(T, -1))
    h = x + f32(attn @ f16(w.w_o).T)
    hg = f16(h / 256.0) * 256.0
    r2 = f32(1.0 / np.sqrt(np.sum(h * h, axis=1, keepdims=True) / H + s.rms_eps))
    wgu = f16(w.w_gate_up * w.g_post)
    gu = r2 * f32(hg @ wgu.T)
    g, u = f16(gu[:, :I]), f16(gu[:, I:])
    act = f16(g / (1.0 + np.exp(-g)) * u / 16.0) * 16.0
    # ---- backward
    do16 = f16(dout)
    dw_down = f32(do16.T @ act)
    dact = f32(do16 @ f16(w.w_down))
    sg = 1.0 / (1.0 + np.exp(-g))
    a = dact * r2
    dgu = np.concatenate([f16(a * u * sg * (1.0 + g * (1.0 - sg))), f16(a * g * sg)], axis=1)
    dwp = f32(dgu.T @ hg)
    dw_gate_up = dwp * w.g_post
    dg_post = np.sum(w.w_gate_up * dwp, axis=0)
    du2 = f32(dgu @ wgu)
    dot2 = np.sum(du2 * hg, axis=1, keepdims=True)
    dh = dout + du2 - hg * r2 * r2 * dot2 / H
    dh16 = f16(dh)
    dw_o = f32(dh16.T @ attn)
    do_a = f16(f32(dh16 @ f16(w.w_o))).reshape(T, Hq, d)
    D = np.sum(do_a * attn.reshape(T, Hq, d), axis=2)
    dq = np.zeros((T, Hq, d))
    dk = np.zeros((T, Hkv, d))
    dv = np.zeros((T, Hkv, d))
    for a0, a1 in seqs:
        L = a1 - a0
        mask = np.triu(np.full((L, L), -np.inf), k=1)
        for hh in range(Hq):
            g_ = hh // n_rep
            sc = f32(q[a0:a1, hh] @ k[a0:a1, g_].T) * scale + mask
            # P recomputed by the packed exp2 (exponent and result in fp16);
            # dz and dV's product take the same fp16 P
            p16 = f16(np.exp2(f16(f32(sc - lse[a0:a1, hh][:, None]))))
            dp = f32(do_a[a0:a1, hh] @ v[a0:a1, g_].T)
            dz = f16(p16 * f32(dp - D[a0:a1, hh][:, None]))
            dq[a0:a1, hh] = f32(dz @ k[a0:a1, g_]) / math.sqrt(d)
            dk[a0:a1, g_] += f32(dz.T @ q[a0:a1, hh]) / math.sqrt(d)
            dv[a0:a1, g_] += f32(p16.T @ do_a[a0:a1, hh])
    dqkv = np.concatenate([rope_t(dq).reshape(T, -1), rope_t(dk).reshape(T, -1),
                           f16(dv).reshape(T, -1)], axis=1)
    dwq = f32(dqkv.T @ xn)
    dw_qkv = dwq * w.g_in
    dg_in = np.sum(w.w_qkv * dwq, axis=0)
    du1 = f32(dqkv @ wqkv)
    dot1 = np.sum(du1 * x, axis=1, keepdims=True)
    dx = bf16(dh + r1 * du1 - x * r1 ** 3 * dot1 / H)
    return dict(dx=dx, dw_qkv=dw_qkv, dw_o=dw_o, dw_gate_up=dw_gate_up, dw_down=dw_down,
                dg_in=dg_in, dg_post=dg_post)


def test_emulated_backward_rounding_fits_the_backward_bound():
    """Every emulated gradient inside the bounds (dx after its own bf16
    rounding), with a margin of 1.5; dx's largest raw error past 2e-2 * RMS
    comes from the output rounding alone."""
    s = synth.WORKLOADS["8b"].shape
    inp = synth.make_inputs(synth.custom_workload("bwd_8b_short", s, "padded", index=301,
                                                  batch=2, seq=256))
    dout = synth.to_f64(synth.make_dout(inp))
    em = emulate_backward(inp, dout)
    ref = decoder_layer_backward(synth.to_f64(inp.x), weights_f64(inp.weights), s,
                                 inp.positions, inp.cu_seqlens, dout)
    for k_ in GRADS:
        mx, mean = err(em[k_], ref[k_])
        print(f"[emulated] backward {k_}: max_abs/rms={mx:.4g} mean_rel={mean:.4g}")
        assert mean * 1.5 <= 5e-3, (k_, mean)
        if k_ != "dx":
            assert mx * 1.5 <= 2e-2, (k_, mx)
    rms = math.sqrt(float(np.mean(ref["dx"] ** 2)))
    excess = np.abs(em["dx"] - ref["dx"]) - 2.0 ** -8 * np.abs(ref["dx"])
    assert excess.max() * 1.5 <= 2e-2 * rms
    # the exact dx, rounded to bf16 once, is as far off at its largest error
    rounded = bf16(ref["dx"])
    mx_exact, _ = err(rounded, ref["dx"])
    mx_em, _ = err(em["dx"], ref["dx"])
    print(f"[emulated] exact dx rounded to bf16: max_abs/rms={mx_exact:.4g}")
    assert mx_exact > 2e-2 and abs(mx_exact - mx_em) <= 0.1 * mx_em
