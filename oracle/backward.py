"""Backward pass of the decoder layer in plain numpy float64: the gradients of
a loss L with respect to the layer's input and weights, given dL/d(out).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages train these layers (the nanotron tutorial ch. 9 and the verl
parallel attention are training frameworks); they print the forward only, so
every step below is the chain rule applied to the forward of ``layer.py``,
taken in reverse order of the forward's steps:

  out = h + act W_down^T,        act = silu(gate) * up,
  [gate | up] = hn W_gate_up^T,  hn = RMSNorm(h) g_post,
  h = x + attn W_o^T,            attn = softmax(q' k'^T / sqrt(d) + mask) v,
  q', k' = RoPE(q, k),           [q | k | v] = xn W_qkv^T,  xn = RMSNorm(x) g_in.

Facts used (each a one-line derivation):
  * RMSNorm y = a * r * g with r = (mean(a^2) + eps)^(-1/2):
    dg = sum over rows of dy * a * r;
    da = r * (dy * g) - a * r^3 * mean((dy * g) * a)   (per row).
  * RoPE y = a cos + rotate_half(a) sin with rotate_half(a) = [-a2, a1]; the
    transpose of rotate_half is b -> [b2, -b1], so
    da = dy cos + [ (dy sin)_2, -(dy sin)_1 ].
  * softmax rows: dS = P * (dP - rowsum(dP * P)).
  * silu(z) = z s(z) with s the logistic function: silu'(z) = s (1 + z (1 - s)).
  * repeat_kv: a kv head's gradient is the sum over its n_rep query heads.
"""

from __future__ import annotations

import math

import numpy as np

from .layer import (_split_qkv, apply_rope, layer_inv_freq, repeat_kv, rms_norm,
                    rope_cos_sin)


def rms_norm_backward(a: np.ndarray, g: np.ndarray, eps: float, dy: np.ndarray):
    """(da, dg) of y = a / sqrt(mean(a^2) + eps) * g, per row."""
    r = 1.0 / np.sqrt(np.mean(a * a, axis=-1, keepdims=True) + eps)
    dyg = dy * g
    da = r * dyg - a * r ** 3 * np.mean(dyg * a, axis=-1, keepdims=True)
    dg = np.sum(dy * a * r, axis=0)
    return da, dg


def rope_backward(dy: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """da of y = a cos + rotate_half(a) sin; dy [T, heads, d], cos / sin [T, d]."""
    c, s = cos[:, None, :], sin[:, None, :]
    z = dy * s
    half = dy.shape[-1] // 2
    return dy * c + np.concatenate([z[..., half:], -z[..., :half]], axis=-1)


def silu_grad(z: np.ndarray) -> np.ndarray:
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def decoder_layer_backward(x: np.ndarray, w, cfg, positions: np.ndarray,
                           cu_seqlens: np.ndarray, dout: np.ndarray) -> dict:
    """Gradients of the prefill layer (padded or packed sequences).

    x, dout [T, hidden] float64; ``w`` as decoder_layer takes.  Returns dx
    and dw_qkv, dw_o, dw_gate_up, dw_down, dg_in, dg_post (the shapes of the
    inputs they belong to).
    """
    T = x.shape[0]
    d = cfg.head_dim
    n_rep = cfg.n_heads // cfg.n_kv_heads
    I = w.w_down.shape[1]
    # ---- forward, keeping what the backward reads
    xn = rms_norm(x, w.g_in, cfg.rms_eps)
    qkv = xn @ w.w_qkv.T
    q, k, v = _split_qkv(qkv, cfg)
    cos, sin = rope_cos_sin(positions, layer_inv_freq(cfg))
    qr, kr = apply_rope(q, cos, sin), apply_rope(k, cos, sin)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    probs = []  # per sequence: P [heads, L, L]
    attn = np.zeros((T, cfg.n_heads, d))
    for a, b in zip(cu[:-1], cu[1:]):
        L = b - a
        K, V = repeat_kv(kr[a:b], n_rep), repeat_kv(v[a:b], n_rep)
        S = np.einsum("thd,uhd->htu", qr[a:b], K) / math.sqrt(d)
        S = S + np.triu(np.full((L, L), -np.inf), k=1)[None]
        S = S - S.max(axis=-1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=-1, keepdims=True)
        probs.append(P)
        attn[a:b] = np.einsum("htu,uhd->thd", P, V)
    attn2 = attn.reshape(T, -1)
    h = x + attn2 @ w.w_o.T
    hn = rms_norm(h, w.g_post, cfg.rms_eps)
    gu = hn @ w.w_gate_up.T
    gate, up = gu[:, :I], gu[:, I:]
    sg = gate / (1.0 + np.exp(-gate))
    act = sg * up

    # ---- backward
    dw_down = dout.T @ act
    dact = dout @ w.w_down
    dgate = dact * up * silu_grad(gate)
    dup = dact * sg
    dgu = np.concatenate([dgate, dup], axis=1)
    dw_gate_up = dgu.T @ hn
    dhn = dgu @ w.w_gate_up
    dh_norm, dg_post = rms_norm_backward(h, w.g_post, cfg.rms_eps, dhn)
    dh = dout + dh_norm
    dw_o = dh.T @ attn2
    dattn = (dh @ w.w_o).reshape(T, cfg.n_heads, d)
    dqr = np.zeros_like(qr)
    dkr = np.zeros_like(kr)
    dv = np.zeros_like(v)
    for (a, b), P in zip(zip(cu[:-1], cu[1:]), probs):
        K, V = repeat_kv(kr[a:b], n_rep), repeat_kv(v[a:b], n_rep)
        dO = dattn[a:b]
        dV = np.einsum("htu,thd->uhd", P, dO)
        dP = np.einsum("thd,uhd->htu", dO, V)
        dS = P * (dP - np.sum(dP * P, axis=-1, keepdims=True)) / math.sqrt(d)
        dqr[a:b] = np.einsum("htu,uhd->thd", dS, K)
        dK = np.einsum("htu,thd->uhd", dS, qr[a:b])
        # query heads g n_rep .. g n_rep + n_rep - 1 read kv head g
        L = b - a
        dkr[a:b] = dK.reshape(L, cfg.n_kv_heads, n_rep, d).sum(axis=2)
        dv[a:b] = dV.reshape(L, cfg.n_kv_heads, n_rep, d).sum(axis=2)
    dq = rope_backward(dqr, cos, sin)
    dk = rope_backward(dkr, cos, sin)
    dqkv = np.concatenate([dq.reshape(T, -1), dk.reshape(T, -1), dv.reshape(T, -1)],
                          axis=1)
    dw_qkv = dqkv.T @ xn
    dxn = dqkv @ w.w_qkv
    dx_norm, dg_in = rms_norm_backward(x, w.g_in, cfg.rms_eps, dxn)
    dx = dh + dx_norm
    return dict(dx=dx, dw_qkv=dw_qkv, dw_o=dw_o, dw_gate_up=dw_gate_up,
                dw_down=dw_down, dg_in=dg_in, dg_post=dg_post)
