"""The decoder layer in plain numpy float64, step by step as the pages give it.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pages cited (title, then the section or figure on it):
  [nanotron]  "模型层：从 Embedding 到 Loss 的实现" (nanotron tutorial ch. 9):
              9.3 CausalSelfAttention, 9.4 MLP (SwiGLU), 9.5 DecoderLayer.
  [verl]      "parallel_attention.py — LLaMA 并行注意力": 1 RoPE 旋转位置编码,
              2 ParallelLlamaAttention, 3 ParallelLlamaAttentionRmPad.
  [the7]      "llama3 结构详解": 3.1 RMSNorm (formula and Meta source),
              3.2 Attention (Meta Attention.forward with the KV cache).
  [csdn]      Llama-3 model.py walkthrough (un.csdn.net): "1. RMSNorm",
              "2. 旋转位置编码" (precompute_freqs_cis / apply_scaling),
              "3. 注意力机制" (KV cache), "4. 前馈网络", "5. Transformer"
              (causal mask).
  [nju]       NJU LLM course lecture 5: "LlamaDecoderLayer内部结构",
              "手搓RMSNorm", "RoPE高效实现", "SwiGLU模块".

Readings taken where the pages are silent or disagree:
  * eps sits inside the square root ([the7] Meta source, [nju] 手搓RMSNorm;
    the [the7] formula omits it).
  * RoPE pairs dimension i with i + d/2 (rotate_half, [nju]); the complex form
    of [csdn] pairs neighbours and equals this one after a permutation.
  * Llama3 frequency scaling: the pages only describe it (keep the high
    frequencies, divide the low ones by the factor, interpolate smoothly in
    between; [verl] 1, [csdn] 2).  Written out with wavelength 2*pi/f and the
    band edges original_max_pos / high_freq_factor and
    original_max_pos / low_freq_factor; inside the band the weight of the
    unscaled frequency is (original_max_pos / wavelength - low) / (high - low).
  * Query head h reads kv head h // n_rep (repeat_kv repeats each kv head
    n_rep times in a row).
  * q | k | v and gate | up are the row orders of the fused weights.
"""

from __future__ import annotations

import math

import numpy as np


# --------------------------------------------------------------------------
# RMSNorm  ([the7] 3.1 formula and Meta source; [nju] 手搓RMSNorm)
# --------------------------------------------------------------------------
def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """a_i / RMS(a) * g_i with RMS(a) = sqrt(mean(a^2) + eps), per row."""
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * g


# --------------------------------------------------------------------------
# RoPE  ([verl] 1; [csdn] 2; [nju] RoPE高效实现)
# --------------------------------------------------------------------------
def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """inv_freq_i = 1 / base^(2i/d), i = 0 .. d/2 - 1."""
    two_i = np.arange(0, head_dim, 2, dtype=np.float64)
    return 1.0 / (base ** (two_i / head_dim))


def llama3_scale_inv_freq(inv_freq: np.ndarray, factor: float,
                          low_freq_factor: float, high_freq_factor: float,
                          original_max_pos: int) -> np.ndarray:
    """Llama3 piecewise scaling: keep high, divide low, interpolate the middle."""
    wavelen = 2.0 * math.pi / inv_freq
    short_edge = original_max_pos / high_freq_factor  # below: keep
    long_edge = original_max_pos / low_freq_factor  # above: divide
    out = np.empty_like(inv_freq)
    for i, (f, lam) in enumerate(zip(inv_freq, wavelen)):
        if lam < short_edge:
            out[i] = f
        elif lam > long_edge:
            out[i] = f / factor
        else:
            s = (original_max_pos / lam - low_freq_factor) / (
                high_freq_factor - low_freq_factor)
            out[i] = (1.0 - s) * f / factor + s * f
    return out


def linear_scale_inv_freq(inv_freq: np.ndarray, factor: float) -> np.ndarray:
    """Linear position scaling ([verl] 1, LlamaLinearScalingRotaryEmbedding:
    t = t / scaling_factor): the angle (t / factor) * f_i is t * (f_i / factor),
    so every inverse frequency is divided by the factor."""
    return inv_freq / factor


def dynamic_ntk_base(base: float, head_dim: int, factor: float, table_len: int,
                     original_max_pos: int) -> float:
    """Dynamic NTK scaling ([verl] 1, LlamaDynamicNTKScalingRotaryEmbedding:
    the base is adjusted to the length).  The pages name the method only; the
    reading taken is the published NTK-aware rule for a table of table_len
    positions: beyond the original context the base becomes
    base * (factor * table_len / original_max_pos - (factor - 1)) ** (d / (d - 2)),
    which leaves the highest frequency (i = 0) as it is and divides the
    lowest (i = d/2 - 1) by exactly the bracketed scale; within the original
    context the base is unchanged."""
    if table_len <= original_max_pos:
        return base
    scale = factor * table_len / original_max_pos - (factor - 1.0)
    return base * scale ** (head_dim / (head_dim - 2.0))


def layer_inv_freq(cfg) -> np.ndarray:
    """The inverse frequencies a layer config asks for (rope_scaling 0: none,
    1: Llama3, 2: linear, 3: dynamic NTK for a table of max_position rows)."""
    base = cfg.rope_base
    if cfg.rope_scaling == 3:
        base = dynamic_ntk_base(base, cfg.head_dim, cfg.rope_factor,
                                cfg.max_position, cfg.rope_original_max_pos)
    f = rope_inv_freq(cfg.head_dim, base)
    if cfg.rope_scaling == 1:
        f = llama3_scale_inv_freq(f, cfg.rope_factor, cfg.rope_low_freq_factor,
                                  cfg.rope_high_freq_factor,
                                  cfg.rope_original_max_pos)
    elif cfg.rope_scaling == 2:
        f = linear_scale_inv_freq(f, cfg.rope_factor)
    return f


def rope_cos_sin(positions: np.ndarray, inv_freq: np.ndarray):
    """freqs = outer(t, inv_freq); emb = cat(freqs, freqs); cos / sin of emb."""
    freqs = np.outer(np.asarray(positions, dtype=np.float64), inv_freq)
    emb = np.concatenate([freqs, freqs], axis=-1)
    return np.cos(emb), np.sin(emb)


def rotate_half(x: np.ndarray) -> np.ndarray:
    """cat(-x2, x1) over the last axis, x1 / x2 its first / second half."""
    half = x.shape[-1] // 2
    return np.concatenate([-x[..., half:], x[..., :half]], axis=-1)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x [T, heads, d]; cos / sin [T, d]: x * cos + rotate_half(x) * sin."""
    return x * cos[:, None, :] + rotate_half(x) * sin[:, None, :]


# --------------------------------------------------------------------------
# Grouped-query causal attention
# ([verl] 2 steps 3-4, 3 varlen; [the7] 3.2; [csdn] 5 causal mask)
# --------------------------------------------------------------------------
def repeat_kv(kv: np.ndarray, n_rep: int) -> np.ndarray:
    """[T, Hkv, d] -> [T, Hkv * n_rep, d], kv head g repeated n_rep times."""
    return np.repeat(kv, n_rep, axis=1)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     cu_seqlens: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(d) + mask) v per sequence and head.

    q [T, Hq, d]; k, v [T, Hkv, d]; cu_seqlens [n+1] splits the T tokens into
    sequences; a token sees the tokens of its own sequence up to itself.
    Returns [T, Hq, d].
    """
    T, n_heads, d = q.shape
    n_rep = n_heads // k.shape[1]
    keys = repeat_kv(k, n_rep)
    values = repeat_kv(v, n_rep)
    out = np.zeros_like(q)
    for a, b in zip(cu_seqlens[:-1], cu_seqlens[1:]):
        a, b = int(a), int(b)
        if b == a:
            continue
        L = b - a
        mask = np.triu(np.full((L, L), -np.inf), k=1)
        for h in range(n_heads):
            scores = q[a:b, h] @ keys[a:b, h].T / math.sqrt(d) + mask
            scores = scores - scores.max(axis=-1, keepdims=True)
            p = np.exp(scores)
            p = p / p.sum(axis=-1, keepdims=True)
            out[a:b, h] = p @ values[a:b, h]
    return out


# --------------------------------------------------------------------------
# MLP  ([nanotron] 9.4; [csdn] 4; [nju] SwiGLU模块)
# --------------------------------------------------------------------------
def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x)."""
    return x / (1.0 + np.exp(-x))


def swiglu_mlp(hn: np.ndarray, w_gate_up: np.ndarray,
               w_down: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """down(silu(gate) * up) with gate, up = chunk(gate_up(hn), 2).

    Returns (act, mlp_out) where act = silu(gate) * up.
    """
    gate_up = hn @ w_gate_up.T
    inter = gate_up.shape[-1] // 2
    gate, up = gate_up[..., :inter], gate_up[..., inter:]
    act = silu(gate) * up
    return act, act @ w_down.T


# --------------------------------------------------------------------------
# The layer  ([nanotron] 9.3 + 9.5; [the7] 3.2; [nju] LlamaDecoderLayer内部结构)
# --------------------------------------------------------------------------
def _split_qkv(qkv: np.ndarray, cfg):
    qs, ks = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    T = qkv.shape[0]
    q = qkv[:, :qs].reshape(T, cfg.n_heads, cfg.head_dim)
    k = qkv[:, qs:qs + ks].reshape(T, cfg.n_kv_heads, cfg.head_dim)
    v = qkv[:, qs + ks:].reshape(T, cfg.n_kv_heads, cfg.head_dim)
    return q, k, v


def decoder_layer(x: np.ndarray, w, cfg, positions: np.ndarray,
                  cu_seqlens: np.ndarray) -> dict:
    """Prefill forward over T tokens (padded batch or packed varlen).

    x [T, hidden] float64; ``w`` has w_qkv [Nqkv, H], w_o [H, Hq*d],
    w_gate_up [2I, H], w_down [H, I], g_in [H], g_post [H] (float64).
    Returns the intermediates: q, k (after RoPE), v, attn [T, Hq*d], h, act
    and out [T, H].
    """
    T = x.shape[0]
    residual = x
    xn = rms_norm(x, w.g_in, cfg.rms_eps)
    qkv = xn @ w.w_qkv.T
    q, k, v = _split_qkv(qkv, cfg)
    cos, sin = rope_cos_sin(positions, layer_inv_freq(cfg))
    q, k = apply_rope(q, cos, sin), apply_rope(k, cos, sin)
    attn = causal_attention(q, k, v, cu_seqlens).reshape(T, -1)
    h = residual + attn @ w.w_o.T
    hn = rms_norm(h, w.g_post, cfg.rms_eps)
    act, mlp = swiglu_mlp(hn, w.w_gate_up, w.w_down)
    out = h + mlp
    return dict(q=q, k=k, v=v, attn=attn, h=h, act=act, out=out)


def decoder_layer_rows(x: np.ndarray, w, cfg, positions: np.ndarray,
                       cu_seqlens: np.ndarray, rows) -> dict:
    """The same layer for the selected output rows only.

    Each selected token needs the keys and values of its own sequence up to
    itself, so those are projected for the sequence prefix; every other step
    runs on the selected rows alone.  Returns out / h / attn / act for
    ``rows`` (in the order given).
    """
    rows = np.asarray(rows, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    inv_freq = layer_inv_freq(cfg)
    qs, ks = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    n_rep = cfg.n_heads // cfg.n_kv_heads
    d = cfg.head_dim
    seq_of = np.searchsorted(cu, rows, side="right") - 1
    attn = np.zeros((len(rows), qs))
    for s in np.unique(seq_of):
        a = int(cu[s])
        sel = np.nonzero(seq_of == s)[0]
        last = int(rows[sel].max())
        xn = rms_norm(x[a:last + 1], w.g_in, cfg.rms_eps)
        kv = xn @ w.w_qkv[qs:].T
        k = kv[:, :ks].reshape(-1, cfg.n_kv_heads, d)
        v = kv[:, ks:].reshape(-1, cfg.n_kv_heads, d)
        cos, sin = rope_cos_sin(positions[a:last + 1], inv_freq)
        k = apply_rope(k, cos, sin)
        keys, values = repeat_kv(k, n_rep), repeat_kv(v, n_rep)
        for j in sel:
            t = int(rows[j])
            q = (xn[t - a] @ w.w_qkv[:qs].T).reshape(1, cfg.n_heads, d)
            q = apply_rope(q, cos[t - a:t - a + 1], sin[t - a:t - a + 1])[0]
            for hh in range(cfg.n_heads):
                sc = keys[: t - a + 1, hh] @ q[hh] / math.sqrt(d)
                sc = sc - sc.max()
                p = np.exp(sc)
                p = p / p.sum()
                attn[j, hh * d:(hh + 1) * d] = p @ values[: t - a + 1, hh]
    h = x[rows] + attn @ w.w_o.T
    hn = rms_norm(h, w.g_post, cfg.rms_eps)
    act, mlp = swiglu_mlp(hn, w.w_gate_up, w.w_down)
    return dict(attn=attn, h=h, act=act, out=h + mlp)


def decoder_layer_decode(x: np.ndarray, w, cfg, cache_rows,
                         start_pos: np.ndarray) -> dict:
    """One new token per sequence against a KV cache ([the7] 3.2; [csdn] 3).

    x [B, hidden]; ``cache_rows(b, n)`` returns the first n cached (already
    rotated) keys and the values of sequence b as float64 [n, Hkv, d].  The
    new token of sequence b sits at position start_pos[b]: its rotated key and
    value are written at cache row start_pos[b], and it attends to rows
    0 .. start_pos[b].  Returns out [B, H], the new cache rows k_new / v_new
    [B, Hkv, d] and the intermediates.
    """
    B = x.shape[0]
    d = cfg.head_dim
    n_rep = cfg.n_heads // cfg.n_kv_heads
    xn = rms_norm(x, w.g_in, cfg.rms_eps)
    qkv = xn @ w.w_qkv.T
    q, k, v = _split_qkv(qkv, cfg)
    cos, sin = rope_cos_sin(start_pos, layer_inv_freq(cfg))
    q, k = apply_rope(q, cos, sin), apply_rope(k, cos, sin)
    attn = np.zeros((B, cfg.n_heads, d))
    for b in range(B):
        sp = int(start_pos[b])
        old_k, old_v = cache_rows(b, sp)
        keys = repeat_kv(np.concatenate([old_k, k[b:b + 1]], axis=0), n_rep)
        values = repeat_kv(np.concatenate([old_v, v[b:b + 1]], axis=0), n_rep)
        for hh in range(cfg.n_heads):
            sc = keys[:, hh] @ q[b, hh] / math.sqrt(d)
            sc = sc - sc.max()
            p = np.exp(sc)
            p = p / p.sum()
            attn[b, hh] = p @ values[:, hh]
    attn = attn.reshape(B, -1)
    h = x + attn @ w.w_o.T
    hn = rms_norm(h, w.g_post, cfg.rms_eps)
    act, mlp = swiglu_mlp(hn, w.w_gate_up, w.w_down)
    return dict(q=q, k_new=k, v_new=v, attn=attn, h=h, act=act, out=h + mlp)


def decoder_layer_cached(x: np.ndarray, w, cfg, cache_rows, start_pos: np.ndarray,
                         S: int) -> dict:
    """S new tokens per sequence against a KV cache: the general form of the
    Meta Attention.forward with start_pos and seqlen > 1 ([the7] 3.2: the new
    keys / values go to cache rows start_pos .. start_pos + S - 1 and the
    queries attend to rows 0 .. start_pos + S - 1; [csdn] "5. Transformer":
    the mask is zeros over the start_pos cached columns followed by the
    causal triangle over the new tokens).

    x [B * S, hidden], rows b * S .. b * S + S - 1 the new tokens of sequence
    b at positions start_pos[b] .. start_pos[b] + S - 1; ``cache_rows(b, n)``
    as for decoder_layer_decode.  Returns out [B * S, H], the new cache rows
    k_new / v_new [B * S, Hkv, d] and the intermediates.
    """
    BS = x.shape[0]
    B = BS // S
    d = cfg.head_dim
    n_rep = cfg.n_heads // cfg.n_kv_heads
    positions = (np.repeat(np.asarray(start_pos, dtype=np.int64), S) +
                 np.tile(np.arange(S), B))
    xn = rms_norm(x, w.g_in, cfg.rms_eps)
    qkv = xn @ w.w_qkv.T
    q, k, v = _split_qkv(qkv, cfg)
    cos, sin = rope_cos_sin(positions, layer_inv_freq(cfg))
    q, k = apply_rope(q, cos, sin), apply_rope(k, cos, sin)
    attn = np.zeros((BS, cfg.n_heads, d))
    for b in range(B):
        sp = int(start_pos[b])
        old_k, old_v = cache_rows(b, sp)
        new = slice(b * S, (b + 1) * S)
        keys = repeat_kv(np.concatenate([old_k, k[new]], axis=0), n_rep)
        values = repeat_kv(np.concatenate([old_v, v[new]], axis=0), n_rep)
        # mask row i: the sp cached columns, then new columns 0 .. i
        mask = np.concatenate([np.zeros((S, sp)),
                               np.triu(np.full((S, S), -np.inf), k=1)], axis=1)
        for hh in range(cfg.n_heads):
            sc = q[new, hh] @ keys[:, hh].T / math.sqrt(d) + mask
            sc = sc - sc.max(axis=1, keepdims=True)
            p = np.exp(sc)
            p = p / p.sum(axis=1, keepdims=True)
            attn[new, hh] = p @ values[:, hh]
    attn = attn.reshape(BS, -1)
    h = x + attn @ w.w_o.T
    hn = rms_norm(h, w.g_post, cfg.rms_eps)
    act, mlp = swiglu_mlp(hn, w.w_gate_up, w.w_down)
    return dict(q=q, k_new=k, v_new=v, attn=attn, h=h, act=act, out=h + mlp)


def model_forward(x: np.ndarray, layers, cfg, positions: np.ndarray,
                  cu_seqlens: np.ndarray, g_final: np.ndarray, w_lm: np.ndarray) -> dict:
    """A stack of decoder layers, the final RMSNorm and the output projection
    ([nanotron] 9.5, the layers applied in turn; [csdn] "5. Transformer":
    h = layer(h) for every layer, then the norm, then the output projection
    to the vocabulary logits).  ``layers`` holds one weight set per layer (as
    decoder_layer takes); w_lm [vocab, hidden].  Returns the last hidden
    state, its normalised form and the logits [T, vocab]."""
    h = x
    for w in layers:
        h = decoder_layer(h, w, cfg, positions, cu_seqlens)["out"]
    hn = rms_norm(h, g_final, cfg.rms_eps)
    return dict(hidden=h, normed=hn, logits=hn @ w_lm.T)
