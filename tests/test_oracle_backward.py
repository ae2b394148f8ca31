"""The layer's fp64 backward oracle against two independent references:
torch.autograd over a separate float64 torch forward, and central finite
differences of the numpy forward."""

import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle.backward import decoder_layer_backward

RNG = np.random.default_rng(21)


def cfg(scaling=0, d=16, hq=4, hkv=2, H=32, I=48):
    return types.SimpleNamespace(
        hidden=H, n_heads=hq, n_kv_heads=hkv, head_dim=d, intermediate=I,
        rms_eps=1e-5, rope_base=10000.0, rope_scaling=scaling, rope_factor=8.0,
        rope_low_freq_factor=1.0, rope_high_freq_factor=4.0,
        rope_original_max_pos=64, max_position=64)


def weights(c):
    nqkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim
    return types.SimpleNamespace(
        w_qkv=0.2 * RNG.standard_normal((nqkv, c.hidden)),
        w_o=0.2 * RNG.standard_normal((c.hidden, c.n_heads * c.head_dim)),
        w_gate_up=0.2 * RNG.standard_normal((2 * c.intermediate, c.hidden)),
        w_down=0.2 * RNG.standard_normal((c.hidden, c.intermediate)),
        g_in=1.0 + 0.1 * RNG.standard_normal(c.hidden),
        g_post=1.0 + 0.1 * RNG.standard_normal(c.hidden))


def torch_forward(x, W, c, positions, cu, inv_freq):
    """The layer written again with torch ops (autograd differentiates it)."""
    def norm(a, g):
        return a * torch.rsqrt(a.pow(2).mean(-1, keepdim=True) + c.rms_eps) * g

    d, T = c.head_dim, x.shape[0]
    qs, ks = c.n_heads * d, c.n_kv_heads * d
    qkv = norm(x, W["g_in"]) @ W["w_qkv"].T
    q = qkv[:, :qs].reshape(T, c.n_heads, d)
    k = qkv[:, qs:qs + ks].reshape(T, c.n_kv_heads, d)
    v = qkv[:, qs + ks:].reshape(T, c.n_kv_heads, d)
    ang = torch.as_tensor(positions, dtype=torch.float64)[:, None] * inv_freq[None]
    cos = torch.cat([ang, ang], -1).cos()[:, None]
    sin = torch.cat([ang, ang], -1).sin()[:, None]

    def rot(a):
        return a * cos + torch.cat([-a[..., d // 2:], a[..., :d // 2]], -1) * sin

    q, k = rot(q), rot(k)
    rep = c.n_heads // c.n_kv_heads
    outs = []
    for a, b in zip(cu[:-1], cu[1:]):
        Q = q[a:b].transpose(0, 1)
        K = k[a:b].repeat_interleave(rep, 1).transpose(0, 1)
        V = v[a:b].repeat_interleave(rep, 1).transpose(0, 1)
        L = b - a
        mask = torch.triu(torch.full((L, L), float("-inf"), dtype=torch.float64), 1)
        P = torch.softmax(Q @ K.transpose(1, 2) / d ** 0.5 + mask, -1)
        outs.append((P @ V).transpose(0, 1).reshape(L, -1))
    h = x + torch.cat(outs) @ W["w_o"].T
    gu = norm(h, W["g_post"]) @ W["w_gate_up"].T
    I = c.intermediate
    return h + (F.silu(gu[:, :I]) * gu[:, I:]) @ W["w_down"].T


@pytest.mark.parametrize("scaling", [0, 1])
def test_backward_matches_autograd(scaling):
    c = cfg(scaling)
    w = weights(c)
    lens = [3, 1, 6]
    cu = np.concatenate([[0], np.cumsum(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    x = RNG.standard_normal((cu[-1], c.hidden))
    dout = RNG.standard_normal(x.shape)
    inv = torch.as_tensor(oracle.layer_inv_freq(c)) if scaling else \
        1.0 / c.rope_base ** (torch.arange(0, c.head_dim, 2, dtype=torch.float64) / c.head_dim)
    xt = torch.tensor(x, requires_grad=True)
    W = {k: torch.tensor(getattr(w, k), requires_grad=True) for k in vars(w)}
    out = torch_forward(xt, W, c, pos, cu.tolist(), inv)
    np.testing.assert_allclose(out.detach().numpy(),
                               oracle.decoder_layer(x, w, c, pos, cu)["out"],
                               rtol=1e-11, atol=1e-12)  # the same forward
    out.backward(torch.tensor(dout))
    got = decoder_layer_backward(x, w, c, pos, cu, dout)
    np.testing.assert_allclose(got["dx"], xt.grad.numpy(), rtol=1e-9, atol=1e-11)
    for k in ("w_qkv", "w_o", "w_gate_up", "w_down", "g_in", "g_post"):
        np.testing.assert_allclose(got["d" + k], W[k].grad.numpy(), rtol=1e-9,
                                   atol=1e-11, err_msg=k)


def test_backward_matches_finite_differences():
    c = cfg()
    w = weights(c)
    cu = np.array([0, 5])
    pos = np.arange(5)
    x = RNG.standard_normal((5, c.hidden))
    dout = RNG.standard_normal(x.shape)
    got = decoder_layer_backward(x, w, c, pos, cu, dout)

    def loss(xx, ww):
        return float(np.sum(dout * oracle.decoder_layer(xx, ww, c, pos, cu)["out"]))

    eps = 1e-6
    for (t, j) in [(0, 3), (4, 17), (2, 31)]:
        xp, xm = x.copy(), x.copy()
        xp[t, j] += eps
        xm[t, j] -= eps
        fd = (loss(xp, w) - loss(xm, w)) / (2 * eps)
        assert abs(fd - got["dx"][t, j]) <= 1e-6 * max(1.0, abs(fd))
    for name, idx in [("w_qkv", (5, 7)), ("w_qkv", (70, 2)), ("w_o", (3, 9)),
                      ("w_gate_up", (60, 11)), ("w_down", (8, 40)), ("g_in", (6,)),
                      ("g_post", (13,))]:
        wp = types.SimpleNamespace(**{k: v.copy() for k, v in vars(w).items()})
        wm = types.SimpleNamespace(**{k: v.copy() for k, v in vars(w).items()})
        getattr(wp, name)[idx] += eps
        getattr(wm, name)[idx] -= eps
        fd = (loss(x, wp) - loss(x, wm)) / (2 * eps)
        an = got["d" + name][idx]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, an)
