"""Pins for the oracle's RMSNorm and RoPE (CPU only).

Each ``pin_*`` takes the function under test, so the ``*_catches_*`` tests can
plant a mistake in a copy of the oracle and show that the pin fails on it.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.default_rng(7)


# ----------------------------------------------------------------- RMSNorm
def pin_rms_unit(rms_norm_fn):
    """RMS of x_n / g equals sqrt(ms / (ms + eps)) exactly (closed form)."""
    x = RNG.standard_normal((5, 48)) * 3.0
    g = 1.0 + 0.1 * RNG.standard_normal(48)
    for eps in (0.0, 1e-5, 0.3):
        y = rms_norm_fn(x, g, eps) / g
        ms = np.mean(x * x, axis=-1)
        got = np.sqrt(np.mean(y * y, axis=-1))
        np.testing.assert_allclose(got, np.sqrt(ms / (ms + eps)), rtol=1e-13)


def test_rms_norm_unit_rms():
    pin_rms_unit(oracle.rms_norm)


def test_rms_norm_matches_torch():
    x = RNG.standard_normal((7, 64))
    g = 1.0 + 0.1 * RNG.standard_normal(64)
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(g), 1e-5)
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-5), ref.numpy(),
                               rtol=1e-13, atol=1e-14)


def test_rms_norm_catches_eps_outside_sqrt():
    def mutant(x, g, eps):
        return x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * g
    with pytest.raises(AssertionError):
        pin_rms_unit(mutant)


# ----------------------------------------------------------------- inv_freq
def test_inv_freq_closed_form():
    for d, base in ((64, 1e4), (128, 5e5)):
        f = oracle.rope_inv_freq(d, base)
        assert f.shape == (d // 2,)
        assert f[0] == 1.0
        np.testing.assert_allclose(f[1:] / f[:-1], base ** (-2.0 / d),
                                   rtol=1e-12)
        np.testing.assert_allclose(f[-1], base ** (-(d - 2) / d), rtol=1e-12)


def _bands(f, fs, factor):
    keep = int(np.sum(fs == f))
    scaled = int(np.sum(fs == f / factor))
    return keep, len(f) - keep - scaled, scaled


def pin_llama3(scale_fn):
    # factor 1 leaves every frequency where it was
    f = oracle.rope_inv_freq(128, 5e5)
    np.testing.assert_allclose(scale_fn(f, 1.0, 1.0, 4.0, 8192), f, rtol=1e-15)
    # band sizes: wavelength 2*pi*base^(2i/d) against 8192/4 and 8192/1,
    # solved by hand: d=64 -> i<=14 keep, i>=18 scaled; d=128 -> i<=28, i>=35
    for d, factor, want in ((64, 32.0, (15, 3, 14)), (128, 8.0, (29, 6, 29))):
        f = oracle.rope_inv_freq(d, 5e5)
        fs = scale_fn(f, factor, 1.0, 4.0, 8192)
        assert _bands(f, fs, factor) == want
        # scaled values lie between f / factor and f and keep decreasing
        assert np.all(fs <= f * (1 + 1e-15))
        assert np.all(fs >= f / factor * (1 - 1e-15))
        assert np.all(np.diff(fs) < 0)
    # continuity: a frequency exactly on an edge of the middle band
    edges = np.array([2 * math.pi / 2048.0, 2 * math.pi / 8192.0])
    fs = scale_fn(edges, 8.0, 1.0, 4.0, 8192)
    np.testing.assert_allclose(fs, [edges[0], edges[1] / 8.0], rtol=1e-13)


def test_llama3_scaling():
    pin_llama3(oracle.llama3_scale_inv_freq)


def test_llama3_catches_swapped_interpolation_weight():
    def mutant(inv_freq, factor, low, high, orig):
        out = []
        for f in inv_freq:
            lam = 2 * math.pi / f
            if lam < orig / high:
                out.append(f)
            elif lam > orig / low:
                out.append(f / factor)
            else:
                s = (orig / lam - low) / (high - low)
                out.append(s * f / factor + (1 - s) * f)
        return np.array(out)
    with pytest.raises(AssertionError):
        pin_llama3(mutant)


# ----------------------------------------------------------------- RoPE
def _rope(apply_fn, x, pos, d, base=1e4):
    cos, sin = oracle.rope_cos_sin(pos, oracle.rope_inv_freq(d, base))
    return apply_fn(x, cos, sin)


def pin_rope_unit_vectors(apply_fn):
    """e_i -> cos e_i + sin e_{i+d/2}; e_{i+d/2} -> -sin e_i + cos e_{i+d/2}."""
    d = 16
    f = oracle.rope_inv_freq(d, 1e4)
    for p in (0, 1, 5, 1000):
        for i in range(d // 2):
            for j, (ci, cj) in ((i, (1, 0)), (i + d // 2, (0, 1))):
                e = np.zeros((1, 1, d))
                e[0, 0, j] = 1.0
                y = _rope(apply_fn, e, np.array([p]), d)[0, 0]
                c, s = math.cos(p * f[i]), math.sin(p * f[i])
                want = np.zeros(d)
                want[i] = ci * c - cj * s
                want[i + d // 2] = ci * s + cj * c
                np.testing.assert_allclose(y, want, atol=1e-15)


def test_rope_unit_vectors():
    pin_rope_unit_vectors(oracle.apply_rope)


def test_rope_catches_sign_flip():
    def mutant(x, cos, sin):
        return x * cos[:, None, :] - oracle.rotate_half(x) * sin[:, None, :]
    with pytest.raises(AssertionError):
        pin_rope_unit_vectors(mutant)


def test_rope_position_zero_is_identity():
    x = RNG.standard_normal((3, 4, 64))
    y = _rope(oracle.apply_rope, x, np.zeros(3, dtype=np.int64), 64)
    np.testing.assert_array_equal(y, x)


def test_rope_preserves_pair_norms():
    d = 128
    x = RNG.standard_normal((6, 3, d))
    y = _rope(oracle.apply_rope, x, np.array([0, 1, 7, 100, 4095, 8191]), d,
              5e5)
    n_in = x[..., : d // 2] ** 2 + x[..., d // 2:] ** 2
    n_out = y[..., : d // 2] ** 2 + y[..., d // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_rope_dot_depends_on_offset_only():
    d = 64
    q = RNG.standard_normal((1, 1, d))
    k = RNG.standard_normal((1, 1, d))
    for m, n in ((5, 2), (40, 3), (100, 100)):
        ref = None
        for shift in (0, 1, 17, 900):
            qm = _rope(oracle.apply_rope, q, np.array([m + shift]), d)
            kn = _rope(oracle.apply_rope, k, np.array([n + shift]), d)
            dot = float(np.sum(qm * kn))
            if ref is None:
                ref = dot
            assert abs(dot - ref) < 1e-11 * max(1.0, abs(ref))


def test_rope_matches_complex_form():
    """The polar/complex form on neighbouring pairs equals rotate_half on the
    (i, i + d/2) pairs once each head's dims are interleaved."""
    d = 32
    x = RNG.standard_normal((5, 2, d))
    pos = np.array([0, 3, 11, 200, 7000])
    f = oracle.llama3_scale_inv_freq(oracle.rope_inv_freq(d, 5e5), 8.0, 1.0,
                                     4.0, 8192)
    cos, sin = oracle.rope_cos_sin(pos, f)
    y = oracle.apply_rope(x, cos, sin)
    inter = np.empty_like(x)
    inter[..., 0::2], inter[..., 1::2] = x[..., : d // 2], x[..., d // 2:]
    z = inter[..., 0::2] + 1j * inter[..., 1::2]
    freqs_cis = np.exp(1j * np.outer(pos, f))[:, None, :]
    zr = z * freqs_cis
    np.testing.assert_allclose(y[..., : d // 2], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[..., d // 2:], zr.imag, atol=1e-12)


# ------------------------------------------- linear and dynamic NTK scaling
def _cfg(scaling, factor=4.0, max_position=4096, original=1024, d=64, base=10000.0):
    import types
    return types.SimpleNamespace(head_dim=d, rope_base=base, rope_scaling=scaling,
                                 rope_factor=factor, rope_low_freq_factor=1.0,
                                 rope_high_freq_factor=4.0,
                                 rope_original_max_pos=original,
                                 max_position=max_position)


def test_linear_scaling_divides_the_positions():
    # the page's statement t = t / factor: the scaled table at position p is
    # the unscaled table at p / factor (non-integer positions included)
    f = 4.0
    p = np.array([0, 1, 3, 7, 100, 4095], dtype=np.float64)
    cos_s, sin_s = oracle.rope_cos_sin(p, oracle.layer_inv_freq(_cfg(2, factor=f)))
    cos_u, sin_u = oracle.rope_cos_sin(p / f, oracle.rope_inv_freq(64, 10000.0))
    np.testing.assert_allclose(cos_s, cos_u, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sin_s, sin_u, rtol=0, atol=1e-12)


def test_dynamic_ntk_leaves_the_original_context_alone():
    plain = oracle.rope_inv_freq(64, 10000.0)
    for L in (512, 1024):  # at or within the original 1024 positions
        np.testing.assert_array_equal(
            oracle.layer_inv_freq(_cfg(3, max_position=L)), plain)


def test_dynamic_ntk_divides_the_lowest_frequency_by_the_scale():
    # beyond the original context: the highest frequency stays 1 and the
    # lowest is divided by exactly scale = factor * L / orig - (factor - 1),
    # the property the d / (d - 2) exponent is chosen for
    for d, f, L, orig in ((64, 4.0, 4096, 1024), (128, 8.0, 12000, 8192)):
        plain = oracle.rope_inv_freq(d, 500000.0)
        got = oracle.layer_inv_freq(_cfg(3, factor=f, max_position=L, original=orig,
                                         d=d, base=500000.0))
        scale = f * L / orig - (f - 1.0)
        assert got[0] == 1.0
        np.testing.assert_allclose(got[-1], plain[-1] / scale, rtol=1e-12)
        assert np.all(got <= plain) and np.all(np.diff(got) < 0)


def test_dynamic_ntk_is_continuous_at_the_original_length():
    # scale = 1 at L = orig, so the table does not jump there
    just = oracle.layer_inv_freq(_cfg(3, max_position=1025))
    plain = oracle.rope_inv_freq(64, 10000.0)
    assert just[0] == plain[0] == 1.0
    assert np.all(just[1:] < plain[1:])  # one row past: already (slightly) scaled
    np.testing.assert_allclose(just, plain, rtol=1e-2)
