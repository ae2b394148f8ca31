"""The algorithmic work bench.py divides by (no GPU needed): FLOPs of the
prefill workloads, bytes of the decode workloads, FLOPs of the model stack."""

import numpy as np
import pytest

import bench
from llama_decoder_layer_prologue_b300 import synth


@pytest.mark.parametrize("name,linear_per_token", [("1b", 121.6e6), ("8b", 436.2e6)])
def test_prefill_linear_flops_per_token(name, linear_per_token):
    inp = synth.make_inputs(name, with_cache=False, x_only=True)
    w = bench.algorithmic_work(inp)
    linear = sum(v for k, v in w["flops"].items() if k != "attention")
    assert abs(linear / inp.tokens - linear_per_token) < 0.05e6


def test_prefill_attention_counts_visible_pairs():
    # causal: sequence of L tokens has L (L + 1) / 2 visible (q, k) pairs, each
    # 2 d FLOPs for q.k and 2 d for p.v, per query head
    inp = synth.make_inputs("1b", with_cache=False, x_only=True)
    s = inp.workload.shape
    L, n = 2048, 4
    pairs = n * L * (L + 1) / 2
    assert bench.algorithmic_work(inp)["flops"]["attention"] == pytest.approx(
        pairs * 4 * s.head_dim * s.n_heads)


def test_decode_bytes():
    inp = synth.make_inputs("decode", with_cache=False)
    s = inp.workload.shape
    w = bench.algorithmic_work(inp)
    kv = float(np.sum(inp.start_pos.astype(np.float64))) * 2 * s.n_kv_heads * s.head_dim * 2
    assert w["kv_read"] == pytest.approx(kv)
    assert w["weight_bytes"] == pytest.approx(436.2e6, rel=1e-3)
    assert 1.4e9 < w["total_bytes"] < 1.7e9


def test_model_flops_are_layers_plus_the_output_projection():
    inp = synth.make_inputs("1b", with_cache=False, x_only=True)
    s = inp.workload.shape
    layer = bench.algorithmic_work(inp)["total_flops"]
    lens = np.diff(inp.cu_seqlens)
    got = bench.model_flops(s, lens, 16, 128256)
    assert got == pytest.approx(16 * layer + 2.0 * inp.tokens * s.hidden * 128256)
