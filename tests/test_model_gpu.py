"""The model-level stack on the GPU against the fp64 oracle: decoder layers in
turn, the final RMSNorm and the output projection to the vocabulary logits."""

import numpy as np
import pytest
import torch

import oracle
from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device
from llama_decoder_layer_prologue_b300.model import LlamaModel

from parity import errors, report, to_f64, weights_f64

pytestmark = pytest.mark.gpu


def _shape(H=256, hq=4, hkv=2, d=64, I=256):
    return synth.LayerShape(hidden=H, n_heads=hq, n_kv_heads=hkv, head_dim=d,
                            intermediate=I, rms_eps=1e-5, rope_base=500000.0,
                            rope_scaling=0, max_position=1024, dtype="bf16")


def test_rmsnorm_matches_the_oracle():
    rng = np.random.default_rng(4)
    rows, H = 300, 512
    x = synth.bf16_round_bits(3.0 * rng.standard_normal((rows, H), dtype=np.float32))
    g = synth.bf16_round_bits(1.0 + 0.1 * rng.standard_normal(H, dtype=np.float32))
    out = torch.empty(rows, H, dtype=torch.bfloat16, device="cuda")
    xd, gd = to_device(x), to_device(g)  # alive until the kernel has run
    B.llama_rmsnorm_bf16(xd.data_ptr(), gd.data_ptr(), out.data_ptr(), rows, H, 1e-5,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = oracle.rms_norm(synth.to_f64(x), synth.to_f64(g), 1e-5)
    got = to_f64(out)
    # one bf16 rounding of an fp32 product: within 2^-8 relative
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("kind", ["padded", "varlen"])
def test_model_logits_match_the_oracle(kind):
    s = _shape()
    kw = dict(batch=2, seq=100) if kind == "padded" else dict(
        total_tokens=300, min_len=1, max_len=200)
    w = synth.custom_workload("model", s, kind, **kw)
    m_in = synth.make_model_inputs(w, n_layers=2, vocab=1024)
    inp = m_in.first
    model = LlamaModel.from_numpy(s, m_in)
    x = to_device(inp.x)
    if kind == "padded":
        logits = model.forward(x, n_seq=2, seq_len=100)
    else:
        S = int(np.diff(inp.cu_seqlens).max())
        cu = to_device(inp.cu_seqlens)
        logits = model.forward(x, cu_seqlens=cu, seq_len=S)
    torch.cuda.synchronize()
    assert model.status() == B.LLAMA_OK
    ref = oracle.model_forward(synth.to_f64(inp.x), [weights_f64(l) for l in m_in.layers],
                               s, inp.positions, inp.cu_seqlens,
                               synth.to_f64(m_in.g_final), synth.to_f64(m_in.w_lm))
    e = errors(to_f64(logits), ref["logits"])
    report(f"model logits ({kind})", e)
    # two layers, each handing on bf16 hidden states, then bf16 logits
    assert e["finite"]
    assert e["mean_rel"] <= 1e-2
    assert e["max_abs"] <= 4e-2 * e["rms_ref"]
    model.close()

