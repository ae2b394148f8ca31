"""The same call twice gives the same bits: the layer adds every sum that
several tiles or CTAs contribute to in a fixed order (the row sums of
squares of h for the second RMSNorm, in the prefill GEMM's and the decode
finalize kernels' slots; the RMSNorm^T row dots; the norm-weight gradients'
row-group sums), so the result does not depend on the order in which tiles
finish.  Checked on the 8B-shaped layer (hidden 4096: 32 slots a row) for
the prefill forward, the backward and a decode step."""

import numpy as np
import pytest
import torch

from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

from parity import build_layer, poison_cache

pytestmark = pytest.mark.gpu


def test_forward_and_backward_repeat_bit_for_bit():
    s = synth.WORKLOADS["8b"].shape
    inp = synth.make_inputs(synth.custom_workload("repro_8b", s, "padded", index=340,
                                                  batch=2, seq=256))
    layer = build_layer(inp)
    x = to_device(inp.x)
    dout = to_device(synth.make_dout(inp))
    args = dict(n_seq=2, seq_len=256)
    outs = [layer.forward(x, **args).clone() for _ in range(3)]
    grads = [{k: v.clone() for k, v in layer.backward(x, dout, **args).items()}
             for _ in range(3)]
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    for g in grads[1:]:
        for k in g:
            assert torch.equal(g[k], grads[0][k]), k
    layer.close()


def test_decode_repeats_bit_for_bit():
    inp = synth.make_inputs(synth.custom_workload(
        "repro_dec", synth.WORKLOADS["8b"].shape, "decode", index=341, batch=24,
        max_seq=1024, min_start=100))
    layer = build_layer(inp)
    x = to_device(inp.x)
    sp = to_device(inp.start_pos)
    outs = []
    for _ in range(3):
        ck = to_device(poison_cache(inp.cache_k, inp.start_pos))
        cv = to_device(poison_cache(inp.cache_v, inp.start_pos))
        outs.append(layer.decode(x, ck, cv, sp).clone())
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    layer.close()
