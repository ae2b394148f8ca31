"""The training pair on the GPU: llama_layer_forward_train (the forward that
keeps the activations the backward reads) and llama_layer_backward_saved (the
backward that reads them instead of recomputing the forward).  The forward
computes what llama_layer_forward computes and the backward what
llama_layer_backward computes, through the same kernels on the same values,
so both are compared bit for bit with those calls (themselves compared with
the fp64 oracle in test_layer_gpu.py and test_backward_gpu.py): every sum
that tiles contribute to (the row sums of squares of h, the RMSNorm^T row
dots, the norm-weight gradients) is added in a fixed order, so a call's
result does not depend on the order in which tiles finish
(test_reproducible_gpu.py).  One case at the 8B shape is compared with the
oracle's chain rule directly.  A saved backward whose
arguments do not match the training forward, or whose workspace another call
has written since, is refused before anything is launched."""

import numpy as np
import pytest
import torch

from oracle.backward import decoder_layer_backward
from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

from parity import assert_close, build_layer, to_f64, weights_f64
from test_backward_gpu import GRADS, L3, assert_close_bf16_result, shape

pytestmark = pytest.mark.gpu


def batch_args(inp, varlen):
    if varlen:
        return dict(cu_seqlens=to_device(inp.cu_seqlens),
                    seq_len=int(np.diff(inp.cu_seqlens).max()))
    return dict(n_seq=len(inp.cu_seqlens) - 1, seq_len=int(inp.cu_seqlens[1]))


CASES = [
    ("padded_llama3", shape(256, 4, 2, 64, 384, **L3), "padded", dict(batch=2, seq=130)),
    ("varlen_d128", shape(512, 4, 2, 128, 256, **L3), "varlen",
     dict(total_tokens=500, min_len=1, max_len=200)),
    ("gqa8", shape(768, 8, 1, 64, 256, **L3), "padded", dict(batch=2, seq=90)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_train_step_equals_forward_and_backward(case):
    name, s, kind, kw = case
    inp = synth.make_inputs(synth.custom_workload(name, s, kind, index=310, **kw))
    varlen = kind == "varlen"
    layer = build_layer(inp)
    x = to_device(inp.x)
    dout = to_device(synth.make_dout(inp))
    args = batch_args(inp, varlen)
    out_ref = layer.forward(x, **args).clone()
    g_ref = {k: v.clone() for k, v in layer.backward(x, dout, **args).items()}
    out = layer.forward_train(x, **args)
    g1 = {k: v.clone() for k, v in layer.backward_saved(x, dout, **args).items()}
    # a second backward from the same kept activations
    g2 = layer.backward_saved(x, dout, **args)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    assert torch.equal(out, out_ref), name
    for k in GRADS:
        for g in (g1, g2):
            assert torch.equal(g[k], g_ref[k]), (name, k)
    layer.close()


def test_saved_backward_matches_oracle_8b_shaped():
    """The 8B-shaped layer on 16 x 256 tokens: M 4096 GEMM grids and more
    attention work items than CTAs (256 for dK/dV, 1024 for dQ)."""
    s = synth.WORKLOADS["8b"].shape
    inp = synth.make_inputs(synth.custom_workload("train_8b_short", s, "padded", index=311,
                                                  batch=16, seq=256))
    layer = build_layer(inp)
    x = to_device(inp.x)
    dout = to_device(synth.make_dout(inp))
    args = batch_args(inp, False)
    layer.forward_train(x, **args)
    g = layer.backward_saved(x, dout, **args)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    got = {k: to_f64(v) for k, v in g.items()}
    layer.close()
    ref = decoder_layer_backward(synth.to_f64(inp.x), weights_f64(inp.weights), s,
                                 inp.positions, inp.cu_seqlens,
                                 synth.to_f64(synth.make_dout(inp)))
    for k in GRADS:
        if k == "dx":
            assert_close_bf16_result(got[k], ref[k], f"8b-shaped saved {k}")
        else:
            assert_close(got[k], ref[k], "bf16", f"8b-shaped saved {k}")


def test_saved_backward_refuses_mismatches():
    s = shape(256, 4, 2, 64, 256)
    inp = synth.make_inputs(synth.custom_workload("train_refuse", s, "padded", index=312,
                                                  batch=2, seq=64))
    layer = build_layer(inp)
    x = to_device(inp.x)
    dout = to_device(synth.make_dout(inp))
    args = batch_args(inp, False)

    def refused(**kw):
        with pytest.raises(B.LlamaError) as e:
            layer.backward_saved(kw.pop("x", x), dout, **kw)
        assert e.value.code == B.LLAMA_ERR_INVALID_ARG

    refused(**args)                      # no training forward yet
    layer.forward_train(x, **args)
    refused(x=x.clone(), **args)         # another input tensor
    refused(n_seq=1, seq_len=128)        # another batch layout
    layer.backward_saved(x, dout, **args)  # the matching call runs
    layer.forward(x, **args)             # a forward through the same workspace
    refused(**args)
    layer.forward_train(x, **args)
    layer.backward(x, dout, **args)      # the recomputing backward writes it too
    refused(**args)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    layer.close()


@pytest.mark.parametrize("case", CASES[:2], ids=lambda c: c[0])
def test_train_step_from_host_equals_the_device_pair(case):
    # host x and dL/d(out) in, dx out; dL/d(out) crosses on a second stream
    # while the forward runs: the same bits as the device-resident pair
    name, s, kind, kw = case
    inp = synth.make_inputs(synth.custom_workload(name, s, kind, index=311, **kw))
    layer = build_layer(inp)
    x = to_device(inp.x)
    dout = to_device(synth.make_dout(inp))
    args = batch_args(inp, kind == "varlen")
    y_ref = layer.forward_train(x, **args).clone()
    g_ref = {k: v.clone() for k, v in layer.backward_saved(x, dout, **args).items()}
    x_h, dout_h = to_device(inp.x, pin=True), to_device(synth.make_dout(inp), pin=True)
    dx_h = torch.full_like(x_h, float("nan")).pin_memory()
    x_d, dout_d, y_d, dx_d = (torch.empty_like(x) for _ in range(4))
    for _ in range(2):  # the second call reuses the staging buffers
        g = layer.train_step_from_host(x_h, dout_h, dx_h, x_d, dout_d, y_d, dx_d, **args)
    torch.cuda.current_stream().synchronize()
    assert layer.status() == B.LLAMA_OK
    assert torch.equal(y_d, y_ref)
    assert torch.equal(dx_h, g_ref["dx"].cpu())
    for k in GRADS:
        assert torch.equal(g[k], g_ref[k]), k
    layer.close()
