"""The workloads at their full sizes, in the launch configuration the bench
times.  Prefill workloads compare every row of every stage (q|k|v,
attention, h, act, output) with the oracle run on the whole batch; decode
and the 16 x 4 chunked prefill compare every new token and the cache rows
written."""

import numpy as np
import pytest
import torch

import oracle
from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

from parity import (assert_close, assert_stage_close, build_layer, oracle_qkv, poison_cache,
                    run_forward, to_f64, weights_f64)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["1b", "8b", "varlen"])
def test_prefill_workload_every_row(name):
    """Every row of every stage at the full size, in the bench's launch
    configuration: the persistent GEMM schedule (all tile rounds, the
    split-tile phase of the long-K GEMMs) and the attention's full work-item
    order are all covered."""
    inp = synth.make_inputs(name)
    s = inp.workload.shape
    varlen = inp.workload.kind == "varlen"
    layer = build_layer(inp)
    out = run_forward(layer, inp, varlen)
    assert layer.status() == B.LLAMA_OK
    st = layer.stages(inp.tokens)
    got = {k: to_f64(st[k]) for k in ("qkv", "attn", "h", "act")}
    got["out"] = to_f64(out)
    layer.close()
    del st, out
    torch.cuda.empty_cache()
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights), s,
                               inp.positions, inp.cu_seqlens)
    assert_stage_close(got["qkv"], oracle_qkv(ref), s.dtype, f"{name} qkv")
    assert_stage_close(got["attn"], ref["attn"], s.dtype, f"{name} attn")
    assert_stage_close(got["h"], ref["h"], s.dtype, f"{name} h")
    assert_stage_close(got["act"], ref["act"], s.dtype, f"{name} act")
    assert_close(got["out"], ref["out"], s.dtype, f"{name} out")


def test_decode_workload():
    inp = synth.make_inputs("decode")
    s = inp.workload.shape
    layer = build_layer(inp)
    ck = to_device(poison_cache(inp.cache_k, inp.start_pos))
    cv = to_device(poison_cache(inp.cache_v, inp.start_pos))
    out = layer.decode(to_device(inp.x), ck, cv, to_device(inp.start_pos))
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    rows = lambda b, n: (synth.to_f64(inp.cache_k[b, :n]),
                         synth.to_f64(inp.cache_v[b, :n]))
    ref = oracle.decoder_layer_decode(synth.to_f64(inp.x),
                                      weights_f64(inp.weights), s, rows,
                                      inp.start_pos)
    assert_close(to_f64(out), ref["out"], s.dtype, "out")
    st = layer.stages(inp.tokens, decode=True)
    assert_stage_close(to_f64(st["attn"]), ref["attn"], s.dtype, "attn")
    b_idx = torch.arange(len(inp.start_pos), device="cuda")
    sp = torch.as_tensor(inp.start_pos, device="cuda").long()
    assert_stage_close(to_f64(ck[b_idx, sp]), ref["k_new"], s.dtype, "k rows")
    assert_stage_close(to_f64(cv[b_idx, sp]), ref["v_new"], s.dtype, "v rows")
    layer.close()


def test_chunked_workload():
    """16 sequences x 4 new tokens against 8192-row caches (prefixes
    512..8188): the split-KV attention with the four tokens of a sequence in
    one tile, reading each prefix once."""
    inp = synth.make_inputs("chunked")
    s = inp.workload.shape
    S = inp.workload.seq_tokens
    layer = build_layer(inp)
    ck = to_device(poison_cache(inp.cache_k, inp.start_pos))
    cv = to_device(poison_cache(inp.cache_v, inp.start_pos))
    out = layer.forward_cached(to_device(inp.x), ck, cv, to_device(inp.start_pos), S)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    rows = lambda b, n: (synth.to_f64(inp.cache_k[b, :n]),
                         synth.to_f64(inp.cache_v[b, :n]))
    ref = oracle.decoder_layer_cached(synth.to_f64(inp.x), weights_f64(inp.weights), s,
                                      rows, inp.start_pos, S)
    assert_close(to_f64(out), ref["out"], s.dtype, "chunked out")
    for b, p in enumerate(inp.start_pos):
        new = slice(b * S, (b + 1) * S)
        assert_stage_close(to_f64(ck[b, p:p + S]), ref["k_new"][new], s.dtype, "k rows")
        assert_stage_close(to_f64(cv[b, p:p + S]), ref["v_new"][new], s.dtype, "v rows")
    layer.close()
