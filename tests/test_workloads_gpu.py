"""The five workloads at their full sizes, in the launch configuration the
bench times.  Prefill workloads compare sampled rows (first, last and random
rows of the sequences; the oracle computes each row from its sequence prefix)
at every stage; decode compares every sequence and the cache rows written."""

import numpy as np
import pytest
import torch

import oracle
from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

from parity import (assert_close, assert_stage_close, build_layer, poison_cache, run_forward,
                    sample_rows, to_f64, weights_f64)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,per_seq,max_seqs", [
    ("1b", 6, None), ("8b", 8, None), ("varlen", 3, 8)])
def test_prefill_workload_sampled_rows(name, per_seq, max_seqs):
    inp = synth.make_inputs(name)
    s = inp.workload.shape
    varlen = inp.workload.kind == "varlen"
    layer = build_layer(inp)
    out = run_forward(layer, inp, varlen)
    assert layer.status() == B.LLAMA_OK
    rows = sample_rows(inp.cu_seqlens, per_seq, seed=inp.workload.seed,
                       max_seqs=max_seqs)
    ref = oracle.decoder_layer_rows(synth.to_f64(inp.x),
                                    weights_f64(inp.weights), s,
                                    inp.positions, inp.cu_seqlens, rows)
    st = layer.stages(inp.tokens)
    idx = torch.as_tensor(rows, device="cuda")
    assert_stage_close(to_f64(st["attn"][idx]), ref["attn"], s.dtype, "attn")
    assert_stage_close(to_f64(st["h"][idx]), ref["h"], s.dtype, "h")
    assert_stage_close(to_f64(st["act"][idx]), ref["act"], s.dtype, "act")
    assert_close(to_f64(out[idx]), ref["out"], s.dtype, "out")
    # every output row is finite (rows the oracle did not recompute included)
    assert torch.isfinite(out.float()).all()
    layer.close()


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
