"""GPU vs oracle parity through the C ABI on small shapes that still span
several tiles and ragged tails, plus the edge cases and the device-side input
checks.  Full-size workloads are in test_workloads_gpu.py."""

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

L3 = dict(rope_scaling=1, rope_factor=8.0, rope_low_freq_factor=1.0,
          rope_high_freq_factor=4.0, rope_original_max_pos=8192)


def shape(H, hq, hkv, d, I, dtype="bf16", max_position=4096, **kw):
    args = dict(rms_eps=1e-5, rope_base=500000.0, rope_scaling=0)
    args.update(kw)
    return synth.LayerShape(hidden=H, n_heads=hq, n_kv_heads=hkv, head_dim=d,
                            intermediate=I, max_position=max_position,
                            dtype=dtype, **args)


def check_forward(inp, varlen, with_positions=False, stages=True):
    s = inp.workload.shape
    layer = build_layer(inp)
    out = run_forward(layer, inp, varlen, with_positions)
    assert layer.status() == B.LLAMA_OK
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights),
                               s, inp.positions, inp.cu_seqlens)
    T = inp.tokens
    if stages:
        st = layer.stages(T)
        assert_stage_close(to_f64(st["qkv"]), oracle_qkv(ref), s.dtype, "qkv")
        assert_stage_close(to_f64(st["attn"]), ref["attn"], s.dtype, "attn")
        assert_stage_close(to_f64(st["h"]), ref["h"], s.dtype, "h")
        assert_stage_close(to_f64(st["act"]), ref["act"], s.dtype, "act")
    assert_close(to_f64(out), ref["out"], s.dtype, "out")
    layer.close()


def test_tiny_fp32_workload():
    check_forward(synth.make_inputs("tiny"), varlen=False)


@pytest.mark.parametrize("case", [
    # (name, shape, kind, kwargs)
    ("padded_ragged_llama3", shape(256, 4, 2, 64, 384, **L3), "padded",
     dict(batch=3, seq=100)),
    ("padded_d128_one_kv", shape(512, 4, 1, 128, 256), "padded",
     dict(batch=2, seq=129)),
    ("mha", shape(256, 4, 4, 64, 256), "padded", dict(batch=2, seq=65)),
    ("single_token", shape(256, 4, 2, 64, 256), "padded", dict(batch=1, seq=1)),
    # q|k|v width 320: not a multiple of the 128-row / 256-column tiles
    ("three_heads_one_kv", shape(256, 3, 1, 64, 256), "padded",
     dict(batch=2, seq=70)),
    ("varlen_with_len1", shape(512, 8, 2, 64, 512, **L3), "varlen",
     dict(total_tokens=700, min_len=1, max_len=300)),
    # 8 query heads per kv head: 16 positions per 128-row attention tile
    ("gqa8", shape(512, 8, 1, 64, 256, **L3), "padded", dict(batch=2, seq=90)),
    # 16 query heads per kv head (the largest ratio the library takes)
    ("gqa16", shape(1024, 16, 1, 64, 256), "padded", dict(batch=1, seq=77)),
    # head_dim 128 packed sequences, many shorter than a query tile
    ("varlen_d128_short", shape(512, 4, 2, 128, 256, **L3), "varlen",
     dict(total_tokens=400, min_len=1, max_len=40)),
    # linear and dynamic NTK RoPE scaling (table-only variants)
    ("linear_rope", shape(256, 4, 2, 64, 256, rope_scaling=2, rope_factor=4.0),
     "padded", dict(batch=2, seq=100)),
    ("dynamic_ntk_rope", shape(256, 4, 2, 64, 256, rope_scaling=3, rope_factor=2.0,
                               rope_original_max_pos=1024, max_position=4096),
     "varlen", dict(total_tokens=600, min_len=1, max_len=400)),
    # GEMMs run as single CTAs where CTA pairs would take a round more (a
    # small odd M-tile count), and then fill a partly idle last round with
    # the split-tile phase (tiles cut between two CTAs; 64 K-blocks at
    # least): here QKV (13 M-tiles x 32 N-tiles) ...
    ("split_tiles_qkv", shape(4096, 32, 16, 128, 1024), "padded",
     dict(batch=2, seq=832)),
    # ... and gate_up (3 M-tiles x 76 N-tiles, packed sequences)
    ("split_tiles_gate_up_varlen", shape(4096, 8, 2, 64, 9728, **L3), "varlen",
     dict(total_tokens=300, min_len=1, max_len=200)),
    # CTA pairs on a ragged last M-tile with packed sequences
    ("pairs_down_varlen", shape(512, 8, 2, 64, 4096, **L3), "varlen",
     dict(total_tokens=12700, min_len=1, max_len=1000)),
], ids=lambda case: case[0])
def test_small_bf16_forward(case):
    name, s, kind, kw = case
    w = synth.custom_workload(name, s, kind, **kw)
    check_forward(synth.make_inputs(w), varlen=(kind == "varlen"))


def test_split_tiles_repeated_calls():
    # every launch must find the split-tile flags cleared by the previous one
    # and wait for its own pieces (a new epoch), call after call
    s = shape(4096, 8, 2, 64, 9728, **L3)  # gate_up: 3 x 76 tiles, split
    w = synth.custom_workload("split_rep", s, "padded", batch=3, seq=100)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights),
                               s, inp.positions, inp.cu_seqlens)
    for _ in range(3):
        out = run_forward(layer, inp, varlen=False)
        assert layer.status() == B.LLAMA_OK
        assert_close(to_f64(out), ref["out"], s.dtype, "out")
    layer.close()


@pytest.mark.parametrize("chunks", [0, 3, 6])
def test_forward_host_groups_match_the_oracle(chunks):
    # input and output in pinned host memory; groups of whole sequences are
    # copied in, run and copied out on separate streams (0: two groups here)
    s = shape(512, 8, 2, 64, 1024, **L3)
    w = synth.custom_workload("host", s, "padded", batch=6, seq=700)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    T = inp.tokens
    x_dev = to_device(inp.x)
    dev_out = run_forward(layer, inp, varlen=False).clone()
    x_h = x_dev.cpu().pin_memory()
    out_h = torch.full_like(x_h, float("nan")).pin_memory()
    stage_x = torch.empty_like(x_dev)
    stage_out = torch.empty_like(x_dev)
    layer.forward_from_host(x_h, out_h, stage_x, stage_out, n_seq=6, seq_len=700,
                            chunks=chunks)
    torch.cuda.current_stream().synchronize()
    assert layer.status() == B.LLAMA_OK
    assert layer.launch_count() > 0
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights),
                               s, inp.positions, inp.cu_seqlens)
    assert_close(to_f64(out_h), ref["out"], s.dtype, "host out")
    # the same layer on the device-resident input, up to the GEMMs' split of
    # K, which depends on a group's tile count (a bf16 ulp at most)
    d = (out_h.float() - dev_out.cpu().float()).abs()
    assert float(d.max()) <= 2.0 ** -7 * float(dev_out.float().abs().max())
    layer.close()


# (chunks, sequence lengths summing to 900 or None for drawn ones): one group,
# three, eight; empty sequences and a last group of one empty sequence (cut
# at 225 / 450 / 675 tokens: rows 0-305, 305-556, 556-900, none); a long first
# sequence that leaves the second of three groups without rows
PACKED_HOST_CASES = [
    (0, None),
    (1, None),
    (3, None),
    (8, None),
    (4, [0, 5, 0, 300, 1, 0, 250, 344, 0]),
    (8, [700, 100, 100]),
]


@pytest.mark.parametrize("chunks,lens", PACKED_HOST_CASES)
def test_forward_host_packed_batch(chunks, lens):
    # a packed batch through host buffers: the host cu_seqlens cuts it into
    # groups of whole sequences, each run on its rebased copy
    s = shape(256, 4, 2, 64, 256, **L3)
    w = synth.custom_workload("hostv", s, "varlen", total_tokens=900, min_len=1,
                              max_len=300)
    inp = synth.make_inputs(w)
    if lens is not None:
        assert sum(lens) == inp.tokens
        inp.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        inp.positions = np.concatenate(
            [np.arange(n, dtype=np.int32) for n in lens]).astype(np.int32)
    layer = build_layer(inp)
    x_h = to_device(inp.x, pin=True)
    out_h = torch.full_like(x_h, float("nan")).pin_memory()
    stage_x = torch.empty(x_h.shape, dtype=x_h.dtype, device="cuda")
    stage_out = torch.empty_like(stage_x)
    cu_h = torch.from_numpy(inp.cu_seqlens.copy())
    S = int(np.diff(inp.cu_seqlens).max())
    layer.forward_from_host(x_h, out_h, stage_x, stage_out, cu_seqlens=cu_h, seq_len=S,
                            chunks=chunks)
    torch.cuda.current_stream().synchronize()
    assert layer.status() == B.LLAMA_OK
    assert layer.launch_count() > 0
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights),
                               s, inp.positions, inp.cu_seqlens)
    assert_close(to_f64(out_h), ref["out"], s.dtype, "host out (packed)")
    # twice more on the same handle without a synchronise between the calls
    # (the second waits for the first's copy of the rebased arrays)
    out_h2 = torch.full_like(x_h, float("nan")).pin_memory()
    for o in (out_h, out_h2):
        layer.forward_from_host(x_h, o, stage_x, stage_out, cu_seqlens=cu_h,
                                seq_len=S, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    assert layer.status() == B.LLAMA_OK
    assert torch.equal(out_h2, out_h)
    layer.close()


@pytest.mark.parametrize("kind", ["varlen", "padded"])
def test_forward_host_five_groups(kind):
    # >= 16384 tokens with chunks = 0: groups cut at 1/16, 1/4, 3/4 and 15/16
    # of the tokens
    s = shape(256, 4, 2, 64, 256, **L3)
    if kind == "varlen":
        w = synth.custom_workload("host5v", s, "varlen", total_tokens=16384, min_len=1,
                                  max_len=700)
    else:
        w = synth.custom_workload("host5p", s, "padded", batch=32, seq=512)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    x_h = to_device(inp.x, pin=True)
    out_h = torch.full_like(x_h, float("nan")).pin_memory()
    stage_x = torch.empty(x_h.shape, dtype=x_h.dtype, device="cuda")
    stage_out = torch.empty_like(stage_x)
    S = int(np.diff(inp.cu_seqlens).max())
    if kind == "varlen":
        layer.forward_from_host(x_h, out_h, stage_x, stage_out,
                                cu_seqlens=torch.from_numpy(inp.cu_seqlens.copy()),
                                seq_len=S)
    else:
        layer.forward_from_host(x_h, out_h, stage_x, stage_out, n_seq=32, seq_len=S)
    torch.cuda.current_stream().synchronize()
    assert layer.status() == B.LLAMA_OK
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights),
                               s, inp.positions, inp.cu_seqlens)
    assert_close(to_f64(out_h), ref["out"], s.dtype, "host out (five groups)")
    # the whole batch on the device in one call: equal up to the GEMMs'
    # split of K, which depends on a group's tile count (a bf16 ulp at most)
    dev = run_forward(layer, inp, varlen=kind == "varlen").cpu().float()
    d = (out_h.float() - dev).abs()
    assert float(d.max()) <= 2.0 ** -7 * float(dev.abs().max())
    layer.close()


@pytest.mark.parametrize("kind", ["padded", "varlen"])
def test_forward_host_fp32(kind):
    # the fp32 layer through host buffers: rows of 4-byte values, groups of
    # whole sequences (three), the fp32 bound
    s = shape(256, 4, 2, 64, 512, dtype="fp32")
    if kind == "padded":
        w = synth.custom_workload("hostf", s, "padded", batch=3, seq=40)
    else:
        w = synth.custom_workload("hostfv", s, "varlen", total_tokens=150, min_len=1,
                                  max_len=60)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    x_h = to_device(inp.x, pin=True)
    out_h = torch.full_like(x_h, float("nan")).pin_memory()
    stage_x = torch.empty(x_h.shape, dtype=x_h.dtype, device="cuda")
    stage_out = torch.empty_like(stage_x)
    S = int(np.diff(inp.cu_seqlens).max())
    if kind == "padded":
        layer.forward_from_host(x_h, out_h, stage_x, stage_out, n_seq=3, seq_len=S, chunks=3)
    else:
        layer.forward_from_host(x_h, out_h, stage_x, stage_out,
                                cu_seqlens=torch.from_numpy(inp.cu_seqlens.copy()),
                                seq_len=S, chunks=3)
    torch.cuda.current_stream().synchronize()
    assert layer.status() == B.LLAMA_OK
    ref = oracle.decoder_layer(synth.to_f64(inp.x), weights_f64(inp.weights),
                               s, inp.positions, inp.cu_seqlens)
    assert_close(to_f64(out_h), ref["out"], s.dtype, "host out (fp32)")
    layer.close()


def test_forward_host_rejects_bad_host_cu_seqlens():
    s = shape(256, 4, 2, 64, 256, **L3)
    w = synth.custom_workload("hostbad", s, "varlen", total_tokens=64, min_len=1,
                              max_len=32)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    x_h = to_device(inp.x, pin=True)
    out_h = torch.empty_like(x_h).pin_memory()
    stage_x = torch.empty(x_h.shape, dtype=x_h.dtype, device="cuda")
    stage_out = torch.empty_like(stage_x)
    for bad in ([1, 30, 64], [0, 40, 30, 64], [0, 30, 63], [0, 10, 64]):
        cu_h = torch.tensor(bad, dtype=torch.int32)
        with pytest.raises(B.LlamaError) as e:
            layer.forward_from_host(x_h, out_h, stage_x, stage_out, cu_seqlens=cu_h,
                                    seq_len=32, chunks=2)
        assert e.value.code == B.LLAMA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        layer.forward_from_host(x_h, out_h, stage_x, stage_out,
                                cu_seqlens=to_device(inp.cu_seqlens), seq_len=32)
    assert layer.status() == B.LLAMA_OK
    layer.close()


def test_explicit_position_ids():
    s = shape(256, 4, 2, 64, 256, **L3)
    w = synth.custom_workload("pos", s, "padded", batch=2, seq=64)
    inp = synth.make_inputs(w)
    inp.positions = (inp.positions * 7 + 3).astype(np.int32)  # any positions
    check_forward(inp, varlen=False, with_positions=True)


def test_varlen_equals_padded_on_the_gpu():
    s = shape(256, 4, 2, 64, 256)
    w = synth.custom_workload("vp", s, "padded", batch=3, seq=96)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    padded = run_forward(layer, inp, varlen=False).clone()
    varlen = run_forward(layer, inp, varlen=True)
    # same tokens, same sequences: the two launch paths agree exactly
    assert torch.equal(padded, varlen)
    layer.close()


def check_decode(s, batch, max_seq, start_pos, stages=True):
    w = synth.custom_workload("dec", s, "decode", batch=batch, max_seq=max_seq,
                              min_start=0)
    inp = synth.make_inputs(w)
    inp.start_pos = np.asarray(start_pos, dtype=np.int32)
    inp.cache_k = synth._make_cache(np.random.SeedSequence(5), w, inp.start_pos)
    inp.cache_v = synth._make_cache(np.random.SeedSequence(6), w, inp.start_pos)
    layer = build_layer(inp)
    ck = to_device(poison_cache(inp.cache_k, inp.start_pos))
    cv = to_device(poison_cache(inp.cache_v, inp.start_pos))
    ck0, cv0 = ck.clone(), cv.clone()
    x = to_device(inp.x)
    sp = to_device(inp.start_pos)
    out = layer.decode(x, ck, cv, sp)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    rows = lambda b, n: (synth.to_f64(inp.cache_k[b, :n]),
                         synth.to_f64(inp.cache_v[b, :n]))
    ref = oracle.decoder_layer_decode(synth.to_f64(inp.x),
                                      weights_f64(inp.weights), s, rows,
                                      inp.start_pos)
    assert_close(to_f64(out), ref["out"], s.dtype, "decode out")
    if stages:  # the workspace holds one pass of at most 256 tokens
        st = layer.stages(batch, decode=True)
        assert_stage_close(to_f64(st["attn"]), ref["attn"], s.dtype, "decode attn")
    for b, p in enumerate(inp.start_pos):
        assert_stage_close(to_f64(ck[b, p]), ref["k_new"][b], s.dtype, "k row")
        assert_stage_close(to_f64(cv[b, p]), ref["v_new"][b], s.dtype, "v row")
        # nothing else in the cache changed (NaN rows stay NaN)
        assert torch.equal(ck[b, :p], ck0[b, :p])
        assert torch.equal(cv[b, :p], cv0[b, :p])
        assert torch.isnan(ck[b, p + 1:].float()).all()
        assert torch.isnan(cv[b, p + 1:].float()).all()
    layer.close()


def check_cached(s, batch, S, max_seq, start_pos):
    # S new tokens per sequence against the cache (chunked prefill)
    w = synth.custom_workload("chunk", s, "decode", batch=batch, max_seq=max_seq,
                              min_start=0)
    inp = synth.make_inputs(w)
    sp = np.asarray(start_pos, dtype=np.int32)
    ck_np = synth._make_cache(np.random.SeedSequence(5), w, sp)
    cv_np = synth._make_cache(np.random.SeedSequence(6), w, sp)
    rng = np.random.default_rng(17)
    x_np = synth.bf16_round_bits(rng.standard_normal((batch * S, s.hidden),
                                                     dtype=np.float32))
    layer = build_layer(inp)
    ck = to_device(poison_cache(ck_np, sp))
    cv = to_device(poison_cache(cv_np, sp))
    ck0, cv0 = ck.clone(), cv.clone()
    out = layer.forward_cached(to_device(x_np), ck, cv, to_device(sp), S)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_OK
    rows = lambda b, n: (synth.to_f64(ck_np[b, :n]), synth.to_f64(cv_np[b, :n]))
    ref = oracle.decoder_layer_cached(synth.to_f64(x_np), weights_f64(inp.weights),
                                      s, rows, sp, S)
    assert_close(to_f64(out), ref["out"], s.dtype, f"chunk out (S={S})")
    for b, p in enumerate(sp):
        new = slice(b * S, (b + 1) * S)
        assert_stage_close(to_f64(ck[b, p:p + S]), ref["k_new"][new], s.dtype, "k rows")
        assert_stage_close(to_f64(cv[b, p:p + S]), ref["v_new"][new], s.dtype, "v rows")
        assert torch.equal(ck[b, :p], ck0[b, :p])  # the prefix is untouched
        assert torch.equal(cv[b, :p], cv0[b, :p])
        assert torch.isnan(ck[b, p + S:].float()).all()  # nothing after the chunk
        assert torch.isnan(cv[b, p + S:].float()).all()
    layer.close()


@pytest.mark.parametrize("S,hq,hkv", [
    # 2 query heads per kv head: up to 8 new tokens share one split-KV tile
    (1, 4, 2), (3, 4, 2), (4, 4, 2), (8, 4, 2),
    # one head per kv head: 15 tokens in one 16-row tile
    (15, 4, 4),
    # 8 query heads per kv head: groups of 2 tokens; 4 tokens are two groups
    # (split-KV), 5 are three (the tensor-core attention over the cache)
    (4, 8, 1), (5, 8, 1),
    # 4 query heads per kv head, 12 tokens: three groups of 4 (tensor core)
    (12, 8, 2),
    # 3 query heads per kv head: groups of 5 tokens (15 of the 16 rows)
    (5, 3, 1), (7, 3, 1),
    # 16 query heads per kv head: one token a group; 2 tokens split-KV, 3 the
    # tensor core
    (2, 16, 1), (3, 16, 1),
])
def test_forward_cached_chunks(S, hq, hkv):
    s = shape(max(256, 64 * hq), hq, hkv, 64, 256, **L3)
    # includes an empty prefix and a chunk ending on the last cache row
    check_cached(s, batch=5, S=S, max_seq=300, start_pos=[0, 123, 1, 300 - S, 77])


@pytest.mark.parametrize("S,d,hq,hkv,max_seq,start_pos", [
    # the shortest long chunk, an empty prefix, a chunk ending on the last row
    (16, 64, 4, 2, 300, [0, 123, 1, 284, 77]),
    (64, 64, 8, 2, 700, [0, 600, 257, 636]),
    # a chunk that is not a multiple of the query tiles
    (200, 128, 4, 1, 1000, [0, 799, 130]),
    (512, 128, 8, 2, 1200, [0, 688, 300]),
    # 8 query heads per kv head: 16 positions per 128-row tile
    (64, 64, 8, 1, 500, [436, 5, 128]),
])
def test_forward_cached_long_chunks(S, d, hq, hkv, max_seq, start_pos):
    """Chunks of at least LLAMA_LONG_CHUNK new tokens run the tensor-core
    prefill attention over the cache; rows past each chunk are NaN and must
    neither be written nor change the result."""
    s = shape(128 * hq if d == 128 else 64 * hq, hq, hkv, d, 256, **L3)
    check_cached(s, batch=len(start_pos), S=S, max_seq=max_seq, start_pos=start_pos)


def test_forward_cached_two_passes():
    # 40 x 7 = 280 rows: passes of whole sequences (36 x 7 = 252 rows, then
    # 28); the second pass's attention sees what the first appended
    s = shape(256, 4, 2, 64, 256, **L3)
    sp = [(29 * b) % 180 for b in range(40)]
    check_cached(s, batch=40, S=7, max_seq=192, start_pos=sp)


def test_forward_cached_d128():
    s = shape(512, 8, 2, 128, 384)
    check_cached(s, batch=3, S=5, max_seq=600, start_pos=[512, 0, 37])


def test_decode_small_bf16_edges():
    s = shape(256, 4, 2, 64, 256, **L3)
    check_decode(s, batch=5, max_seq=300, start_pos=[0, 299, 1, 150, 257])


def test_decode_small_d128():
    s = shape(512, 8, 2, 128, 384)
    check_decode(s, batch=3, max_seq=520, start_pos=[513, 7, 64])


def test_decode_qkv_width_not_tile_aligned():
    s = shape(256, 3, 1, 64, 256, **L3)
    check_decode(s, batch=33, max_seq=200, start_pos=list(range(0, 198, 6)))


def test_decode_batch_128_wide_token_tile():
    # 65..128 tokens: the decode GEMMs use 128-wide token tiles
    s = shape(256, 4, 2, 64, 256, **L3)
    sp = [(7 * b) % 190 for b in range(100)]
    check_decode(s, batch=100, max_seq=192, start_pos=sp)


def test_decode_batch_above_256_is_chunked():
    # more than 256 tokens: two decode passes (256 + 44), 256-wide tiles
    s = shape(256, 4, 2, 64, 256)
    sp = [(13 * b) % 60 for b in range(300)]
    check_decode(s, batch=300, max_seq=64, start_pos=sp, stages=False)


def test_decode_tiny_fp32():
    s = synth.WORKLOADS["tiny"].shape
    s = synth.LayerShape(**{**s.__dict__, "max_position": 128})
    check_decode(s, batch=2, max_seq=100, start_pos=[63, 0])


def test_bad_cu_seqlens_are_flagged():
    s = shape(256, 4, 2, 64, 256)
    w = synth.custom_workload("bad", s, "varlen", total_tokens=300, min_len=50,
                              max_len=150)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    cu = inp.cu_seqlens.copy()
    cu[1], cu[2] = cu[2], cu[1]  # not monotone
    out = layer.forward(to_device(inp.x), cu_seqlens=to_device(cu),
                        seq_len=300)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_ERR_DEVICE_BAD_INPUT
    assert layer.status() == B.LLAMA_OK  # the word was cleared
    layer.close()


def test_bad_start_pos_is_flagged():
    s = shape(256, 4, 2, 64, 256)
    w = synth.custom_workload("dec", s, "decode", batch=2, max_seq=64,
                              min_start=0)
    inp = synth.make_inputs(w, with_cache=False)
    layer = build_layer(inp)
    ck = torch.zeros(2, 64, 2, 64, dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    sp = torch.tensor([64, -1], dtype=torch.int32, device="cuda")
    layer.decode(to_device(inp.x), ck, cv, sp)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_ERR_DEVICE_BAD_INPUT
    assert torch.count_nonzero(ck) == 0 and torch.count_nonzero(cv) == 0
    layer.close()


def test_positions_beyond_the_table_are_flagged():
    s = shape(256, 4, 2, 64, 256, max_position=64)
    w = synth.custom_workload("pos", s, "padded", batch=1, seq=32)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    pos = torch.full((32,), 64, dtype=torch.int32, device="cuda")
    layer.forward(to_device(inp.x), position_ids=pos, seq_len=32)
    torch.cuda.synchronize()
    assert layer.status() == B.LLAMA_ERR_DEVICE_BAD_INPUT
    layer.close()


def test_host_checks_launch_nothing():
    s = shape(256, 4, 2, 64, 256)
    w = synth.custom_workload("chk", s, "padded", batch=1, seq=8)
    inp = synth.make_inputs(w)
    layer = build_layer(inp)
    x = to_device(inp.x)
    out = torch.zeros_like(x)
    layer.ensure_workspace(8)
    ws = layer.workspace
    st = torch.cuda.current_stream().cuda_stream
    with pytest.raises(B.LlamaError) as e:  # workspace too small
        B.llama_layer_forward(layer.handle, x.data_ptr(), out.data_ptr(), None,
                              None, 1, 8, 8, ws.data_ptr(), 100, st)
    assert e.value.code == B.LLAMA_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(B.LlamaError) as e:  # n_seq * seq_len != T
        B.llama_layer_forward(layer.handle, x.data_ptr(), out.data_ptr(), None,
                              None, 2, 8, 8, ws.data_ptr(), ws.numel(), st)
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG
    with pytest.raises(B.LlamaError) as e:  # x aliases out
        B.llama_layer_forward(layer.handle, x.data_ptr(), x.data_ptr(), None,
                              None, 1, 8, 8, ws.data_ptr(), ws.numel(), st)
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG
    with pytest.raises(B.LlamaError) as e:  # misaligned output
        B.llama_layer_forward(layer.handle, x.data_ptr(), out.data_ptr() + 2,
                              None, None, 1, 8, 8, ws.data_ptr(), ws.numel(),
                              st)
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    layer.close()
