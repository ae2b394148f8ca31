"""Seeded synthetic inputs for the decoder-layer workloads.

This module only draws random numbers and stores them; it holds none of the
layer's arithmetic.  Both the CUDA path (through the tests and the bench) and
the fp64 oracle are fed from the arrays it returns, so the two sides always see
the same bytes.

Recipe (every workload):
  * x ~ N(0, 1); linear weights ~ N(0, 0.02); RMSNorm weights ~ 1 + N(0, 0.1);
    KV-cache rows ~ N(0, 1).
  * Draw order inside one workload: x, W_qkv, W_o, W_gate_up, W_down, g_in,
    g_post, then the varlen lengths or the decode start positions, then the
    cache.  Each of these draws gets its own child of
    ``SeedSequence(1000 + workload index)``; a large tensor is filled in fixed
    chunks of ``_CHUNK`` elements, chunk ``j`` drawing from the ``j``-th child
    of the tensor's seed, so the values do not depend on how many threads fill
    them.
  * Values are drawn as float32 and scaled in float32.  bf16 workloads store
    them rounded to bf16 with round-to-nearest-even (raw ``uint16`` bit
    patterns); the fp32 workload stores the float32 values.
  * Varlen: lengths ~ U{128..1024} until their sum reaches the token budget;
    the last length is cut so the sum is exact.  Positions restart at 0 in
    every sequence.
  * Decode: start_pos ~ U{512..8191}.  A cache of 8192 rows can take the new
    token's row only at an index <= 8191, so the upper bound 8192 given for
    this workload is read as the cache length.  Rows [0, start_pos) hold
    N(0, 1) values taken to be already-rotated keys / values; the other rows
    are zero here (tests poison them with NaN).  Chunked (seq_tokens > 1):
    start_pos ~ U{512..8192 - seq_tokens}, so every chunk ends in the cache.
  * Backward pass: the incoming gradient dL/d(out) [T, hidden] ~ N(0, 1),
    drawn from ``SeedSequence(5000 + workload index)`` (``make_dout``).
  * Model (stacked layers): x and the first layer's weights are the
    workload's own draws; layer l > 0 draws its weights as the same workload
    with index + 1000 l; the final RMSNorm weight ~ 1 + N(0, 0.1) and the
    output projection [vocab, hidden] ~ N(0, 0.02) draw from the children of
    ``SeedSequence(7000 + workload index)``.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 22


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Dimensions and RoPE settings of one decoder layer."""

    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    rms_eps: float
    rope_base: float
    rope_scaling: int  # 0 = none, 1 = Llama3 piecewise
    rope_factor: float = 1.0
    rope_low_freq_factor: float = 1.0
    rope_high_freq_factor: float = 4.0
    rope_original_max_pos: int = 8192
    max_position: int = 8192
    dtype: str = "bf16"  # "bf16" or "fp32"

    @property
    def q_size(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_size(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def n_qkv(self) -> int:
        return self.q_size + 2 * self.kv_size


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int  # seed = 1000 + index
    shape: LayerShape
    kind: str  # "padded", "varlen" or "decode"
    batch: int = 1
    seq: int = 0  # padded: sequence length
    total_tokens: int = 0  # varlen: token budget
    min_len: int = 128
    max_len: int = 1024
    max_seq: int = 8192  # decode: cache rows per sequence
    min_start: int = 512
    seq_tokens: int = 1  # decode: new tokens per sequence (> 1: chunked prefill)

    @property
    def seed(self) -> int:
        return 1000 + self.index


_SHAPE_8B = LayerShape(
    hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, intermediate=14336,
    rms_eps=1e-5, rope_base=500000.0, rope_scaling=1, rope_factor=8.0,
    rope_low_freq_factor=1.0, rope_high_freq_factor=4.0,
    rope_original_max_pos=8192, max_position=8192)

WORKLOADS = {
    "tiny": Workload(
        "tiny", 0,
        LayerShape(hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
                   intermediate=512, rms_eps=1e-5, rope_base=10000.0,
                   rope_scaling=0, max_position=64, dtype="fp32"),
        "padded", batch=1, seq=64),
    "1b": Workload(
        "1b", 1,
        LayerShape(hidden=2048, n_heads=32, n_kv_heads=8, head_dim=64,
                   intermediate=8192, rms_eps=1e-5, rope_base=500000.0,
                   rope_scaling=1, rope_factor=32.0, rope_low_freq_factor=1.0,
                   rope_high_freq_factor=4.0, rope_original_max_pos=8192,
                   max_position=8192),
        "padded", batch=4, seq=2048),
    "8b": Workload("8b", 2, _SHAPE_8B, "padded", batch=2, seq=4096),
    "varlen": Workload("varlen", 3, _SHAPE_8B, "varlen", total_tokens=16384),
    "decode": Workload("decode", 4, _SHAPE_8B, "decode", batch=64,
                       max_seq=8192, min_start=512),
    "chunked": Workload("chunked", 5, _SHAPE_8B, "decode", batch=16,
                        max_seq=8192, min_start=512, seq_tokens=4),
    # long chunks: the tensor-core prefill attention reads the cache
    "chunk64": Workload("chunk64", 6, _SHAPE_8B, "decode", batch=16,
                        max_seq=8192, min_start=512, seq_tokens=64),
    "chunk512": Workload("chunk512", 7, _SHAPE_8B, "decode", batch=16,
                         max_seq=8192, min_start=512, seq_tokens=512),
}


def bf16_round_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def to_f64(stored: np.ndarray) -> np.ndarray:
    """Stored workload array (bf16 bits or float32) -> float64, exactly."""
    if stored.dtype == np.uint16:
        return bf16_bits_to_f32(stored).astype(np.float64)
    return stored.astype(np.float64)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill_normal(seed: np.random.SeedSequence, n: int, mean: float, std: float,
                 dtype: str) -> np.ndarray:
    """n values mean + std * N(0,1), chunked and reproducible."""
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    n_chunks = (n + _CHUNK - 1) // _CHUNK
    kids = seed.spawn(n_chunks) if n_chunks else []

    def work(j: int) -> None:
        lo, hi = j * _CHUNK, min(n, (j + 1) * _CHUNK)
        v = np.random.Generator(np.random.PCG64(kids[j])).standard_normal(
            hi - lo, dtype=np.float32)
        v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        out[lo:hi] = bf16_round_bits(v) if dtype == "bf16" else v

    if n_chunks <= 1:
        for j in range(n_chunks):
            work(j)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(n_chunks)))
    return out


@dataclasses.dataclass
class LayerWeights:
    """Weights in the pages' nn.Linear layout ([out_features, in_features]).

    w_qkv rows are q | k | v (head-major); w_gate_up rows are gate | up.
    """

    w_qkv: np.ndarray
    w_o: np.ndarray
    w_gate_up: np.ndarray
    w_down: np.ndarray
    g_in: np.ndarray
    g_post: np.ndarray


@dataclasses.dataclass
class LayerInputs:
    workload: Workload
    x: np.ndarray  # [T, hidden]
    weights: LayerWeights
    positions: np.ndarray  # [T] int32
    cu_seqlens: np.ndarray  # [n_seq + 1] int32 (padded: multiples of seq)
    start_pos: np.ndarray | None = None  # decode: [B] int32
    cache_k: np.ndarray | None = None  # decode: [B, max_seq, Hkv, d]
    cache_v: np.ndarray | None = None

    @property
    def tokens(self) -> int:
        return self.x.shape[0]


def varlen_lengths(rng: np.random.Generator, total: int, lo: int, hi: int):
    lens = []
    acc = 0
    while acc < total:
        L = int(rng.integers(lo, hi + 1))
        lens.append(L)
        acc += L
    lens[-1] -= acc - total
    return np.asarray(lens, dtype=np.int64)


def make_inputs(w: Workload | str, with_cache: bool = True,
                x_only: bool = False) -> LayerInputs:
    """Draw every input of workload ``w`` (see the module docstring)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    s = w.shape
    kids = np.random.SeedSequence(w.seed).spawn(10)
    if w.kind == "padded":
        T = w.batch * w.seq
    elif w.kind == "varlen":
        T = w.total_tokens
    else:
        T = w.batch * w.seq_tokens
    H, I = s.hidden, s.intermediate
    x = _fill_normal(kids[0], T * H, 0.0, 1.0, s.dtype).reshape(T, H)

    def lin(k, rows, cols):
        if x_only:
            return None
        return _fill_normal(kids[k], rows * cols, 0.0, 0.02,
                            s.dtype).reshape(rows, cols)

    weights = LayerWeights(
        w_qkv=lin(1, s.n_qkv, H),
        w_o=lin(2, H, s.q_size),
        w_gate_up=lin(3, 2 * I, H),
        w_down=lin(4, H, I),
        g_in=None if x_only else _fill_normal(kids[5], H, 1.0, 0.1, s.dtype),
        g_post=None if x_only else _fill_normal(kids[6], H, 1.0, 0.1, s.dtype),
    )
    rng = np.random.Generator(np.random.PCG64(kids[7]))
    start_pos = cache_k = cache_v = None
    if w.kind == "padded":
        cu = np.arange(0, T + 1, w.seq, dtype=np.int32)
        positions = np.tile(np.arange(w.seq, dtype=np.int32), w.batch)
    elif w.kind == "varlen":
        lens = varlen_lengths(rng, T, w.min_len, w.max_len)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        positions = np.concatenate(
            [np.arange(L, dtype=np.int32) for L in lens])
    else:
        S = w.seq_tokens  # the chunk ends within the cache
        start_pos = rng.integers(w.min_start, w.max_seq - S + 1,
                                 size=w.batch).astype(np.int32)
        cu = np.arange(0, T + 1, S, dtype=np.int32)
        positions = (np.repeat(start_pos, S) +
                     np.tile(np.arange(S, dtype=np.int32), w.batch)).astype(np.int32)
        if with_cache:
            cache_k = _make_cache(kids[8], w, start_pos)
            cache_v = _make_cache(kids[9], w, start_pos)
    return LayerInputs(w, x, weights, positions, cu, start_pos, cache_k,
                       cache_v)


def make_dout(inp: LayerInputs, scale: float = 1.0) -> np.ndarray:
    """The incoming gradient of the backward pass, [T, hidden] ~ scale * N(0, 1)
    in the workload's dtype (see the module docstring)."""
    w = inp.workload
    seed = np.random.SeedSequence(5000 + w.index)
    return _fill_normal(seed, inp.tokens * w.shape.hidden, 0.0, scale,
                        w.shape.dtype).reshape(inp.tokens, w.shape.hidden)


def _make_cache(seed, w: Workload, start_pos):
    s = w.shape
    row = s.n_kv_heads * s.head_dim
    cache = np.zeros((w.batch, w.max_seq, row), dtype=np.uint16
                     if s.dtype == "bf16" else np.float32)
    kids = seed.spawn(w.batch)
    for b in range(w.batch):
        n = int(start_pos[b]) * row
        cache[b, : start_pos[b]] = _fill_normal(
            kids[b], n, 0.0, 1.0, s.dtype).reshape(int(start_pos[b]), row)
    return cache.reshape(w.batch, w.max_seq, s.n_kv_heads, s.head_dim)


def custom_workload(name: str, shape: LayerShape, kind: str, index: int = 50,
                    **kw) -> Workload:
    """A workload with the same recipe and other sizes (edge-case tests)."""
    return Workload(name, index, shape, kind, **kw)


@dataclasses.dataclass
class ModelInputs:
    """Inputs of a stack of decoder layers, the final RMSNorm and the output
    projection (the model-level workload)."""
    first: LayerInputs          # x, positions, cu_seqlens and layer 0's weights
    layers: list                # LayerWeights of every layer (layers[0] is first's)
    g_final: np.ndarray         # [hidden]
    w_lm: np.ndarray            # [vocab, hidden]

    @property
    def tokens(self) -> int:
        return self.first.tokens


def make_model_inputs(w: Workload | str, n_layers: int, vocab: int) -> ModelInputs:
    """Draw the inputs of an n_layers stack with a vocab-wide output
    projection on workload ``w``'s tokens (see the module docstring)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    first = make_inputs(w)
    layers = [first.weights]
    for l in range(1, n_layers):
        wl = dataclasses.replace(w, index=w.index + 1000 * l)
        layers.append(make_inputs(wl, with_cache=False).weights)
    s = w.shape
    kids = np.random.SeedSequence(7000 + w.index).spawn(2)
    g_final = _fill_normal(kids[0], s.hidden, 1.0, 0.1, s.dtype)
    w_lm = _fill_normal(kids[1], vocab * s.hidden, 0.0, 0.02, s.dtype).reshape(
        vocab, s.hidden)
    return ModelInputs(first, layers, g_final, w_lm)
