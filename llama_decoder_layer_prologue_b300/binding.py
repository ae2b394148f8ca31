"""ctypes binding of libllama_layer.so, one Python function per C entry point
(same names, argument marshalling only; every step runs in the library).

Pointers are passed as integers (device addresses, e.g. ``tensor.data_ptr()``),
streams as ``cudaStream_t`` integers (``torch.cuda.current_stream().cuda_stream``).
A negative return code raises ``LlamaError``; ``llama_layer_status`` returns
the code instead.  Loading fails loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libllama_layer.so")

LLAMA_OK = 0
LLAMA_ERR_INVALID_ARG = -1
LLAMA_ERR_UNSUPPORTED_SHAPE = -2
LLAMA_ERR_WORKSPACE_TOO_SMALL = -3
LLAMA_ERR_CUDA = -4
LLAMA_ERR_DEVICE_TIMEOUT = -5
LLAMA_ERR_DEVICE_BAD_INPUT = -6
LLAMA_ERR_UNSUPPORTED_DEVICE = -7

LLAMA_HOST_MAX_CHUNKS = 8  # groups of llama_layer_forward_host

LLAMA_DTYPE_F32 = 0
LLAMA_DTYPE_BF16 = 1
LLAMA_ROPE_NONE = 0
LLAMA_ROPE_LLAMA3 = 1
LLAMA_ROPE_LINEAR = 2
LLAMA_ROPE_DYNAMIC_NTK = 3
LLAMA_WS_NUM = 4
LLAMA_LONG_CHUNK = 16
LLAMA_MAX_STAGES = 16
LLAMA_MAX_TIMED_CALLS = 4096

# Every symbol include/llama_layer.h declares.
EXPORTS = (
    "llama_layer_packed_bytes", "llama_layer_init",
    "llama_layer_workspace_bytes", "llama_layer_forward", "llama_layer_decode",
    "llama_layer_status", "llama_layer_workspace_offsets",
    "llama_layer_destroy", "llama_layer_strerror", "llama_gemm_bf16",
    "llama_layer_set_timing", "llama_layer_stage_times",
    "llama_layer_launch_count", "llama_gemm_bf16_streamk_static",
    "llama_layer_forward_host", "llama_layer_forward_cached",
    "llama_selftest_bounded_waits", "llama_rope_inv_freq", "llama_rmsnorm_bf16",
    "llama_gemm_status", "llama_layer_backward_workspace_bytes", "llama_layer_backward",
    "llama_layer_forward_train", "llama_layer_backward_saved",
)


class llama_layer_config(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("intermediate", ctypes.c_int), ("rms_eps", ctypes.c_float),
        ("rope_base", ctypes.c_double), ("rope_scaling", ctypes.c_int),
        ("rope_factor", ctypes.c_double),
        ("rope_low_freq_factor", ctypes.c_double),
        ("rope_high_freq_factor", ctypes.c_double),
        ("rope_original_max_pos", ctypes.c_int),
        ("max_position", ctypes.c_int), ("dtype", ctypes.c_int),
    ]


class llama_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_qkv", "w_o", "w_gate_up", "w_down", "g_in", "g_post")]


class llama_layer_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("dw_qkv", "dw_o", "dw_gate_up", "dw_down", "dg_in", "dg_post")]


class LlamaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {strerror(code)} ({code})")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """Loads the library once; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m llama_decoder_layer_prologue_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "llama_layer_packed_bytes": (_I, [ctypes.POINTER(llama_layer_config),
                                          ctypes.POINTER(_SZ)]),
        "llama_layer_init": (_I, [ctypes.POINTER(llama_layer_config),
                                  ctypes.POINTER(llama_layer_weights), _P, _SZ,
                                  _P, ctypes.POINTER(_P)]),
        "llama_layer_workspace_bytes": (_I, [_P, _I, _I, _I,
                                             ctypes.POINTER(_SZ)]),
        "llama_layer_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ,
                                     _P]),
        "llama_layer_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _SZ,
                                    _P]),
        "llama_layer_status": (_I, [_P, _P]),
        "llama_layer_workspace_offsets": (_I, [_P, _I, _I,
                                               ctypes.POINTER(_SZ)]),
        "llama_layer_destroy": (None, [_P]),
        "llama_layer_strerror": (ctypes.c_char_p, [_I]),
        "llama_gemm_bf16": (_I, [_P, _P, _P, _I, _I, _I, _P]),
        "llama_layer_set_timing": (_I, [_P, _I]),
        "llama_layer_stage_times": (_I, [_P, _I, _I,
                                         ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_char_p),
                                         ctypes.POINTER(_I)]),
        "llama_layer_launch_count": (_I, [_P]),
        "llama_gemm_bf16_streamk_static": (_I, [_P, _P, _P, _I, _I, _I, _P]),
        "llama_layer_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                          _P, _SZ, _P]),
        "llama_layer_forward_cached": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P,
                                            _SZ, _P]),
        "llama_selftest_bounded_waits": (_I, [ctypes.POINTER(_I), _P]),
        "llama_rope_inv_freq": (_I, [ctypes.POINTER(llama_layer_config),
                                     ctypes.POINTER(ctypes.c_double)]),
        "llama_rmsnorm_bf16": (_I, [_P, _P, _P, _I, _I, ctypes.c_float, _P]),
        "llama_gemm_status": (_I, [_P]),
        "llama_layer_backward_workspace_bytes": (_I, [_P, _I, ctypes.POINTER(_SZ)]),
        "llama_layer_backward": (_I, [_P, ctypes.POINTER(llama_layer_weights), _P, _P, _P,
                                      ctypes.POINTER(llama_layer_grads), _P, _P, _I, _I,
                                      _I, _P, _SZ, _P]),
        "llama_layer_forward_train": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
        "llama_layer_backward_saved": (_I, [_P, ctypes.POINTER(llama_layer_weights), _P, _P,
                                            _P, ctypes.POINTER(llama_layer_grads), _P, _P,
                                            _I, _I, _I, _P, _SZ, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(fn: str, rc: int) -> None:
    if rc != LLAMA_OK:
        raise LlamaError(fn, rc)


def strerror(code: int) -> str:
    return lib().llama_layer_strerror(code).decode()


llama_layer_strerror = strerror


def llama_layer_packed_bytes(cfg: llama_layer_config) -> int:
    n = _SZ()
    _check("llama_layer_packed_bytes",
           lib().llama_layer_packed_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def llama_layer_init(cfg: llama_layer_config, weights: llama_layer_weights,
                     packed: int, packed_bytes: int, stream: int) -> int:
    h = _P()
    _check("llama_layer_init",
           lib().llama_layer_init(ctypes.byref(cfg), ctypes.byref(weights),
                                  packed, packed_bytes, stream,
                                  ctypes.byref(h)))
    return h.value


def llama_layer_workspace_bytes(layer: int, max_tokens: int,
                                decode_batch: int = 0,
                                decode_max_seq: int = 0) -> int:
    n = _SZ()
    _check("llama_layer_workspace_bytes",
           lib().llama_layer_workspace_bytes(layer, max_tokens, decode_batch,
                                             decode_max_seq, ctypes.byref(n)))
    return n.value


def llama_layer_forward(layer: int, x: int, out: int, position_ids: int | None,
                        cu_seqlens: int | None, n_seq: int, seq_len: int,
                        total_tokens: int, workspace: int,
                        workspace_bytes: int, stream: int) -> None:
    _check("llama_layer_forward",
           lib().llama_layer_forward(layer, x, out, position_ids, cu_seqlens,
                                     n_seq, seq_len, total_tokens, workspace,
                                     workspace_bytes, stream))


def llama_layer_forward_host(layer: int, x_host: int, out_host: int, x_dev: int,
                             out_dev: int, cu_seqlens: int | None, n_seq: int,
                             seq_len: int, total_tokens: int, chunks: int,
                             workspace: int, workspace_bytes: int,
                             stream: int) -> None:
    _check("llama_layer_forward_host",
           lib().llama_layer_forward_host(layer, x_host, out_host, x_dev, out_dev,
                                          cu_seqlens, n_seq, seq_len, total_tokens,
                                          chunks, workspace, workspace_bytes, stream))


def llama_layer_forward_cached(layer: int, x: int, out: int, cache_k: int,
                               cache_v: int, start_pos: int, batch: int,
                               seq_tokens: int, max_seq: int, workspace: int,
                               workspace_bytes: int, stream: int) -> None:
    _check("llama_layer_forward_cached",
           lib().llama_layer_forward_cached(layer, x, out, cache_k, cache_v, start_pos,
                                            batch, seq_tokens, max_seq, workspace,
                                            workspace_bytes, stream))


def llama_rope_inv_freq(cfg: "llama_layer_config", head_dim: int) -> list[float]:
    """The layer's RoPE inverse frequencies (host only, no device needed)."""
    out = (ctypes.c_double * (head_dim // 2))()
    _check("llama_rope_inv_freq", lib().llama_rope_inv_freq(ctypes.byref(cfg), out))
    return list(out)


def llama_rmsnorm_bf16(x: int, g: int, out: int, rows: int, hidden: int, eps: float,
                       stream: int) -> None:
    _check("llama_rmsnorm_bf16", lib().llama_rmsnorm_bf16(x, g, out, rows, hidden, eps,
                                                          stream))


def llama_selftest_bounded_waits(stream: int) -> tuple[int, int, int]:
    """(mbarrier wait completed, flag wait completed, status word)."""
    obs = (_I * 3)()
    _check("llama_selftest_bounded_waits", lib().llama_selftest_bounded_waits(obs, stream))
    return tuple(obs)


def llama_layer_decode(layer: int, x: int, out: int, cache_k: int,
                       cache_v: int, start_pos: int, batch: int, max_seq: int,
                       workspace: int, workspace_bytes: int,
                       stream: int) -> None:
    _check("llama_layer_decode",
           lib().llama_layer_decode(layer, x, out, cache_k, cache_v, start_pos,
                                    batch, max_seq, workspace,
                                    workspace_bytes, stream))


def llama_layer_status(layer: int, stream: int) -> int:
    return lib().llama_layer_status(layer, stream)


def llama_layer_workspace_offsets(layer: int, tokens: int,
                                  decode: int = 0) -> list[int]:
    arr = (_SZ * LLAMA_WS_NUM)()
    _check("llama_layer_workspace_offsets",
           lib().llama_layer_workspace_offsets(layer, tokens, decode, arr))
    return list(arr)


def llama_layer_destroy(layer: int) -> None:
    lib().llama_layer_destroy(layer)


def llama_layer_set_timing(layer: int, ring_calls: int) -> None:
    _check("llama_layer_set_timing",
           lib().llama_layer_set_timing(layer, int(ring_calls)))


def llama_layer_stage_times(layer: int, call: int = 0) -> list[tuple[str, float]]:
    """[(stage name, ms)] of recorded call ``call`` (0 = the most recent)."""
    ms = (ctypes.c_float * LLAMA_MAX_STAGES)()
    names = (ctypes.c_char_p * LLAMA_MAX_STAGES)()
    n = _I()
    _check("llama_layer_stage_times",
           lib().llama_layer_stage_times(layer, call, LLAMA_MAX_STAGES, ms,
                                         names, ctypes.byref(n)))
    return [(names[i].decode(), float(ms[i])) for i in range(n.value)]


def llama_layer_launch_count(layer: int) -> int:
    rc = lib().llama_layer_launch_count(layer)
    if rc < 0:
        raise LlamaError("llama_layer_launch_count", rc)
    return rc


def llama_gemm_bf16(A: int, B: int, D: int, M: int, N: int, K: int,
                    stream: int) -> None:
    _check("llama_gemm_bf16", lib().llama_gemm_bf16(A, B, D, M, N, K, stream))


def llama_layer_backward_workspace_bytes(layer: int, max_tokens: int) -> int:
    n = _SZ()
    _check("llama_layer_backward_workspace_bytes",
           lib().llama_layer_backward_workspace_bytes(layer, max_tokens, ctypes.byref(n)))
    return n.value


def llama_layer_backward(layer: int, weights: llama_layer_weights, x: int, dout: int,
                         dx: int, grads: llama_layer_grads, position_ids, cu_seqlens,
                         n_seq: int, seq_len: int, total_tokens: int, workspace: int,
                         workspace_bytes: int, stream: int) -> None:
    _check("llama_layer_backward",
           lib().llama_layer_backward(layer, ctypes.byref(weights), x, dout, dx,
                                      ctypes.byref(grads), position_ids, cu_seqlens,
                                      n_seq, seq_len, total_tokens, workspace,
                                      workspace_bytes, stream))


def llama_layer_forward_train(layer: int, x: int, out: int, position_ids, cu_seqlens,
                              n_seq: int, seq_len: int, total_tokens: int, workspace: int,
                              workspace_bytes: int, stream: int) -> None:
    _check("llama_layer_forward_train",
           lib().llama_layer_forward_train(layer, x, out, position_ids, cu_seqlens, n_seq,
                                           seq_len, total_tokens, workspace,
                                           workspace_bytes, stream))


def llama_layer_backward_saved(layer: int, weights: llama_layer_weights, x: int, dout: int,
                               dx: int, grads: llama_layer_grads, position_ids, cu_seqlens,
                               n_seq: int, seq_len: int, total_tokens: int, workspace: int,
                               workspace_bytes: int, stream: int) -> None:
    _check("llama_layer_backward_saved",
           lib().llama_layer_backward_saved(layer, ctypes.byref(weights), x, dout, dx,
                                            ctypes.byref(grads), position_ids, cu_seqlens,
                                            n_seq, seq_len, total_tokens, workspace,
                                            workspace_bytes, stream))


def llama_gemm_status(stream: int) -> int:
    """Synchronises the stream and returns (and clears) the standalone GEMMs'
    device status: LLAMA_OK or a negative code."""
    return lib().llama_gemm_status(stream)


def llama_gemm_bf16_streamk_static(A: int, B: int, D: int, M: int, N: int,
                                   K: int, stream: int) -> None:
    """Stream-K GEMM whose partial sums live in the library's own fixed
    device array (no caller workspace, no allocation)."""
    _check("llama_gemm_bf16_streamk_static",
           lib().llama_gemm_bf16_streamk_static(A, B, D, M, N, K, stream))
