"""The C-ABI library loads, exports every symbol the header declares, and its
host-only entry points validate arguments (no GPU needed)."""

import ctypes
import os
import re
import subprocess

import pytest

from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import make_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "llama_layer.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(
        r"^\s*(?:LLAMA_API\s+)?(?:const\s+)?[a-z_0-9]+\s*\*?\s*(llama_[a-z_0-9]+)\s*\(", text,
        flags=re.M)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(B.EXPORTS)


def test_header_constants_match_binding():
    # every integer #define of the header that the binding names has the
    # header's value
    defs = dict(re.findall(r"^#define\s+(LLAMA_[A-Z0-9_]+)\s+\(?(-?\d+)\)?",
                           open(HEADER).read(), flags=re.M))
    named = {k: v for k, v in vars(B).items() if k.startswith("LLAMA_") and
             isinstance(v, int)}
    assert "LLAMA_HOST_MAX_CHUNKS" in named
    for k, v in named.items():
        assert k in defs, k
        assert int(defs[k]) == v, k


def test_library_exports_every_declared_symbol():
    L = B.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(declared_functions()) <= exported
    # nothing but the ABI (and no C++ symbols) leaks out of the library
    ours = {s for s in exported if not s.startswith("_")}
    assert ours == set(declared_functions()), ours ^ set(declared_functions())


def test_library_is_built_for_sm103a():
    # the build compiles every source for sm_103a alone (no PTX for other
    # targets, no JIT fallback)
    from llama_decoder_layer_prologue_b300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert all(f != "-arch" and not f.startswith("--gpu-architecture")
               for f in build.FLAGS)


def cfg_of(name):
    return make_config(synth.WORKLOADS[name].shape)


def test_packed_bytes_cover_the_weights():
    for name in ("tiny", "1b", "8b"):
        s = synth.WORKLOADS[name].shape
        es = 2 if s.dtype == "bf16" else 4
        n = B.llama_layer_packed_bytes(cfg_of(name))
        weights = (s.n_qkv * s.hidden + s.hidden * s.q_size +
                   3 * s.intermediate * s.hidden) * es
        table = 2 * s.max_position * (s.head_dim // 2) * 4
        assert weights + table <= n <= weights + table + 64 * 256


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, B.LLAMA_ERR_UNSUPPORTED_SHAPE),
    ("n_kv_heads", 3, B.LLAMA_ERR_UNSUPPORTED_SHAPE),
    ("hidden", 100, B.LLAMA_ERR_UNSUPPORTED_SHAPE),
    ("intermediate", 0, B.LLAMA_ERR_INVALID_ARG),
    ("rms_eps", 0.0, B.LLAMA_ERR_INVALID_ARG),
    ("rope_base", 1.0, B.LLAMA_ERR_INVALID_ARG),
    ("rope_scaling", 7, B.LLAMA_ERR_UNSUPPORTED_SHAPE),
    ("dtype", 5, B.LLAMA_ERR_UNSUPPORTED_SHAPE),
    ("max_position", 0, B.LLAMA_ERR_INVALID_ARG),
])
def test_bad_configs_are_rejected(field, value, code):
    cfg = cfg_of("1b")
    setattr(cfg, field, value)
    with pytest.raises(B.LlamaError) as e:
        B.llama_layer_packed_bytes(cfg)
    assert e.value.code == code


def test_llama3_factors_are_checked():
    cfg = cfg_of("8b")
    cfg.rope_high_freq_factor = cfg.rope_low_freq_factor
    with pytest.raises(B.LlamaError) as e:
        B.llama_layer_packed_bytes(cfg)
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG


@pytest.mark.parametrize("scaling,factor,max_position,d", [
    (B.LLAMA_ROPE_NONE, 1.0, 4096, 64), (B.LLAMA_ROPE_LLAMA3, 8.0, 8192, 128),
    (B.LLAMA_ROPE_LINEAR, 4.0, 4096, 64), (B.LLAMA_ROPE_LINEAR, 2.5, 4096, 128),
    (B.LLAMA_ROPE_DYNAMIC_NTK, 4.0, 16384, 64),  # beyond the original 8192
    (B.LLAMA_ROPE_DYNAMIC_NTK, 2.0, 12000, 128),
    (B.LLAMA_ROPE_DYNAMIC_NTK, 4.0, 8192, 64),  # within it: unscaled
])
def test_library_rope_table_matches_the_oracle(scaling, factor, max_position, d):
    # the cos / sin table the layer uploads comes from these frequencies,
    # computed on the host in double precision
    import oracle
    s = synth.LayerShape(hidden=256, n_heads=4, n_kv_heads=2, head_dim=d,
                         intermediate=256, rms_eps=1e-5, rope_base=500000.0,
                         rope_scaling=scaling, rope_factor=factor,
                         rope_low_freq_factor=1.0, rope_high_freq_factor=4.0,
                         rope_original_max_pos=8192, max_position=max_position)
    got = B.llama_rope_inv_freq(make_config(s), d)
    import numpy as np
    np.testing.assert_allclose(got, oracle.layer_inv_freq(s), rtol=1e-13, atol=0)


@pytest.mark.parametrize("scaling,factor", [(B.LLAMA_ROPE_LINEAR, 0.0),
                                            (B.LLAMA_ROPE_DYNAMIC_NTK, 0.5)])
def test_rope_scaling_factors_are_checked(scaling, factor):
    cfg = cfg_of("1b")
    cfg.rope_scaling, cfg.rope_factor = scaling, factor
    with pytest.raises(B.LlamaError) as e:
        B.llama_layer_packed_bytes(cfg)
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG


def test_init_rejects_null_weights_before_touching_a_device():
    cfg = cfg_of("tiny")
    w = B.llama_layer_weights()
    with pytest.raises(B.LlamaError) as e:
        B.llama_layer_init(cfg, w, 256, 1 << 20, 0)
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG


def test_null_handles_are_rejected():
    L = B.lib()
    assert L.llama_layer_forward(None, None, None, None, None, 1, 1, 1, None,
                                 0, None) == B.LLAMA_ERR_INVALID_ARG
    assert L.llama_layer_decode(None, None, None, None, None, None, 1, 1, None,
                                0, None) == B.LLAMA_ERR_INVALID_ARG
    assert L.llama_layer_forward_host(None, None, None, None, None, None, 1, 1, 1, 0,
                                      None, 0, None) == B.LLAMA_ERR_INVALID_ARG
    assert L.llama_layer_forward_cached(None, None, None, None, None, None, 1, 1, 1,
                                        None, 0, None) == B.LLAMA_ERR_INVALID_ARG
    assert L.llama_layer_status(None, None) == B.LLAMA_ERR_INVALID_ARG
    assert L.llama_layer_forward_train(None, None, None, None, None, 1, 1, 1, None, 0,
                                       None) == B.LLAMA_ERR_INVALID_ARG
    w, g = B.llama_layer_weights(), B.llama_layer_grads()
    for f in (L.llama_layer_backward, L.llama_layer_backward_saved):
        assert f(None, ctypes.byref(w), None, None, None, ctypes.byref(g), None, None, 1, 1,
                 1, None, 0, None) == B.LLAMA_ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert L.llama_layer_workspace_bytes(None, 1, 0, 0, ctypes.byref(n)) == \
        B.LLAMA_ERR_INVALID_ARG
    L.llama_layer_destroy(None)


def test_gemm_argument_checks():
    with pytest.raises(B.LlamaError) as e:
        B.llama_gemm_bf16(256, 256, 256, 128, 48, 64, 0)  # N % 32 != 0
    assert e.value.code == B.LLAMA_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(B.LlamaError) as e:
        B.llama_gemm_bf16(258, 256, 256, 128, 64, 64, 0)  # misaligned A
    assert e.value.code == B.LLAMA_ERR_INVALID_ARG


def test_strerror_covers_every_code():
    for code in range(0, -8, -1):
        assert B.strerror(code) != "unknown error"
    assert B.strerror(-99) == "unknown error"
