"""fp64 CPU oracle for one Llama-style decoder layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library: it takes numpy float64 arrays (the workload's stored bf16 / fp32
values converted exactly) and computes the layer straight from the formulas on
the pages it cites, with no intermediate rounding.

The layer's backward pass (``oracle.backward``) is pinned to torch.autograd
of a separately written float64 forward and to finite differences.

Every function is pinned by ``tests/test_oracle_*.py`` to closed forms,
invariants, library routines or brute force (none is "parity unpinned").
"""

from .layer import (  # noqa: F401
    rms_norm,
    rope_inv_freq,
    llama3_scale_inv_freq,
    linear_scale_inv_freq,
    dynamic_ntk_base,
    rope_cos_sin,
    rotate_half,
    apply_rope,
    repeat_kv,
    causal_attention,
    silu,
    swiglu_mlp,
    decoder_layer,
    decoder_layer_rows,
    decoder_layer_decode,
    decoder_layer_cached,
    model_forward,
    layer_inv_freq,
)
