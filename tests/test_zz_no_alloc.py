"""llama_gemm_bf16_streamk_static: the GEMM entry point that needs no device
memory from its caller besides A, B and D.

It is meant for callers that cannot call cudaMalloc where they run the GEMM
(an engine that has reserved all device memory for its own pool, or a
latency-critical loop where cudaMalloc / cudaFree could synchronise the
device).  Its stream-K partial sums live in a fixed 16 MiB array that the
library defines in device memory; these tests check, through the C ABI, that
two calls in a row (sharing that array) give the same result as the
workspace-free llama_gemm_bf16 within the GEMM tests' tolerance, and that a
call too large for the array is refused before anything is launched.

The file name makes pytest collect it last.
"""

import numpy as np
import pytest
import torch

from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = synth.bf16_round_bits(rng.standard_normal((M, K), dtype=np.float32))
    b = synth.bf16_round_bits(0.05 * rng.standard_normal((N, K), dtype=np.float32))
    return a, b


def _bound(ref, K):
    # the GEMM tests' bound: bf16 output rounding plus fp32 accumulation
    return 2.0 ** -8 * np.abs(ref) + 1e-3 * np.sqrt(K) * 0.05


def test_two_calls_match_llama_gemm_bf16():
    st = torch.cuda.current_stream().cuda_stream
    # decode-like shapes: weight rows x a few tokens; the second call is
    # smaller in M and K and larger in N, so it reuses the shared array with
    # a different tile / slot layout
    for i, (M, N, K) in enumerate([(6144, 64, 4096), (4096, 96, 1024)]):
        a, b = _operands(M, N, K, seed=11 + i)
        A, Bm = to_device(a), to_device(b)
        ref_dev = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.llama_gemm_bf16(A.data_ptr(), Bm.data_ptr(), ref_dev.data_ptr(), M, N, K, st)
        B.llama_gemm_bf16_streamk_static(A.data_ptr(), Bm.data_ptr(), got.data_ptr(),
                                         M, N, K, st)
        torch.cuda.synchronize()
        g = got.float().cpu().numpy().astype(np.float64)
        r = ref_dev.float().cpu().numpy().astype(np.float64)
        exact = synth.to_f64(a) @ synth.to_f64(b).T
        assert np.all(np.isfinite(g))
        bound = _bound(exact, K)
        assert np.all(np.abs(g - exact) <= bound), f"call {i}: vs fp64"
        assert np.all(np.abs(g - r) <= 2 * bound), f"call {i}: vs llama_gemm_bf16"
        assert B.llama_gemm_status(st) == B.LLAMA_OK


@pytest.mark.parametrize("M,N,K", [(300, 8, 256), (129, 40, 64), (1024, 200, 512)])
def test_ragged_shapes_match_fp64(M, N, K):
    """Ragged M (rows past the last full tile are out of bounds for the TMA
    loads and skipped by the reduction), N below the 64-column tile, and the
    256-column tile within the array's limit."""
    st = torch.cuda.current_stream().cuda_stream
    a, b = _operands(M, N, K, seed=M + N + K)
    A, Bm = to_device(a), to_device(b)
    for call in range(2):
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.llama_gemm_bf16_streamk_static(A.data_ptr(), Bm.data_ptr(), got.data_ptr(),
                                         M, N, K, st)
        assert B.llama_gemm_status(st) == B.LLAMA_OK
        g = got.float().cpu().numpy().astype(np.float64)
        exact = synth.to_f64(a) @ synth.to_f64(b).T
        assert np.all(np.isfinite(g)), f"call {call}"
        assert np.all(np.abs(g - exact) <= _bound(exact, K)), f"call {call}"


def test_too_large_for_the_array_is_refused():
    st = torch.cuda.current_stream().cuda_stream
    M, N, K = 6144, 256, 4096  # partials of 48 tiles x >= 4 slots x 128 x 256
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    Bm = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    D = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.LlamaError) as e:
        B.llama_gemm_bf16_streamk_static(A.data_ptr(), Bm.data_ptr(), D.data_ptr(),
                                         M, N, K, st)
    assert e.value.code == B.LLAMA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((D == 7.0).all())
