"""The tcgen05 / TMA GEMM building block (llama_gemm_bf16) against an fp64
matmul of the same bf16 operands, on shapes with ragged M and several
K-slices / tiles."""

import numpy as np
import pytest
import torch

from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64), (128, 256, 128), (1, 32, 8), (300, 512, 192),
    (1000, 768, 4096), (4096, 3072, 2048), (257, 6144, 4096),
])
def test_gemm_matches_fp64(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a = synth.bf16_round_bits(rng.standard_normal((M, K), dtype=np.float32))
    b = synth.bf16_round_bits(
        0.05 * rng.standard_normal((N, K), dtype=np.float32))
    A, Bm = to_device(a), to_device(b)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.llama_gemm_bf16(A.data_ptr(), Bm.data_ptr(), D.data_ptr(), M, N, K,
                      torch.cuda.current_stream().cuda_stream)
    assert B.llama_gemm_status(torch.cuda.current_stream().cuda_stream) == B.LLAMA_OK
    ref = synth.to_f64(a) @ synth.to_f64(b).T
    got = D.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    # bf16 output rounding (2^-9 relative) plus fp32 accumulation
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.sqrt(K) * 0.05)
