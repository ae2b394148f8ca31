"""Failure detection without a GPU fault: the bounded waits of the pipelined
kernels give up after their limit, report it in the status word and end the
kernel, and the context keeps working afterwards."""

import numpy as np
import pytest
import torch

from llama_decoder_layer_prologue_b300 import binding as B
from llama_decoder_layer_prologue_b300 import synth
from llama_decoder_layer_prologue_b300.layer import to_device

pytestmark = pytest.mark.gpu


def test_waits_that_cannot_complete_give_up_and_report():
    st = torch.cuda.current_stream().cuda_stream
    mbar_done, flag_done, status = B.llama_selftest_bounded_waits(st)
    assert (mbar_done, flag_done) == (0, 0)  # both waits gave up
    assert status & 1  # the timeout bit of the status word
    # the same context runs work afterwards: a GEMM through the C ABI
    rng = np.random.default_rng(3)
    a = synth.bf16_round_bits(rng.standard_normal((256, 128), dtype=np.float32))
    b = synth.bf16_round_bits(0.05 * rng.standard_normal((64, 128), dtype=np.float32))
    A, Bm = to_device(a), to_device(b)
    D = torch.empty(256, 64, dtype=torch.bfloat16, device="cuda")
    B.llama_gemm_bf16(A.data_ptr(), Bm.data_ptr(), D.data_ptr(), 256, 64, 128, st)
    torch.cuda.synchronize()
    ref = synth.to_f64(a) @ synth.to_f64(b).T
    got = D.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3)
