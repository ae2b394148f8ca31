"""A stack of decoder layers, the final RMSNorm and the output projection to
the vocabulary logits (the model forward the pages describe: each layer in
turn, then the norm, then the output projection).  Argument marshalling only:
every step runs in the library's kernels (llama_layer_forward per layer,
llama_rmsnorm_bf16, llama_gemm_bf16)."""

from __future__ import annotations

import torch

from . import binding as B
from .layer import LlamaLayer, stream_ptr, to_device


class LlamaModel:
    """n decoder layers of one shape (bf16) + final norm + output projection."""

    def __init__(self, shape, layers: list[LlamaLayer], g_final: torch.Tensor,
                 w_lm: torch.Tensor):
        assert shape.dtype == "bf16", "the model stack runs bf16 layers"
        assert layers and all(l.shape == shape for l in layers)
        for t in (g_final, w_lm):
            assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
        assert g_final.shape == (shape.hidden,) and w_lm.shape[1] == shape.hidden
        self.shape, self.layers = shape, layers
        self.g_final, self.w_lm = g_final, w_lm
        self.vocab = w_lm.shape[0]
        self._bufs = None

    @classmethod
    def from_numpy(cls, shape, inputs, device="cuda") -> "LlamaModel":
        """From synth.ModelInputs (its layers' weights, g_final and w_lm)."""
        layers = [LlamaLayer.from_numpy(shape, w, device) for w in inputs.layers]
        return cls(shape, layers, to_device(inputs.g_final, device),
                   to_device(inputs.w_lm, device))

    def _prepare(self, T: int, like: torch.Tensor) -> None:
        # the layers run one after another on one stream: one workspace
        # serves them all, and two buffers carry the hidden state
        first = self.layers[0]
        first.ensure_workspace(T)
        for l in self.layers[1:]:
            l.workspace = first.workspace
        if self._bufs is None or self._bufs[0].shape[0] < T:
            self._bufs = [torch.empty(T, self.shape.hidden, dtype=like.dtype,
                                      device=like.device) for _ in range(3)]

    def forward(self, x, cu_seqlens=None, n_seq=None, seq_len=None, logits=None):
        """Logits [T, vocab] of the tokens x [T, hidden] (padded batch when
        cu_seqlens is None, as LlamaLayer.forward)."""
        T = x.shape[0]
        self._prepare(T, x)
        h = x
        for i, layer in enumerate(self.layers):
            out = self._bufs[i % 2][:T]
            layer.forward(h, cu_seqlens=cu_seqlens, n_seq=n_seq, seq_len=seq_len, out=out)
            h = out
        normed = self._bufs[2][:T]
        st = stream_ptr()
        B.llama_rmsnorm_bf16(h.data_ptr(), self.g_final.data_ptr(), normed.data_ptr(),
                             T, self.shape.hidden, self.shape.rms_eps, st)
        if logits is None:
            logits = torch.empty(T, self.vocab, dtype=x.dtype, device=x.device)
        B.llama_gemm_bf16(normed.data_ptr(), self.w_lm.data_ptr(), logits.data_ptr(),
                          T, self.vocab, self.shape.hidden, st)
        return logits

    def launch_count(self) -> int:
        """Kernels of the last forward: every layer's, the norm and the GEMM."""
        return sum(l.launch_count() for l in self.layers) + 2

    def status(self) -> int:
        """The first nonzero status of the layers, else that of the output
        projection (a standalone GEMM)."""
        for l in self.layers:
            rc = l.status()
            if rc != B.LLAMA_OK:
                return rc
        return B.llama_gemm_status(stream_ptr())

    def close(self) -> None:
        for l in self.layers:
            l.close()
