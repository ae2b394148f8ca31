"""Torch-side plumbing around the C ABI: allocates the caller-owned device
buffers (packed weights, workspace) with torch and passes raw pointers and the
current stream to ``binding``.  No arithmetic of the layer happens here.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def make_config(shape) -> B.llama_layer_config:
    """llama_layer_config from an object with the LayerShape fields."""
    return B.llama_layer_config(
        hidden=shape.hidden, n_heads=shape.n_heads,
        n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim,
        intermediate=shape.intermediate, rms_eps=shape.rms_eps,
        rope_base=shape.rope_base, rope_scaling=shape.rope_scaling,
        rope_factor=shape.rope_factor,
        rope_low_freq_factor=shape.rope_low_freq_factor,
        rope_high_freq_factor=shape.rope_high_freq_factor,
        rope_original_max_pos=shape.rope_original_max_pos,
        max_position=shape.max_position,
        dtype=B.LLAMA_DTYPE_BF16 if shape.dtype == "bf16" else B.LLAMA_DTYPE_F32)


def torch_dtype(shape) -> torch.dtype:
    return torch.bfloat16 if shape.dtype == "bf16" else torch.float32


def to_device(arr: np.ndarray, device="cuda", pin: bool = False) -> torch.Tensor:
    """A stored workload array (bf16 bits as uint16, float32, int32) as a
    torch tensor of the matching dtype, on `device` (or pinned host memory)."""
    if arr.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(
            torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    if pin:
        return t.pin_memory()
    return t.to(device)


def stream_ptr() -> int:
    return torch.cuda.current_stream().cuda_stream


class LlamaLayer:
    """One decoder layer whose weights were packed by llama_layer_init."""

    def __init__(self, shape, w_qkv, w_o, w_gate_up, w_down, g_in, g_post):
        self.shape = shape
        self.cfg = make_config(shape)
        self.dtype = torch_dtype(shape)
        dev = w_qkv.device
        self.device = dev
        nbytes = B.llama_layer_packed_bytes(self.cfg)
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        ws = [w_qkv, w_o, w_gate_up, w_down, g_in, g_post]
        for t in ws:
            assert t.is_contiguous() and t.dtype == self.dtype and t.is_cuda
        wts = B.llama_layer_weights(*[t.data_ptr() for t in ws])
        self.handle = B.llama_layer_init(self.cfg, wts, self.packed.data_ptr(),
                                         nbytes, stream_ptr())
        self.workspace = torch.empty(0, dtype=torch.uint8, device=dev)
        self._side = None  # train_step_from_host's copy stream
        # the backward pass reads the weights as given (norm-weight gradients)
        self.weights = ws
        self._wts = wts

    @classmethod
    def from_numpy(cls, shape, weights, device="cuda") -> "LlamaLayer":
        d = {k: to_device(getattr(weights, k), device) for k in
             ("w_qkv", "w_o", "w_gate_up", "w_down", "g_in", "g_post")}
        return cls(shape, **d)

    def ensure_workspace(self, tokens=0, decode_batch=0, max_seq=0) -> None:
        n = B.llama_layer_workspace_bytes(self.handle, tokens, decode_batch,
                                          max_seq)
        if self.workspace.numel() < n:
            self.workspace = torch.empty(n, dtype=torch.uint8,
                                         device=self.device)

    def forward(self, x, position_ids=None, cu_seqlens=None, n_seq=None,
                seq_len=None, out=None):
        """Padded batch when cu_seqlens is None (x: [n_seq * seq_len, H])."""
        T = x.shape[0]
        if cu_seqlens is None:
            seq_len = seq_len or T
            n_seq = n_seq or (T // seq_len)
        else:
            n_seq = cu_seqlens.numel() - 1
            assert seq_len is not None, "varlen needs max_seqlen"
        self.ensure_workspace(T)
        if out is None:
            out = torch.empty_like(x)
        B.llama_layer_forward(
            self.handle, x.data_ptr(), out.data_ptr(),
            position_ids.data_ptr() if position_ids is not None else None,
            cu_seqlens.data_ptr() if cu_seqlens is not None else None,
            n_seq, seq_len, T, self.workspace.data_ptr(),
            self.workspace.numel(), stream_ptr())
        return out

    @staticmethod
    def _batch(x, cu_seqlens, n_seq, seq_len):
        """(n_seq, seq_len) of a padded (cu_seqlens None) or packed batch."""
        T = x.shape[0]
        if cu_seqlens is None:
            seq_len = seq_len or T
            return n_seq or (T // seq_len), seq_len
        assert seq_len is not None, "varlen needs max_seqlen"
        return cu_seqlens.numel() - 1, seq_len

    def _ensure_backward_workspace(self, T) -> None:
        n = B.llama_layer_backward_workspace_bytes(self.handle, T)
        if self.workspace.numel() < n:
            self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device)

    def forward_train(self, x, position_ids=None, cu_seqlens=None, n_seq=None,
                      seq_len=None, out=None):
        """The forward of a training step: the output as forward() computes
        it, and the activations the backward reads kept in this layer's
        workspace for backward_saved() (same x and batch layout)."""
        T = x.shape[0]
        n_seq, seq_len = self._batch(x, cu_seqlens, n_seq, seq_len)
        self._ensure_backward_workspace(T)
        if out is None:
            out = torch.empty_like(x)
        B.llama_layer_forward_train(
            self.handle, x.data_ptr(), out.data_ptr(),
            position_ids.data_ptr() if position_ids is not None else None,
            cu_seqlens.data_ptr() if cu_seqlens is not None else None,
            n_seq, seq_len, T, self.workspace.data_ptr(), self.workspace.numel(),
            stream_ptr())
        return out

    def _grads(self, grads):
        if grads is None:
            names = ("dw_qkv", "dw_o", "dw_gate_up", "dw_down", "dg_in", "dg_post")
            grads = {k: torch.empty(w.shape, dtype=torch.float32, device=self.device)
                     for k, w in zip(names, self.weights)}
        g = B.llama_layer_grads(*[grads[k].data_ptr() for k in
                                  ("dw_qkv", "dw_o", "dw_gate_up", "dw_down", "dg_in",
                                   "dg_post")])
        return grads, g

    def backward(self, x, dout, position_ids=None, cu_seqlens=None, n_seq=None,
                 seq_len=None, dx=None, grads=None):
        """Gradients of the prefill layer given dL/d(out) (same batch layout
        as forward), the forward recomputed: returns dict dx (bf16) and
        dw_qkv, dw_o, dw_gate_up, dw_down, dg_in, dg_post (fp32, the weights'
        shapes)."""
        T = x.shape[0]
        n_seq, seq_len = self._batch(x, cu_seqlens, n_seq, seq_len)
        self._ensure_backward_workspace(T)
        if dx is None:
            dx = torch.empty_like(x)
        grads, g = self._grads(grads)
        B.llama_layer_backward(
            self.handle, self._wts, x.data_ptr(), dout.data_ptr(), dx.data_ptr(), g,
            position_ids.data_ptr() if position_ids is not None else None,
            cu_seqlens.data_ptr() if cu_seqlens is not None else None,
            n_seq, seq_len, T, self.workspace.data_ptr(), self.workspace.numel(),
            stream_ptr())
        return dict(dx=dx, **grads)

    def backward_saved(self, x, dout, position_ids=None, cu_seqlens=None, n_seq=None,
                       seq_len=None, dx=None, grads=None):
        """backward() from the activations the last forward_train() kept (the
        same x, batch layout and workspace; the library refuses otherwise)."""
        T = x.shape[0]
        n_seq, seq_len = self._batch(x, cu_seqlens, n_seq, seq_len)
        if dx is None:
            dx = torch.empty_like(x)
        grads, g = self._grads(grads)
        B.llama_layer_backward_saved(
            self.handle, self._wts, x.data_ptr(), dout.data_ptr(), dx.data_ptr(), g,
            position_ids.data_ptr() if position_ids is not None else None,
            cu_seqlens.data_ptr() if cu_seqlens is not None else None,
            n_seq, seq_len, T, self.workspace.data_ptr(), self.workspace.numel(),
            stream_ptr())
        return dict(dx=dx, **grads)

    def train_step_from_host(self, x_host, dout_host, dx_host, x_dev, dout_dev, out_dev,
                             dx_dev, n_seq=None, seq_len=None, cu_seqlens=None,
                             grads=None):
        """One training step whose x, dL/d(out) and dx live in (pinned) host
        memory: x is copied in on the current stream, then dL/d(out) on a
        second stream while forward_train runs; backward_saved waits for it,
        and dx is copied out.  The layer output (out_dev) and the weight
        gradients stay on the device; ``*_dev`` are device buffers of the
        host tensors' shapes.  dx_host is valid once the current stream is
        synchronised."""
        cur = torch.cuda.current_stream()
        if self._side is None:
            self._side = torch.cuda.Stream(device=self.device)
        x_dev.copy_(x_host, non_blocking=True)
        # dout_dev is free once earlier work on `cur` is; its copy starts
        # after x's (the two would share the host link) and runs under the
        # forward
        x_in = torch.cuda.Event()
        x_in.record(cur)
        self._side.wait_event(x_in)
        with torch.cuda.stream(self._side):
            dout_dev.copy_(dout_host, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(self._side)
        self.forward_train(x_dev, n_seq=n_seq, seq_len=seq_len, cu_seqlens=cu_seqlens,
                           out=out_dev)
        cur.wait_event(ready)
        res = self.backward_saved(x_dev, dout_dev, n_seq=n_seq, seq_len=seq_len,
                                  cu_seqlens=cu_seqlens, dx=dx_dev, grads=grads)
        dx_host.copy_(dx_dev, non_blocking=True)
        return res

    def decode(self, x, cache_k, cache_v, start_pos, out=None):
        Bt = x.shape[0]
        max_seq = cache_k.shape[1]
        self.ensure_workspace(0, Bt, max_seq)
        if out is None:
            out = torch.empty_like(x)
        B.llama_layer_decode(self.handle, x.data_ptr(), out.data_ptr(),
                             cache_k.data_ptr(), cache_v.data_ptr(),
                             start_pos.data_ptr(), Bt, max_seq,
                             self.workspace.data_ptr(), self.workspace.numel(),
                             stream_ptr())
        return out

    def forward_cached(self, x, cache_k, cache_v, start_pos, seq_tokens, out=None):
        """seq_tokens new tokens per sequence against the KV cache (x rows
        b * seq_tokens .. are sequence b's, at positions start_pos[b] ..)."""
        rows = x.shape[0]
        assert rows % seq_tokens == 0, "x holds whole chunks"
        max_seq = cache_k.shape[1]
        # long chunks run the prefill kernels (prefill workspace layout)
        long = seq_tokens >= B.LLAMA_LONG_CHUNK
        self.ensure_workspace(rows if long else 0, rows, max_seq)
        if out is None:
            out = torch.empty_like(x)
        B.llama_layer_forward_cached(self.handle, x.data_ptr(), out.data_ptr(),
                                     cache_k.data_ptr(), cache_v.data_ptr(),
                                     start_pos.data_ptr(), rows // seq_tokens,
                                     seq_tokens, max_seq, self.workspace.data_ptr(),
                                     self.workspace.numel(), stream_ptr())
        return out

    def forward_from_host(self, x_host, out_host, x_dev, out_dev,
                          cu_seqlens=None, n_seq=None, seq_len=None, chunks=0):
        """One forward whose input and output live in (pinned) host memory,
        through llama_layer_forward_host: groups of whole sequences are copied
        in, run and copied out with the copies overlapping the layer (chunks =
        0 lets the library pick the groups).  ``x_dev`` / ``out_dev`` are device
        staging buffers of the same shape; out_host is valid once the current
        stream is synchronised.  ``cu_seqlens`` of a packed batch is a host
        int32 tensor: the library cuts the batch into groups with it."""
        T = x_host.shape[0]
        if cu_seqlens is None:
            seq_len = seq_len or T
            n_seq = n_seq or (T // seq_len)
        else:
            if (cu_seqlens.device.type != "cpu" or cu_seqlens.dtype != torch.int32
                    or not cu_seqlens.is_contiguous()):
                raise ValueError("cu_seqlens of forward_from_host: a contiguous "
                                 "host int32 tensor")
            n_seq = cu_seqlens.numel() - 1
            assert seq_len is not None, "varlen needs max_seqlen"
        self.ensure_workspace(T)
        B.llama_layer_forward_host(
            self.handle, x_host.data_ptr(), out_host.data_ptr(), x_dev.data_ptr(),
            out_dev.data_ptr(),
            cu_seqlens.data_ptr() if cu_seqlens is not None else None,
            n_seq, seq_len, T, chunks, self.workspace.data_ptr(),
            self.workspace.numel(), stream_ptr())
        return out_host

    def decode_from_host(self, x_host, out_host, x_dev, out_dev, cache_k,
                         cache_v, start_pos):
        """One decode step with host input / output (see forward_from_host);
        the KV cache stays resident on the device."""
        x_dev.copy_(x_host, non_blocking=True)
        self.decode(x_dev, cache_k, cache_v, start_pos, out=out_dev)
        out_host.copy_(out_dev, non_blocking=True)
        return out_host

    def forward_cached_from_host(self, x_host, out_host, x_dev, out_dev, cache_k,
                                 cache_v, start_pos, seq_tokens):
        """forward_cached with host input / output (see decode_from_host)."""
        x_dev.copy_(x_host, non_blocking=True)
        self.forward_cached(x_dev, cache_k, cache_v, start_pos, seq_tokens, out=out_dev)
        out_host.copy_(out_dev, non_blocking=True)
        return out_host

    def set_timing(self, ring_calls: int) -> None:
        """Record stage events for the last ``ring_calls`` calls (0: off)."""
        B.llama_layer_set_timing(self.handle, ring_calls)

    def stage_times(self, call: int = 0):
        """[(stage, ms)] of recorded call ``call`` (0 = the most recent)."""
        return B.llama_layer_stage_times(self.handle, call)

    def launch_count(self) -> int:
        return B.llama_layer_launch_count(self.handle)

    def status(self) -> int:
        return B.llama_layer_status(self.handle, stream_ptr())

    def stages(self, tokens: int, decode: bool = False) -> dict:
        """The intermediates of the last call with `tokens` rows (element
        types as llama_layer_workspace_offsets documents; for bf16 layers h
        and act are returned already multiplied back by 256 and 16)."""
        off = B.llama_layer_workspace_offsets(self.handle, tokens, int(decode))
        s = self.shape
        bf = self.dtype == torch.bfloat16
        f16 = torch.float16 if bf else torch.float32
        types = {"qkv": (s.n_qkv, torch.bfloat16 if (bf and decode) else f16),
                 "attn": (s.q_size, f16), "h": (s.hidden, f16 if bf else torch.float32),
                 "act": (s.intermediate, f16)}
        views = {}
        for (name, (width, dt)), o in zip(types.items(), off):
            n = tokens * width * torch.tensor([], dtype=dt).element_size()
            views[name] = self.workspace[o:o + n].view(dt).view(tokens, width)
        if bf:
            views["h"] = views["h"].float() * 256.0
            views["act"] = views["act"].float() * 16.0
        return views

    def close(self) -> None:
        if self.handle:
            B.llama_layer_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
