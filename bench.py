"""Throughput of one Llama-style decoder layer on B300: tokens/s plus the
fraction of the roofline reached by the dominant kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one call of the layer (``llama_layer_forward`` for the prefill
workloads, ``llama_layer_decode`` for the decode workload) over one batch of
seeded synthetic input that already sits in HBM.  Between timed steps L2 is
flushed by writing a 256 MiB buffer (outside the step's events).  Each step is
timed with CUDA events on the launching stream.  The library's own stage
events (``llama_layer_set_timing``) time every kernel stage on a separate pass
of up to 200 steps right after the timed region (events between kernels
would serialise them and hide the programmatic-dependent-launch overlap).

N > 1 (under torchrun): every rank runs an independent replica of the layer
on its own GPU with its own copy of the workload (the path has no exchange
step); timing is bracketed by a barrier and a synchronize, and the value is
the tokens of all ranks over the slowest rank's time (weak scaling).

``--impl reference`` times the fp64 CPU oracle instead (rank 0 only), on a
bounded prefix of the same workload per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decoder-layer tokens/sec on 1 B300 (bf16) + % of TC-peak / HBM roofline"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20  # > 126 MB of L2

DESCRIPTIONS = {
    "tiny": "tiny fp32 layer prefill: batch 1 x seq 64, hidden 256, 4 q / 2 kv "
            "heads, head_dim 64, intermediate 512, RoPE base 1e4",
    "1b": "Llama-3.2-1B-shaped layer prefill bf16: batch 4 x seq 2048, hidden "
          "2048, 32 q / 8 kv heads, head_dim 64, intermediate 8192, Llama3 RoPE "
          "(base 5e5, factor 32), causal",
    "8b": "Llama-3-8B-shaped layer prefill bf16: batch 2 x seq 4096, hidden "
          "4096, 32 q / 8 kv heads, head_dim 128, intermediate 14336, Llama3 "
          "RoPE (base 5e5, factor 8), causal",
    "varlen": "packed varlen 8B-shaped layer prefill bf16: 16384 tokens, "
              "sequence lengths U{128..1024} (seeded), cu_seqlens int32, "
              "causal within each sequence",
    "decode": "KV-cache decode 8B-shaped layer bf16: batch 64 x 1 new token, "
              "start_pos U{512..8191} (seeded), cache [64, 8192, 8, 128] bf16",
    "model1b": "Llama-3.2-1B-shaped model forward bf16: 16 decoder layers (the "
               "1b layer shape, seeded weights per layer), final RMSNorm and the "
               "output projection to 128256 logits, batch 4 x seq 2048",
    "chunk64": "chunked prefill with a KV cache, 8B-shaped layer bf16: 16 sequences x 64 "
               "new tokens, start_pos U{512..8128} (seeded), cache [16, 8192, 8, 128] bf16 "
               "(llama_layer_forward_cached, tensor-core attention over the cache)",
    "chunk512": "chunked prefill with a KV cache, 8B-shaped layer bf16: 16 sequences x 512 "
                "new tokens, start_pos U{512..7680} (seeded), cache [16, 8192, 8, 128] bf16 "
                "(llama_layer_forward_cached, tensor-core attention over the cache)",
    "bwd_8b": "backward pass of the Llama-3-8B-shaped layer bf16 (llama_layer_backward: "
              "forward recomputed, then dx and the weight / norm gradients): batch 2 x "
              "seq 4096, dL/d(out) ~ N(0,1) seeded",
    "bwd_1b": "backward pass of the Llama-3.2-1B-shaped layer bf16 (llama_layer_backward): "
              "batch 4 x seq 2048, dL/d(out) ~ N(0,1) seeded",
    "train_8b": "training step of the Llama-3-8B-shaped layer bf16: llama_layer_forward_train "
                "(the forward, keeping the activations the backward reads) then "
                "llama_layer_backward_saved (dx and the weight / norm gradients, the forward "
                "not recomputed): batch 2 x seq 4096, dL/d(out) ~ N(0,1) seeded",
    "chunked": "chunked prefill with a KV cache, 8B-shaped layer bf16: 16 "
               "sequences x 4 new tokens, start_pos U{512..8188} (seeded), cache "
               "[16, 8192, 8, 128] bf16 (llama_layer_forward_cached)",
}

# Kernel sources behind each stage: a recorded DRAM traffic figure is only
# reported while these files are unchanged.
STAGE_SOURCES = {
    "gate_up_swiglu": ["gemm_tc.cu", "gemm_tc.cuh", "common.cuh"],
    "qkv_rope": ["gemm_tc.cu", "gemm_tc.cuh", "common.cuh"],
    "o_proj_residual": ["gemm_tc.cu", "gemm_tc.cuh", "common.cuh"],
    "down_residual": ["gemm_tc.cu", "gemm_tc.cuh", "common.cuh"],
    "attention": ["attn_prefill.cu", "attn_prefill.cuh", "common.cuh"],
    # the decode / chunked workloads' attention is the split-KV kernel
    "attention_decode": ["decode.cu", "decode.cuh", "common.cuh"],
    "bwd_attention": ["attn_bwd.cu", "attn_bwd.cuh", "common.cuh"],
}
for _s in ("bwd_dw_down", "bwd_swiglu", "bwd_dw_gate_up", "bwd_dh_mlp", "bwd_dw_o",
           "bwd_dattn", "bwd_dw_qkv", "bwd_dx_attn"):
    STAGE_SOURCES[_s] = STAGE_SOURCES["gate_up_swiglu"]


# ----------------------------------------------------------------- helpers
def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 2 s of work)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(DESCRIPTIONS),
                    help="the workload of the headline line (default: the packed "
                         "varlen 8B-shaped layer, the largest single-GPU workload)")
    ap.add_argument("--also", default="auto",
                    help="comma-separated workloads measured after the headline and "
                         "reported under 'workloads' in the same line ('auto': "
                         "1b,8b,decode with the default headline, else none; "
                         "'none': no others)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0,
                    help="CPU work of the oracle baseline (0: leave it out)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the host-buffer measurement (0: leave it out)")
    ap.add_argument("--stages", action="store_true",
                    help="print the per-stage table to stderr")
    return ap.parse_args()


HEADLINE = "varlen"
BACKWARD = {"bwd_8b": "8b", "bwd_1b": "1b"}  # backward workload -> its forward workload
TRAIN = {"train_8b": "8b"}  # training-step workload -> its forward workload
ALSO_AUTO = ("1b", "8b", "decode", "bwd_8b", "train_8b", "chunk512")

DEFAULT_STEPS = {"chunk64": 1000, "chunk512": 300, "bwd_8b": 200, "bwd_1b": 600, "train_8b": 200, "tiny": 500, "1b": 2000, "8b": 600, "varlen": 400,
                 "decode": 3000, "chunked": 1500, "model1b": 40}
MODEL = {"model1b": ("1b", 16, 128256)}  # layer workload, layers, vocabulary


def split_kv_attention(shape, seq_tokens: int) -> bool:
    """Whether the library's chunked prefill of seq_tokens new tokens per
    sequence uses the split-KV attention (groups of up to 16 / n_rep tokens
    share a tile; at most two groups a sequence) rather than the tensor-core
    attention over the cache (llama_layer.h, llama_layer_forward_cached)."""
    n_rep = shape.n_heads // shape.n_kv_heads
    tg = min(16 // n_rep, seq_tokens)
    return seq_tokens < 16 and -(-seq_tokens // tg) <= 2


def max_over_ranks(dist, x: float) -> float:
    """The largest x of all ranks (x itself without a process group): the
    job's time is its slowest replica's."""
    if dist is None:
        return float(x)
    import torch

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, tokens_per_step: int, slowest_ms: float) -> float:
    """Tokens per second of the whole job: every replica processed
    steps x tokens_per_step tokens in at most slowest_ms (weak scaling)."""
    return world * steps * tokens_per_step / (slowest_ms / 1e3)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def src_sha(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "llama_decoder_layer_prologue_b300", "csrc",
                               f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def recorded_traffic(workload: str, stage: str):
    """DRAM bytes per launch recorded from an ncu capture
    (profiles/dram_traffic.json), if the kernel sources are unchanged since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    key = stage
    if stage == "attention" and workload in ("decode", "chunked"):
        key = "attention_decode"
    want = src_sha(STAGE_SOURCES.get(key, []))
    with open(TRAFFIC_FILE) as fh:
        rows = json.load(fh).get("launches", [])
    for r in rows:
        if r.get("workload") == workload and r.get("stage") == stage:
            return float(r["dram_bytes"]) if r.get("sources_sha") == want else None
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained",
                                                      p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                source="fallback")


# ----------------------------------------------------------------- work
def algorithmic_work(inp) -> dict:
    """Per-stage algorithmic FLOPs (prefill) or bytes (decode) of one step."""
    import numpy as np

    w = inp.workload
    s = w.shape
    H, I, d, Hq, Hkv = s.hidden, s.intermediate, s.head_dim, s.n_heads, s.n_kv_heads
    q, nqkv = s.q_size, s.n_qkv
    es = 2 if s.dtype == "bf16" else 4
    T = inp.tokens
    weights = es * (nqkv * H + H * q + 2 * I * H + I * H)
    if w.kind != "decode":
        lens = np.diff(inp.cu_seqlens).astype(np.float64)
        attn = float(np.sum(2.0 * d * Hq * lens * (lens + 1)))
        flops = {"qkv_rope": 2.0 * T * H * nqkv, "attention": attn,
                 "o_proj_residual": 2.0 * T * q * H,
                 "gate_up_swiglu": 2.0 * T * H * 2 * I,
                 "down_residual": 2.0 * T * I * H}
        # the row statistics pass reads x once
        return dict(kind="prefill", flops=flops, total_flops=sum(flops.values()),
                    bytes={"rmsnorm_stats": float(T * H * es)}, weight_bytes=weights)
    sp = inp.start_pos.astype(np.float64)
    kv_read = float(np.sum(2.0 * sp * Hkv * d * es))
    S = w.seq_tokens
    if S >= 16:
        # long chunks run the prefill kernels: a tensor-core workload (the
        # prefix of each sequence read once per kv head, the attention over
        # sp + i + 1 visible keys for new token i)
        vis = float(np.sum(S * sp + S * (S + 1) / 2.0))
        flops = {"qkv_rope": 2.0 * T * H * nqkv, "attention": 4.0 * d * Hq * vis,
                 "o_proj_residual": 2.0 * T * q * H,
                 "gate_up_swiglu": 2.0 * T * H * 2 * I,
                 "down_residual": 2.0 * T * I * H}
        return dict(kind="prefill", flops=flops, total_flops=sum(flops.values()),
                    bytes={"rmsnorm_stats": float(T * H * es),
                           "cache_append": float(2 * 2.0 * T * Hkv * d * es)},
                    weight_bytes=weights, kv_read=kv_read)
    append = 2.0 * T * Hkv * d * es
    act = T * es * (2 * H + nqkv + q + H + 2 * I + I + H)  # x, qkv, o, h, act, out
    total = kv_read + append + weights + act
    # per stage: the bytes a stage has to move at the least (weights once,
    # activations in and out; the stream-K partials are not counted)
    stage = {
        "rmsnorm_stats": T * H * es,
        "qkv_gemm": es * nqkv * H + T * H * es,
        "qkv_rope_cache_append": T * nqkv * es + append,
        "attention": kv_read + T * nqkv * es + T * q * es,
        "o_proj_gemm": es * H * q + T * q * es,
        "o_residual": T * H * es + T * H * (4 + es),
        "gate_up_gemm": es * 2 * I * H + T * H * es,
        "swiglu": T * I * es,
        "down_gemm": es * I * H + T * I * es,
        "down_residual": T * H * (4 + es),
    }
    return dict(kind="decode", bytes={k: float(v) for k, v in stage.items()},
                total_bytes=total, kv_read=kv_read, weight_bytes=weights, flops={})


def algorithmic_work_backward(inp) -> dict:
    """Per-stage algorithmic FLOPs of one llama_layer_backward call: the
    forward it recomputes (every stage but down_proj) and the backward
    proper (each projection twice: dX and dW; the attention's five products
    of the visible pairs, 2.5 x its forward's two), plus the bytes of the
    row passes."""
    w = algorithmic_work(inp)
    f = w["flops"]
    s = inp.workload.shape
    T, H, I, q, nqkv = inp.tokens, s.hidden, s.intermediate, s.q_size, s.n_qkv
    flops = {k: f[k] for k in ("qkv_rope", "attention", "o_proj_residual", "gate_up_swiglu")}
    flops.update({
        "bwd_dw_down": 2.0 * T * H * I, "bwd_swiglu": 2.0 * T * H * I,
        "bwd_dw_gate_up": 2.0 * T * 2 * I * H, "bwd_dh_mlp": 2.0 * T * 2 * I * H,
        "bwd_dw_o": 2.0 * T * H * q, "bwd_dattn": 2.0 * T * H * q,
        "bwd_attention": 2.5 * f["attention"],
        "bwd_dw_qkv": 2.0 * T * nqkv * H, "bwd_dx_attn": 2.0 * T * nqkv * H})
    # the norm-weight gradients' per-32-row-group column sums, added up
    groups = 8 * (-(-nqkv // 256) + -(-(2 * I) // 256))
    by = {"rmsnorm_stats": float(T * H * 2), "bwd_dout_f16": float(T * H * 4),
          "bwd_norm2": float(T * H * (2 + 4 + 2 + 4 + 2)),
          "bwd_norm1": float(T * H * (4 + 4 + 2 + 2)),
          "bwd_dg": float(groups * H * 4 + 2 * H * 4)}
    return dict(kind="prefill", flops=flops, total_flops=sum(flops.values()), bytes=by,
                weight_bytes=w["weight_bytes"])


def algorithmic_work_train(inp) -> dict:
    """Per-stage algorithmic FLOPs of one training step: the whole forward
    (llama_layer_forward_train) and the backward proper
    (llama_layer_backward_saved, no recomputation)."""
    w = algorithmic_work(inp)
    b = algorithmic_work_backward(inp)
    flops = dict(w["flops"])
    flops.update({k: v for k, v in b["flops"].items() if k.startswith("bwd_")})
    by = dict(b["bytes"])
    return dict(kind="prefill", flops=flops, total_flops=sum(flops.values()), bytes=by,
                weight_bytes=w["weight_bytes"])


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples the SM clock, power and clock-event reasons of one GPU while
    running (read only): NVML every 20 ms when pynvml imports, else an
    ``nvidia-smi -lms 100`` child process."""

    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x2: "applications_clocks_setting"}
    QUERY = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"

    def __init__(self, device_index: int, pci_bus_id: str | None = None):
        self.samples = []  # (sm MHz, power W, reason bits)
        self.error = None
        self.max_mhz = None
        self.source = None
        self.nv = None
        self.proc = None
        self._stop = threading.Event()
        self._t = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(pci_bus_id) if pci_bus_id
                      else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml, 20 ms"
        except Exception as e:  # noqa: BLE001
            self.nv = None
            self.error = f"nvml: {e}"
            self.target = pci_bus_id or str(device_index)

    def _reasons(self):
        nv = self.nv
        for fn in ("nvmlDeviceGetCurrentClocksEventReasons",
                   "nvmlDeviceGetCurrentClocksThrottleReasons"):
            if hasattr(nv, fn):
                return int(getattr(nv, fn)(self.h))
        return 0

    def _nvml_sample(self):
        nv = self.nv
        try:
            self.samples.append((nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM),
                                 nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0,
                                 self._reasons()))
        except Exception as e:  # noqa: BLE001
            self.error = str(e)

    def _run(self):
        while not self._stop.is_set():
            self._nvml_sample()
            time.sleep(0.02)

    def __enter__(self):
        if self.nv is not None:
            self._nvml_sample()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
            return self
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 100 ms"
            time.sleep(0.3)  # let the first sample land before the timed work
        except Exception as e:  # noqa: BLE001
            self.error = f"{self.error}; nvidia-smi: {e}"
        return self

    def __exit__(self, *a):
        if self._t is not None:
            self._stop.set()
            self._t.join()
            self._nvml_sample()
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            for line in out.splitlines():
                f = [c.strip() for c in line.split(",")]
                try:
                    self.max_mhz = float(f[1])
                    self.samples.append((float(f[0]), float(f[2]), int(f[3], 16)))
                except (ValueError, IndexError):
                    continue

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "note": self.error or "no samples"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[2]
        reasons = [n for b, n in sorted(self.BITS.items()) if bits & b]
        return {"sm_mhz": float(statistics.median(mhz)), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(mhz), "power_w_max": max(s[1] for s in self.samples),
                "reasons": reasons, "samples": len(self.samples), "source": self.source}


# ----------------------------------------------------------------- oracle
def clock_sampler() -> "ClockSampler":
    """A sampler of the current CUDA device, found in NVML by its PCI bus id
    (NVML numbers the GPUs without regard to CUDA_VISIBLE_DEVICES)."""
    import torch

    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    bus = None
    if hasattr(p, "pci_bus_id"):
        bus = "%08X:%02X:%02X.0" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id,
                                    getattr(p, "pci_device_id", 0))
    return ClockSampler(torch.cuda.current_device(), bus)


def _f64_weights(inp):
    import types

    from llama_decoder_layer_prologue_b300 import synth
    return types.SimpleNamespace(**{k: synth.to_f64(getattr(inp.weights, k)) for k in
                                    ("w_qkv", "w_o", "w_gate_up", "w_down", "g_in",
                                     "g_post")})


class OracleRunner:
    """Runs the fp64 oracle on a sample of the workload: a prefix of the
    token stream cut at whole sequences when it spans more than one, or the
    first b sequences of a decode batch.  Prefixes of a causal sequence are
    exact sub-problems (their outputs do not depend on later tokens)."""

    def __init__(self, inp, backward: bool = False):
        import numpy as np

        import oracle
        from llama_decoder_layer_prologue_b300 import synth

        self.np, self.oracle, self.synth = np, oracle, synth
        self.inp = inp
        self.w = _f64_weights(inp)
        self.backward = backward
        self.dout = synth.to_f64(synth.make_dout(inp)) if backward else None

    def units(self, n: int):
        """A sample of n tokens: (callable, tokens, description)."""
        np, inp, synth = self.np, self.inp, self.synth
        s = inp.workload.shape
        if inp.workload.kind == "decode":
            S = inp.workload.seq_tokens
            nseq = inp.workload.batch
            b = max(1, min(-(-n // S), nseq))  # whole sequences
            x = synth.to_f64(inp.x[:b * S])
            sp = inp.start_pos[:b]

            def rows(i, k):
                return (synth.to_f64(inp.cache_k[i, :k]), synth.to_f64(inp.cache_v[i, :k]))

            if S == 1:
                def run():
                    self.oracle.decoder_layer_decode(x, self.w, s, rows, sp)
                return run, b, f"first {b} of {nseq} decode sequences"

            def run():
                self.oracle.decoder_layer_cached(x, self.w, s, rows, sp, S)
            return run, b * S, f"first {b} of {nseq} sequences x {S} new tokens"
        cu = inp.cu_seqlens.astype(np.int64)
        n = max(1, min(n, inp.tokens))
        whole = int(np.searchsorted(cu, n, side="right") - 1)
        if whole >= 1:
            n = int(cu[whole])
            cut = cu[: whole + 1]
            what = f"first {whole} of {len(cu) - 1} sequences ({n} tokens)"
        else:
            cut = np.array([0, n], dtype=np.int64)
            what = f"prefix of {n} tokens of sequence 0 (length {int(cu[1])})"
        x = synth.to_f64(inp.x[:n])
        pos = inp.positions[:n]

        if self.backward:
            from oracle.backward import decoder_layer_backward
            dout = self.dout[:n]

            def run():
                decoder_layer_backward(x, self.w, s, pos, cut, dout)
            return run, n, what + " (backward pass)"

        def run():
            self.oracle.decoder_layer(x, self.w, s, pos, cut)
        return run, n, what

    def calibrate(self, budget_s: float) -> int:
        """Sample size (tokens) taking about budget_s seconds."""
        small = 16 if self.inp.workload.kind == "decode" else 128
        run, n, _ = self.units(small)
        t = time.perf_counter()
        run()
        dt = max(time.perf_counter() - t, 1e-6)
        return max(1, int(n * budget_s / dt))


def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = [p.get("num_threads", 1) for p in threadpool_info()
                if p.get("user_api") == "blas"]
        if info:
            return int(max(info))
    except Exception:  # noqa: BLE001
        pass
    return os.cpu_count() or 1


def cpu_baseline(inp, budget_s: float, backward: bool = False) -> dict:
    r = OracleRunner(inp, backward)
    n = r.calibrate(min(budget_s, 2.0) / 4)
    n = max(1, int(n * budget_s / (min(budget_s, 2.0) / 4)))
    run, tokens, what = r.units(n)
    t = time.perf_counter()
    run()
    dt = time.perf_counter() - t
    return {"value": tokens / dt, "unit": UNIT, "cores": oracle_threads(),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{what} of the workload, fp64 numpy oracle, one pass"}


# ----------------------------------------------------------------- model
def model_flops(shape, tokens_per_seq, n_layers: int, vocab: int) -> float:
    """Algorithmic FLOPs of one model step: every layer's linears and causal
    attention (visible pairs only) plus the output projection."""
    import numpy as np

    s = shape
    lens = np.asarray(tokens_per_seq, dtype=np.float64)
    T = float(lens.sum())
    linear = 2.0 * T * (s.hidden * s.n_qkv + s.q_size * s.hidden +
                        2 * s.hidden * s.intermediate + s.intermediate * s.hidden)
    attn = float(np.sum(2.0 * s.head_dim * s.n_heads * lens * (lens + 1)))
    return n_layers * (linear + attn) + 2.0 * T * s.hidden * vocab


def model_oracle_sample(m_in, n_tokens: int):
    """The oracle on the first n tokens of sequence 0 (a causal prefix is an
    exact sub-problem): (callable, tokens, description)."""
    import numpy as np

    import oracle
    from llama_decoder_layer_prologue_b300 import synth

    inp = m_in.first
    n = max(1, min(n_tokens, int(inp.cu_seqlens[1])))
    x = synth.to_f64(inp.x[:n])
    ws = [_f64_layer(l) for l in m_in.layers]
    g, wl = synth.to_f64(m_in.g_final), synth.to_f64(m_in.w_lm)
    pos = inp.positions[:n]
    cut = np.array([0, n], dtype=np.int64)

    def run():
        oracle.model_forward(x, ws, inp.workload.shape, pos, cut, g, wl)
    return run, n, f"first {n} tokens of sequence 0 through all {len(ws)} layers"


def _f64_layer(lw):
    import types

    from llama_decoder_layer_prologue_b300 import synth
    return types.SimpleNamespace(**{k: synth.to_f64(getattr(lw, k)) for k in
                                    ("w_qkv", "w_o", "w_gate_up", "w_down", "g_in",
                                     "g_post")})


def run_model(args, rank, local_rank, world, dist=None):
    """The model step: every layer, the final norm and the output projection
    (LlamaModel.forward), timed like the layer workloads."""
    import numpy as np
    import torch

    from llama_decoder_layer_prologue_b300 import synth
    from llama_decoder_layer_prologue_b300.layer import to_device
    from llama_decoder_layer_prologue_b300.model import LlamaModel

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local_rank)
    base, n_layers, vocab = MODEL[args.workload]
    m_in = synth.make_model_inputs(base, n_layers, vocab)
    inp = m_in.first
    s = inp.workload.shape
    model = LlamaModel.from_numpy(s, m_in)
    K = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    W = args.warmup
    x = to_device(inp.x)
    n_seq = len(inp.cu_seqlens) - 1
    seq = int(inp.cu_seqlens[1])
    logits = torch.empty(inp.tokens, vocab, dtype=torch.bfloat16, device="cuda")

    def step():
        model.forward(x, n_seq=n_seq, seq_len=seq, logits=logits)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for i in range(W):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = clock_sampler() if rank == 0 else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if sampler:
        sampler.__enter__()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.__exit__()
    region_s = time.perf_counter() - t0
    if dist is not None:
        dist.barrier()
    rc = model.status()
    if rc != 0:
        raise RuntimeError(f"model status after the timed steps: {rc}")
    total_ms = max_over_ranks(dist, float(sum(a.elapsed_time(b) for a, b in ev)))
    tokens = inp.tokens
    value = job_throughput(world, K, tokens, total_ms)
    ms_step = total_ms / K
    pk = peaks()
    flops = model_flops(s, np.diff(inp.cu_seqlens), n_layers, vocab)

    # host input -> model -> the last position's logits of every sequence
    # (what a generator reads back) to the host, copies inside the events
    e2e = None
    n_e2e = args.e2e_steps if args.e2e_steps is not None else min(K, 20)
    if n_e2e > 0:
        x_h = to_device(inp.x, pin=True)
        last = torch.as_tensor(inp.cu_seqlens[1:] - 1, dtype=torch.long, device="cuda")
        out_h = torch.empty(n_seq, vocab, dtype=torch.bfloat16).pin_memory()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_e2e)]
        # one untimed pass first: the copies and the index gather run here
        # for the first time (module loading, pinned-copy setup)
        x.copy_(x_h, non_blocking=True)
        model.forward(x, n_seq=n_seq, seq_len=seq, logits=logits)
        out_h.copy_(logits.index_select(0, last), non_blocking=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(n_e2e):
            flush.fill_(i & 0xFF)
            ev2[i][0].record(stream)
            x.copy_(x_h, non_blocking=True)
            model.forward(x, n_seq=n_seq, seq_len=seq, logits=logits)
            out_h.copy_(logits.index_select(0, last), non_blocking=True)
            ev2[i][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(dist, float(sum(a.elapsed_time(b) for a, b in ev2)))
        e2e = {"value": job_throughput(world, n_e2e, tokens, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(x_h.numel() * x_h.element_size()),
               "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()),
               "steps": n_e2e, "ms_per_step": e2e_ms / n_e2e,
               "api": "LlamaModel.forward (pinned host input, the last position's "
                      "logits of every sequence copied back)"}
    if rank != 0:
        return None

    achieved = flops / (ms_step / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": f"whole model step ({n_layers} layers, "
                "norm, output projection; all launches)",
                "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"],
                "peak_source": f"{pk['source']} bf16 burst",
                "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
                "algorithmic_per_launch": flops, "launch_ms": ms_step,
                "share_of_step": 1.0, "traffic": None}
    cpu = None
    if args.cpu_baseline_seconds > 0:
        run, n, what = model_oracle_sample(m_in, 4)
        t = time.perf_counter()
        run()
        per_tok = (time.perf_counter() - t) / n
        n = max(1, int(args.cpu_baseline_seconds / max(per_tok, 1e-6)))
        run, n, what = model_oracle_sample(m_in, n)
        t = time.perf_counter()
        run()
        dt = time.perf_counter() - t
        cpu = {"value": n / dt, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
               "seconds": round(dt, 3), "sample": f"{what}, fp64 numpy oracle, one pass"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded x ~ N(0,1), weights ~ N(0,0.02) (each layer its "
                "own draw), RMSNorm weights ~ 1+N(0,0.1), no trained weights",
        "config": {"workload": DESCRIPTIONS[args.workload], "name": args.workload,
                   "tokens_per_step": tokens, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (256 MiB write, outside the "
                         "step's events)", "region_s": round(region_s, 3)},
        "roofline": roofline, "layer_roofline": None, "stages": None,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(K * model.launch_count()),
        "launches_per_step": model.launch_count(),
        "clocks": sampler.summary() if sampler else None,
    }
    return line


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, local_rank, world, dist=None, wl=None, cpu_seconds=None):
    """One workload on our library: the JSON line (rank 0) or None."""
    import numpy as np
    import torch

    from llama_decoder_layer_prologue_b300 import binding as B
    from llama_decoder_layer_prologue_b300 import synth
    from llama_decoder_layer_prologue_b300.layer import LlamaLayer, to_device

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local_rank)
    wl = wl or args.workload
    if cpu_seconds is None:
        cpu_seconds = args.cpu_baseline_seconds

    train = wl in TRAIN
    bwd = wl in BACKWARD or train
    inp = synth.make_inputs(BACKWARD.get(wl) or TRAIN.get(wl) or wl)
    w = inp.workload
    s = w.shape
    layer = LlamaLayer.from_numpy(s, inp.weights)
    K = args.steps if args.steps is not None else DEFAULT_STEPS[wl]
    W = args.warmup
    x = to_device(inp.x)
    out = torch.empty_like(x)
    decode = w.kind == "decode"
    S_new = w.seq_tokens
    if decode:
        ck, cv = to_device(inp.cache_k), to_device(inp.cache_v)
        sp = to_device(inp.start_pos)

        def step(o=out):
            if S_new == 1:
                layer.decode(x, ck, cv, sp, out=o)
            else:
                layer.forward_cached(x, ck, cv, sp, S_new, out=o)
    else:
        varlen = w.kind == "varlen"
        cu = to_device(inp.cu_seqlens) if varlen else None
        seq = int(np.diff(inp.cu_seqlens).max())
        n_seq = len(inp.cu_seqlens) - 1

        def step(o=out):
            if varlen:
                layer.forward(x, cu_seqlens=cu, seq_len=seq, out=o)
            else:
                layer.forward(x, n_seq=n_seq, seq_len=seq, out=o)

        if bwd:  # dL/d(out) in, dx (in `out`) and the weight gradients out
            dout = to_device(synth.make_dout(inp))
            grads = layer.backward(x, dout, n_seq=n_seq, seq_len=seq, dx=out)
            grads.pop("dx")

            def step(o=out):
                layer.backward(x, dout, n_seq=n_seq, seq_len=seq, dx=o, grads=grads)

        if train:  # the layer output too, from the forward that keeps its activations
            y = torch.empty_like(x)

            def step(o=out):
                layer.forward_train(x, n_seq=n_seq, seq_len=seq, out=y)
                layer.backward_saved(x, dout, n_seq=n_seq, seq_len=seq, dx=o, grads=grads)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(W):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    rc = layer.status()
    if rc != 0:
        raise RuntimeError(f"layer status after warm-up: {rc}")
    launches_per_step = layer.launch_count()
    if train:  # two library calls a step
        layer.forward_train(x, n_seq=n_seq, seq_len=seq, out=y)
        n_fwd = layer.launch_count()
        layer.backward_saved(x, dout, n_seq=n_seq, seq_len=seq, dx=out, grads=grads)
        launches_per_step = n_fwd + layer.launch_count()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = clock_sampler() if rank == 0 else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if sampler:
        sampler.__enter__()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.__exit__()
    region_s = time.perf_counter() - t0
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = float(sum(step_ms))
    # Stage durations: the library's stage events put a stream operation
    # between consecutive kernels, which serialises them (no programmatic
    # dependent launch overlap), so they are taken on a separate pass of
    # n_stage steps right after the timed region, with the same L2 flushes.
    n_stage = min(K, 200)
    layer.set_timing(n_stage)
    for i in range(n_stage):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    stages = {}
    for c in range(n_stage):
        for name, ms in layer.stage_times(c):
            stages.setdefault(name, []).append(ms)
    layer.set_timing(0)
    rc = layer.status()
    if rc != 0:
        raise RuntimeError(f"layer status after the timed steps: {rc}")

    total_ms = max_over_ranks(dist, total_ms)

    tokens = inp.tokens
    value = job_throughput(world, K, tokens, total_ms)
    work = (algorithmic_work_train(inp) if train else
            algorithmic_work_backward(inp) if bwd else algorithmic_work(inp))
    pk = peaks()

    # ---- end to end: host input -> layer -> host output, copies timed
    e2e = None
    n_e2e = args.e2e_steps if args.e2e_steps is not None else min(K, 200)
    if n_e2e > 0:
        x_h = to_device(inp.x, pin=True)
        out_h = torch.empty_like(x_h).pin_memory()
        extra_h, extra_d = [], []
        if decode:
            extra_h.append(to_device(inp.start_pos, pin=True))
            extra_d.append(sp)
        cu_h = None
        if w.kind == "varlen" and not decode and not bwd:
            # the host-buffer forward reads the host cu_seqlens to cut the
            # batch into groups and copies each group's rebased prefix sums
            cu_h = torch.from_numpy(inp.cu_seqlens.copy())
        elif w.kind == "varlen":
            extra_h.append(to_device(inp.cu_seqlens, pin=True))
            extra_d.append(cu)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_e2e)]

        if bwd:
            dout_h = to_device(synth.make_dout(inp), pin=True)
            if not train:  # the training step copies it itself
                extra_h.append(dout_h)
                extra_d.append(dout)

        def host_step():
            for h_, d_ in zip(extra_h, extra_d):
                d_.copy_(h_, non_blocking=True)
            if train:
                layer.train_step_from_host(x_h, dout_h, out_h, x, dout, y, out, n_seq=n_seq,
                                           seq_len=seq, grads=grads)
            elif bwd:
                x.copy_(x_h, non_blocking=True)
                step()
                out_h.copy_(out, non_blocking=True)
            elif decode and S_new > 1:
                layer.forward_cached_from_host(x_h, out_h, x, out, ck, cv, sp, S_new)
            elif decode:
                layer.decode_from_host(x_h, out_h, x, out, ck, cv, sp)
            elif w.kind == "varlen":
                layer.forward_from_host(x_h, out_h, x, out, cu_seqlens=cu_h, seq_len=seq)
            else:
                layer.forward_from_host(x_h, out_h, x, out, n_seq=n_seq, seq_len=seq)

        host_step()  # untimed: first use of the copy streams and pinned copies
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(n_e2e):
            flush.fill_(i & 0xFF)
            ev2[i][0].record(stream)
            host_step()
            ev2[i][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = float(sum(a.elapsed_time(b) for a, b in ev2))
        e2e_ms = max_over_ranks(dist, e2e_ms)
        bi = x_h.numel() * x_h.element_size() + sum(
            h_.numel() * h_.element_size() for h_ in extra_h)
        if train:
            bi += dout_h.numel() * dout_h.element_size()
        if cu_h is not None:  # the groups' rebased copies: n_seq + groups entries
            groups = (5 if inp.tokens >= 16384 else
                      min(max(1, inp.tokens // 2048), cu_h.numel() - 1,
                          B.LLAMA_HOST_MAX_CHUNKS))
            bi += 4 * (cu_h.numel() + groups)
        bo = out_h.numel() * out_h.element_size()
        e2e = {"value": job_throughput(world, n_e2e, tokens, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
               "steps": n_e2e, "ms_per_step": e2e_ms / n_e2e,
               "api": ("LlamaLayer.train_step_from_host: forward_train + backward_saved "
                       "(pinned host x copied in, dL/d(out) copied in on a second stream "
                       "during the forward, dx copied out; the layer output and the "
                       "weight gradients stay on the device)") if train else
                      ("LlamaLayer.backward (pinned host x and dL/d(out) copied in, "
                       "dx copied out; the weight gradients stay on the device for the "
                       "optimizer)") if bwd else
                      ("LlamaLayer.%s_from_host (pinned host buffers, "
                       "cudaMemcpyAsync on the layer's stream)"
                       % ("decode" if S_new == 1 else "forward_cached") if decode else
                       "LlamaLayer.forward_from_host -> llama_layer_forward_host "
                       "(pinned host buffers; groups of whole sequences, copies "
                       "in and out on two streams overlapping the layer)")}

    if rank != 0:
        return None

    stage_ms = {k: statistics.mean(v) for k, v in stages.items()}
    # the dominant kernel: the stage with the largest share of the step
    dom = max(stage_ms, key=stage_ms.get) if stage_ms else None
    roofline = None
    if dom:
        dom_ms = stage_ms[dom]
        launches = ("2 launches: split-KV + combine" if (
            dom == "attention" and w.kind == "decode" and split_kv_attention(s, S_new)) else
            "2 launches: dQ + dK/dV" if dom == "bwd_attention" else "1 launch")
        share = dom_ms / (sum(stage_ms.values()) or 1.0)
        if dom in work["flops"]:
            achieved = work["flops"][dom] / (dom_ms / 1e3) / 1e12
            roofline = {"bound": "tensor", "kernel": f"{dom} ({launches})",
                        "achieved": achieved, "peak": pk["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                        "peak_source": f"{pk['source']} bf16 burst",
                        "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
                        "algorithmic_per_launch": work["flops"][dom],
                        "launch_ms": dom_ms, "share_of_step": share}
        else:
            achieved = work["bytes"][dom] / (dom_ms / 1e3) / 1e9
            roofline = {"bound": "hbm", "kernel": f"{dom} ({launches})",
                        "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / pk["hbm_gbs"],
                        "peak_source": f"{pk['source']} HBM copy",
                        "algorithmic_per_launch": work["bytes"][dom],
                        "launch_ms": dom_ms, "share_of_step": share}
        roofline["traffic"] = recorded_traffic(wl, dom)
        roofline["stage_timing"] = (
            f"library CUDA stage events on {n_stage} steps run right after the timed "
            "region (events between kernels disable the launch overlap, so stage "
            "durations are upper bounds)")
    ms_step = total_ms / K
    if work["kind"] == "prefill":
        achieved = work["total_flops"] / (ms_step / 1e3) / 1e12
        layer_roof = {"bound": "tensor", "achieved": achieved, "unit": "TFLOP/s",
                      "frac": achieved / pk["bf16_tflops"],
                      "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
                      "algorithmic_per_step": work["total_flops"]}
    else:
        achieved = work["total_bytes"] / (ms_step / 1e3) / 1e9
        layer_roof = {"bound": "hbm", "achieved": achieved, "unit": "GB/s",
                      "frac": achieved / pk["hbm_gbs"],
                      "frac_of_8tbs": achieved / 8000.0,
                      "algorithmic_per_step": work["total_bytes"]}

    stage_roof = {}
    for name, ms in stage_ms.items():
        e = {"ms": ms}
        if name in work["flops"]:
            tf = work["flops"][name] / (ms / 1e3) / 1e12
            e.update(tflops=tf, frac=tf / pk["bf16_tflops"])
        if name in work.get("bytes", {}):
            gb = work["bytes"][name] / (ms / 1e3) / 1e9
            e.update(gbs=gb, frac=gb / pk["hbm_gbs"])
        stage_roof[name] = e

    cpu = None
    if cpu_seconds > 0:
        cpu = cpu_baseline(inp, cpu_seconds, backward=bwd)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if s.dtype == "bf16" else "f32",
        "data": "synthetic: seeded x ~ N(0,1), weights ~ N(0,0.02), RMSNorm "
                "weights ~ 1+N(0,0.1), no trained weights",
        "config": {"workload": DESCRIPTIONS[wl], "name": wl,
                   "tokens_per_step": tokens, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (256 MiB write, outside "
                         "the step's events)",
                   "region_s": round(region_s, 3)},
        "roofline": roofline,
        "layer_roofline": layer_roof,
        "stages": stage_roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(K * launches_per_step),
        "launches_per_step": launches_per_step,
        "clocks": sampler.summary() if sampler else None,
    }
    if args.stages:
        for name, e in stage_roof.items():
            print(f"{name:>24s} {e['ms']:9.4f} ms  "
                  + (f"{e['tflops']:8.1f} TF/s " if "tflops" in e else "")
                  + (f"{e['gbs']:8.1f} GB/s " if "gbs" in e else "")
                  + (f"frac {e['frac']:.3f}" if "frac" in e else ""),
                  file=sys.stderr)
    return line


# ----------------------------------------------------------------- reference
def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, K timed steps of a bounded sample."""
    if rank != 0:
        return None
    from llama_decoder_layer_prologue_b300 import synth

    K = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    W = args.warmup
    per_step = min(4.0, 150.0 / max(1, K + W))  # whole run within minutes
    if args.workload in MODEL:
        base, n_layers, vocab = MODEL[args.workload]
        m_in = synth.make_model_inputs(base, n_layers, vocab)
        inp = m_in.first
        run0, n0, _ = model_oracle_sample(m_in, 2)
        t = time.perf_counter()
        run0()
        per_tok = (time.perf_counter() - t) / n0
        run, tokens, what = model_oracle_sample(m_in, max(1, int(per_step / per_tok)))
    else:
        inp = synth.make_inputs(BACKWARD.get(args.workload) or TRAIN.get(args.workload)
                                or args.workload)
        r = OracleRunner(inp, args.workload in BACKWARD or args.workload in TRAIN)
        n = r.calibrate(per_step)
        run, tokens, what = r.units(n)
    for _ in range(min(W, 1)):
        run()
    times = []
    for _ in range(K):
        t = time.perf_counter()
        run()
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = K * tokens / total
    s = inp.workload.shape
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": min(W, 1), "ms_per_step": 1e3 * total / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (same seeded inputs as the CUDA arm)",
        "config": {"workload": DESCRIPTIONS[args.workload], "name": args.workload,
                   "tokens_per_step": tokens, "parallelism": "host cores, rank 0"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(),
                         "kind": "oracle",
                         "sample": f"{what} per step (bounded so the run ends "
                                   f"within minutes), fp64 numpy oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "note": f"dtype of the workload is {s.dtype}; the oracle computes in fp64",
    }


def summary_of(line: dict) -> dict:
    """The figures of one workload's line kept under 'workloads'."""
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "roofline",
            "layer_roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks")
    out = {k: line.get(k) for k in keep}
    out["workload"] = line["config"]["workload"]
    out["tokens_per_step"] = line["config"]["tokens_per_step"]
    return out


def also_list(args) -> list:
    """The workloads measured after the headline one (see --also)."""
    if args.also == "auto":
        return list(ALSO_AUTO) if args.workload == HEADLINE else []
    if args.also in ("", "none"):
        return []
    names = [n.strip() for n in args.also.split(",") if n.strip()]
    for n in names:
        if n not in DESCRIPTIONS or n in MODEL:
            raise SystemExit(f"--also: unknown layer workload {n!r}")
    return [n for n in names if n != args.workload]


def check_world(gpus: int, world: int) -> None:
    """One process per GPU: N > 1 needs torchrun (WORLD_SIZE = N); a plain
    `--gpus N` run would time one replica and report it as N GPUs."""
    if gpus != world:
        raise SystemExit(
            f"--gpus {gpus} but WORLD_SIZE={world}: launch N > 1 with "
            f"`python -m torch.distributed.run --nproc-per-node {gpus} bench.py "
            f"--gpus {gpus}`")


def main():
    args = parse_args()
    rank, local_rank, world = dist_env()
    check_world(args.gpus, world)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.workload in MODEL:
            line = run_model(args, rank, local_rank, world, dist)
        else:
            line = run_ours(args, rank, local_rank, world, dist)
            others = {}
            for name in also_list(args):
                torch.cuda.empty_cache()
                sub = run_ours(args, rank, local_rank, world, dist, wl=name,
                               cpu_seconds=min(args.cpu_baseline_seconds, 4.0))
                if sub is not None:
                    others[name] = summary_of(sub)
            if line is not None and others:
                line["workloads"] = others
    finally:
        if dist is not None:
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
