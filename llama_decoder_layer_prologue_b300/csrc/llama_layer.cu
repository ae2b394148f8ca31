// The C ABI of libllama_layer.so (declared in include/llama_layer.h):
// argument checks, weight repacking, the RoPE table, workspace layout, and the
// launch sequence of each call.  All device memory belongs to the caller.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "../../include/llama_layer.h"
#include "common.cuh"
#include "attn_bwd.cuh"
#include "attn_prefill.cuh"
#include "decode.cuh"
#include "gemm_tc.cuh"
#include "kernels.h"

using namespace llama;

namespace {

constexpr size_t kAlign = 256;
// Split-tile phase of the prefill GEMMs: CTAs (one per SM) it supports, and
// the fp32 slot of one 128 x 256 tile piece.
constexpr int kMaxSkCtas = 160;
// Work-item counter pairs in the packed buffer: the prefill attention
// (plain or cached), the attention backward's dQ and dK / dV kernels (which
// may overlap under programmatic dependent launch).
constexpr int kSchedAttn = 0, kSchedDq = 2;  // the dK / dV pair follows the dQ pair
constexpr size_t kSkSlotBytes = 128 * 256 * sizeof(float);

size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

struct PackedLayout {
  size_t wqkv, wo, wgu, wd, gpost, cos_t, sin_t, status, skflag, sched, total;
};

PackedLayout packed_layout(const llama_layer_config& c) {
  size_t es = c.dtype == LLAMA_DTYPE_BF16 ? 2 : 4;
  size_t nqkv = (size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  size_t qs = (size_t)c.n_heads * c.head_dim;
  PackedLayout p;
  size_t o = 0;
  p.wqkv = o; o = align_up(o + nqkv * c.hidden * es);
  p.wo = o; o = align_up(o + (size_t)c.hidden * qs * es);
  p.wgu = o; o = align_up(o + 2 * (size_t)c.intermediate * c.hidden * es);
  p.wd = o; o = align_up(o + (size_t)c.hidden * c.intermediate * es);
  p.gpost = o; o = align_up(o + (size_t)c.hidden * es);
  size_t table = (size_t)c.max_position * (c.head_dim / 2) * sizeof(float);
  p.cos_t = o; o = align_up(o + table);
  p.sin_t = o; o = align_up(o + table);
  p.status = o; o = align_up(o + 64);
  p.skflag = o; o = align_up(o + (kMaxSkCtas + 1) * sizeof(uint32_t));
  // the attention kernels' work-item counter pairs (kSched*), zeroed at init
  p.sched = o; o = align_up(o + 16 * sizeof(int));
  p.total = o;
  return p;
}

int check_config(const llama_layer_config* c) {
  if (!c) return LLAMA_ERR_INVALID_ARG;
  if (c->dtype != LLAMA_DTYPE_F32 && c->dtype != LLAMA_DTYPE_BF16)
    return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
      c->intermediate <= 0 || c->max_position <= 0)
    return LLAMA_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (c->n_heads % c->n_kv_heads != 0 || c->n_heads / c->n_kv_heads > 16)
    return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden % 128 != 0 || c->intermediate % 128 != 0)
    return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (!(c->rms_eps > 0.f) || !(c->rope_base > 1.0)) return LLAMA_ERR_INVALID_ARG;
  if (c->rope_scaling == LLAMA_ROPE_LLAMA3) {
    if (!(c->rope_factor >= 1.0) || !(c->rope_low_freq_factor > 0.0) ||
        !(c->rope_high_freq_factor > c->rope_low_freq_factor) ||
        c->rope_original_max_pos <= 0)
      return LLAMA_ERR_INVALID_ARG;
  } else if (c->rope_scaling == LLAMA_ROPE_LINEAR) {
    if (!(c->rope_factor > 0.0)) return LLAMA_ERR_INVALID_ARG;
  } else if (c->rope_scaling == LLAMA_ROPE_DYNAMIC_NTK) {
    if (!(c->rope_factor >= 1.0) || c->rope_original_max_pos <= 0)
      return LLAMA_ERR_INVALID_ARG;
  } else if (c->rope_scaling != LLAMA_ROPE_NONE) {
    return LLAMA_ERR_UNSUPPORTED_SHAPE;
  }
  return LLAMA_OK;
}

// RoPE inverse frequencies in double precision ("parallel_attention.py"
// section 1: inv_freq_i = 1 / base^(2i/d); the Llama3, linear and dynamic NTK
// scalings as stated in llama_layer.h).
void rope_inv_freq(const llama_layer_config& c, double* f) {
  const int half = c.head_dim / 2;
  double base = c.rope_base;
  if (c.rope_scaling == LLAMA_ROPE_DYNAMIC_NTK &&
      c.max_position > c.rope_original_max_pos) {
    const double scale = c.rope_factor * c.max_position / c.rope_original_max_pos -
                         (c.rope_factor - 1.0);
    base *= pow(scale, (double)c.head_dim / (c.head_dim - 2.0));
  }
  for (int i = 0; i < half; ++i) {
    double v = pow(base, -2.0 * i / c.head_dim);
    if (c.rope_scaling == LLAMA_ROPE_LINEAR) v /= c.rope_factor;
    if (c.rope_scaling == LLAMA_ROPE_LLAMA3) {
      const double wl = 2.0 * M_PI / v;
      const double orig = c.rope_original_max_pos;
      const double lo = c.rope_low_freq_factor, hi = c.rope_high_freq_factor;
      if (wl < orig / hi) {
        // high frequency: unchanged
      } else if (wl > orig / lo) {
        v = v / c.rope_factor;
      } else {
        const double s = (orig / wl - lo) / (hi - lo);
        v = (1.0 - s) * v / c.rope_factor + s * v;
      }
    }
    f[i] = v;
  }
}

struct WsLayout {
  size_t pos, r1, ss2, xn, qkv, attn, h, hg, act, sk, cu, total;
};

// Fixed-order row sums of a GEMM with `N` output columns in 256-column
// tiles: two slots (column halves) per tile, so that the sum of a row does
// not depend on the order in which tiles finish (TcEpiArgs::ss_np).
int row_sum_slots(int N) { return 2 * ((N + 255) / 256); }

// TcEpiArgs::pair of the pair GEMMs: 2 runs one M = 256 tcgen05.mma
// (cta_group::2) per pair and K step.
constexpr int kPairMode = 2;

WsLayout ws_layout(const llama_layer_config& c, int tokens) {
  size_t es = c.dtype == LLAMA_DTYPE_BF16 ? 2 : 4;
  size_t T = (size_t)(tokens > 0 ? tokens : 0);
  size_t nqkv = (size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  WsLayout w;
  size_t o = 0;
  w.pos = o; o = align_up(o + T * 4);
  w.r1 = o; o = align_up(o + T * 4);
  // bf16 layers: the slots of sum(h^2) per row; fp32 layers: one float
  w.ss2 = o; o = align_up(o + T * 4 * (es == 2 ? row_sum_slots(c.hidden) : 1));
  w.xn = o;  // bf16 layers: fp16 x / RMS(x), the QKV operand
  if (es == 2) o = align_up(o + T * c.hidden * 2);
  w.qkv = o; o = align_up(o + T * nqkv * es);
  w.attn = o; o = align_up(o + T * c.n_heads * c.head_dim * es);
  // h: fp32 layers keep it in fp32 (w.h) and scale it by g_post into w.hg;
  // bf16 layers keep only the fp16 copy h / 256 in w.hg, which is both the
  // MLP input and the residual of down_proj
  w.h = o; if (es == 4) o = align_up(o + T * c.hidden * 4);
  w.hg = o; o = align_up(o + T * c.hidden * es);
  w.act = o; o = align_up(o + T * c.intermediate * es);
  w.sk = o;  // split-tile pieces of the tensor-core GEMMs (bf16 layers)
  if (c.dtype == LLAMA_DTYPE_BF16 && T > 0) o = align_up(o + kMaxSkCtas * kSkSlotBytes);
  // llama_layer_forward_host on a packed batch: the groups' rebased
  // cu_seqlens (n_seq + groups <= T + LLAMA_HOST_MAX_CHUNKS entries).  Last,
  // so that a group's forward on fewer rows, whose regions all lie below its
  // own w.cu, never reaches it.
  w.cu = o; o = align_up(o + (T + LLAMA_HOST_MAX_CHUNKS + 1) * 4);
  w.total = o;
  return w;
}

}  // namespace

struct llama_layer {
  llama_layer_config cfg;
  Dims dm;
  bool bf16;
  char* packed;
  PackedLayout pl;
  int* status;
  int sm_count;
  CUtensorMap tm_wqkv, tm_wo, tm_wgu, tm_wd;  // bf16 weights as B, 256 rows
  CUtensorMap ta_wqkv, ta_wo, ta_wgu, ta_wd;  // bf16 weights as A, 128 rows
  // Stage timing (llama_layer_set_timing): a ring of `ring` call records.
  // In record c, event i is recorded on the call's stream where stage i
  // begins and the last one where the call ends.
  int ring;                  // 0 = timing off
  int calls;                 // calls recorded since timing was switched on
  cudaEvent_t* ev;           // [ring][LLAMA_MAX_STAGES + 1]
  const char** stage_name;   // [ring][LLAMA_MAX_STAGES]
  int* n_marks;              // [ring]
  int launches;  // kernels launched by the last forward / decode call
  uint32_t* sk_flag;  // split-tile flags (packed buffer, zeroed at init)
  int* sched;         // attention work-item counters (packed buffer, zeroed at init)
  uint32_t sk_epoch;  // value of the last split-tile launch's flags
  // llama_layer_forward_host: copy streams and events, created on first use
  cudaStream_t h2d, d2h;
  cudaEvent_t ev_start, ev_done, ev_in[LLAMA_HOST_MAX_CHUNKS],
      ev_comp[LLAMA_HOST_MAX_CHUNKS];
  bool host_ready;
  // packed batches: the groups' cu_seqlens arrays, each rebased to start at
  // 0, in page-locked memory (cu_cap entries) until ev_cu says that the
  // copy which reads them has run
  int32_t* cu_host;
  size_t cu_cap;
  cudaEvent_t ev_cu;
  bool cu_pending;
  // The activations the last llama_layer_forward_train call kept in its
  // workspace, for llama_layer_backward_saved: that call's arguments.  Any
  // other call through the layer whose workspace overlaps [ws, ws + bytes)
  // clears `valid`.
  struct {
    const char* ws;
    size_t bytes;
    const void* x;
    const int32_t *pos, *cu;
    int n_seq, seq_len, tokens;
    bool valid;
  } saved;
};

namespace {

int cuda_err(cudaError_t e) { return e == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA; }

// A call is about to write [ws, ws + bytes): the kept activations are lost
// if that overlaps them.
void clobber(llama_layer* L, const void* ws, size_t bytes) {
  const char* p = static_cast<const char*>(ws);
  if (L->saved.valid && p < L->saved.ws + L->saved.bytes && L->saved.ws < p + bytes)
    L->saved.valid = false;
}

// Starts stage `name` (or ends the call when name is null) on stream s.
void mark(llama_layer* L, cudaStream_t s, const char* name) {
  if (!L->ring) return;
  const int c = (L->calls - 1) % L->ring;
  int& n = L->n_marks[c];
  if (n > LLAMA_MAX_STAGES) return;
  if (!name && n == LLAMA_MAX_STAGES + 1) return;
  if (name && n == LLAMA_MAX_STAGES) return;  // keep the last event for the end
  cudaEventRecord(L->ev[(size_t)c * (LLAMA_MAX_STAGES + 1) + n], s);
  if (name) L->stage_name[(size_t)c * LLAMA_MAX_STAGES + n] = name;
  ++n;
}

void begin_call(llama_layer* L) {
  L->launches = 0;
  if (!L->ring) return;
  ++L->calls;
  L->n_marks[(L->calls - 1) % L->ring] = 0;
}

void free_timing(llama_layer* L) {
  if (L->ev) {
    for (size_t i = 0; i < (size_t)L->ring * (LLAMA_MAX_STAGES + 1); ++i)
      if (L->ev[i]) cudaEventDestroy(L->ev[i]);
  }
  delete[] L->ev;
  delete[] L->stage_name;
  delete[] L->n_marks;
  L->ev = nullptr;
  L->stage_name = nullptr;
  L->n_marks = nullptr;
  L->ring = 0;
  L->calls = 0;
}

// What the backward pass keeps from its forward recomputation beyond the
// forward's own workspace: the attention's log2 softmax denominators and the
// gate / up pre-activations.  With saves the forward stops after gate_up.
struct FwdSaves {
  float* lse;  // [T, n_heads]
  void* gu;    // [T, 2 I] fp16, packed gate|up order
};

// A long chunk of S new tokens per sequence against the KV cache
// (llama_layer_forward_cached with seq_tokens >= LLAMA_LONG_CHUNK): the
// prefill path with positions start_pos[b] + i, the chunk's keys and values
// appended to the cache, and the attention reading the cache.
struct ChunkArgs {
  void *cache_k, *cache_v;
  const int32_t* start_pos;
  int max_seq;
};

int forward_impl(llama_layer* L, const void* x, void* out, const int32_t* pos_in,
                 const int32_t* cu, int n_seq, int seq_len, int T, char* ws,
                 cudaStream_t s, const FwdSaves* sv = nullptr,
                 const ChunkArgs* ch = nullptr) {
  const llama_layer_config& c = L->cfg;
  const Dims& dm = L->dm;
  const bool b16 = L->bf16;
  WsLayout w = ws_layout(c, T);
  int32_t* pos = pos_in ? const_cast<int32_t*>(pos_in)
                        : reinterpret_cast<int32_t*>(ws + w.pos);
  float* r1 = reinterpret_cast<float*>(ws + w.r1);
  float* ss2 = reinterpret_cast<float*>(ws + w.ss2);
  void* qkv = ws + w.qkv;
  void* attn = ws + w.attn;
  void* h = ws + w.h;
  void* act = ws + w.act;
  const char* P = L->packed;
  const float* cos_t = reinterpret_cast<const float*>(P + L->pl.cos_t);
  const float* sin_t = reinterpret_cast<const float*>(P + L->pl.sin_t);

  begin_call(L);
  mark(L, s, "rmsnorm_stats");
  if (ch) {
    if (chunk_positions(ch->start_pos, n_seq, seq_len, ch->max_seq, dm.max_pos,
                        reinterpret_cast<int32_t*>(ws + w.pos), L->status, s) != cudaSuccess)
      return LLAMA_ERR_CUDA;
  } else {
    launch_positions(cu, n_seq, seq_len, T, reinterpret_cast<int32_t*>(ws + w.pos),
                     pos_in == nullptr, L->status, s);
  }
  if (b16)
    simt_row_norm_f16(x, T, dm.H, dm.eps, r1, nullptr, ws + w.xn, s);
  else
    simt_row_rms(b16, x, T, dm.H, dm.eps, r1, ss2, s);
  L->launches += 2;
  if (b16) {
    cudaError_t e;
    CUtensorMap ta;
    // CTA pairs (one M = 256 MMA per pair, the 128-row-box weight maps)
    // unless the pairs' tiles, rounded up to whole pairs of M-tiles, take a
    // round more on the SMs than single CTAs' tiles (a small odd M-tile
    // count); single CTAs then fill a partly idle last round with the
    // split-tile phase.  Measured with the cta_group::2 pairs on one B300:
    // the 8B QKV 3.6 % faster as pairs than as split single CTAs, the 1B
    // down_proj the same either way.
    auto pairs = [&](int N) {
      const long m_tiles = (T + 127) / 128, n_tiles = (N + 255) / 256;
      const long slots = L->sm_count, pair_slots = std::max(1, L->sm_count / 2);
      const long rounds_single = (m_tiles * n_tiles + slots - 1) / slots;
      const long rounds_pair = ((m_tiles + 1) / 2 * n_tiles + pair_slots - 1) / pair_slots;
      return rounds_pair <= rounds_single ? kPairMode : 0;
    };
    // Split-tile phase: pieces in the workspace, flags in the packed buffer,
    // a new nonzero epoch per launch.
    auto split = [&](TcEpiArgs& a) {
      if (L->sm_count > kMaxSkCtas) return;
      a.sk_part = reinterpret_cast<float*>(ws + w.sk);
      a.sk_flag = L->sk_flag;
      if (++L->sk_epoch == 0) ++L->sk_epoch;
      a.sk_epoch = L->sk_epoch;
    };
    TcEpiArgs ep;
    ep.status = L->status;
    ep.pdl = 1;
    // a2 + a3: QKV projection of x / RMS(x) (fp16) with the g_in-folded
    // fp16 weights, RoPE on q and k.
    if (!tc_encode_bf16(&ta, ws + w.xn, T, dm.H, 128)) return LLAMA_ERR_CUDA;
    ep.ab_f16 = 1;
    ep.out = qkv; ep.ldo = dm.Nqkv; ep.pos = pos;
    ep.cos_t = cos_t; ep.sin_t = sin_t; ep.head_dim = dm.d;
    ep.rope_cols = (dm.Hq + dm.Hkv) * dm.d; ep.max_pos = dm.max_pos;
    // q | k | v in fp16 for the attention; bf16 for a cached chunk, whose
    // keys and values join the bf16 cache the attention reads them from
    ep.out_f16 = ch ? 0 : 1;
    mark(L, s, "qkv_rope");
    split(ep);
    ep.pair = pairs(dm.Nqkv);
    e = tc_gemm(TC_QKV, 256, ta, ep.pair ? L->ta_wqkv : L->tm_wqkv, T, dm.Nqkv, dm.H, ep,
                L->sm_count, s);
    if (e != cudaSuccess) return LLAMA_ERR_CUDA;
    ++L->launches;
    if (ch) {
      mark(L, s, "cache_append");
      if (chunk_append(static_cast<const __nv_bfloat16*>(qkv), dm.Nqkv, dm.Hq * dm.d,
                       dm.Hkv * dm.d, static_cast<__nv_bfloat16*>(ch->cache_k),
                       static_cast<__nv_bfloat16*>(ch->cache_v), ch->start_pos, n_seq,
                       seq_len, ch->max_seq, dm.max_pos, L->sm_count, s) != cudaSuccess)
        return LLAMA_ERR_CUDA;
      ++L->launches;
    }
    // a4 / a5: causal GQA attention (padded or varlen).
    AttnArgs aa;
    aa.qkv = static_cast<const __half*>(qkv);
    aa.out = static_cast<__half*>(attn);
    aa.cu = cu; aa.tokens = T; aa.seq_len = seq_len; aa.nqkv = dm.Nqkv;
    aa.n_heads = dm.Hq; aa.n_kv_heads = dm.Hkv; aa.head_dim = dm.d;
    aa.status = L->status;
    aa.sched = L->sched + kSchedAttn;
    if (sv) aa.lse = sv->lse;
    mark(L, s, "attention");
    if (ch) {
      aa.cache_k = static_cast<const __nv_bfloat16*>(ch->cache_k);
      aa.cache_v = static_cast<const __nv_bfloat16*>(ch->cache_v);
      aa.start_pos = ch->start_pos;
      aa.max_seq = ch->max_seq;
      aa.max_pos = dm.max_pos;
      if (attn_prefill_cached(aa, n_seq, L->sm_count, s) != cudaSuccess)
        return LLAMA_ERR_CUDA;
    } else if (attn_prefill(aa, n_seq, seq_len, L->sm_count, s) != cudaSuccess) {
      return LLAMA_ERR_CUDA;
    }
    ++L->launches;
    // a7: o_proj + residual, row sums of h^2 for the second RMSNorm.
    if (!tc_encode_bf16(&ta, attn, T, dm.Hq * dm.d, 128)) return LLAMA_ERR_CUDA;
    ep = TcEpiArgs();
    ep.status = L->status;
    ep.pdl = 1;
    ep.out = ws + w.hg; ep.ldo = dm.H; ep.residual = x;
    ep.ss_out = ss2; ep.ss_np = row_sum_slots(dm.H);
    ep.ab_f16 = 1; ep.out_f16 = 1; ep.out_scale = kHgScale;
    mark(L, s, "o_proj_residual");
    split(ep);
    ep.pair = pairs(dm.H);
    e = tc_gemm(TC_RESID_SS, 256, ta, ep.pair ? L->ta_wo : L->tm_wo, T, dm.H, dm.Hq * dm.d,
                ep, L->sm_count, s);
    if (e != cudaSuccess) return LLAMA_ERR_CUDA;
    ++L->launches;
    // a8: gate_up (g_post folded into its packed weights) on h with the
    // RMSNorm row scale, silu(gate) * up.
    if (!tc_encode_bf16(&ta, ws + w.hg, T, dm.H, 128)) return LLAMA_ERR_CUDA;
    ep = TcEpiArgs();
    ep.status = L->status;
    ep.pdl = 1;
    ep.out = act; ep.ldo = dm.I; ep.ss_in = ss2; ep.ss_np = row_sum_slots(dm.H);
    ep.inv_h = 1.0f / dm.H; ep.eps = dm.eps;
    ep.ab_f16 = 1; ep.in_scale = 1.0f / kHgScale; ep.out_f16 = 1; ep.out_scale = kActScale;
    if (sv) ep.aux_out = sv->gu;
    mark(L, s, "gate_up_swiglu");
    split(ep);
    ep.pair = pairs(2 * dm.I);
    e = tc_gemm(TC_SWIGLU, 256, ta, ep.pair ? L->ta_wgu : L->tm_wgu, T, 2 * dm.I, dm.H, ep,
                L->sm_count, s);
    if (e != cudaSuccess) return LLAMA_ERR_CUDA;
    ++L->launches;
    // the backward's recomputation (no output) continues from here
    if (sv && !out) return cuda_err(cudaGetLastError());
    // a9: down_proj + residual.
    if (!tc_encode_bf16(&ta, act, T, dm.I, 128)) return LLAMA_ERR_CUDA;
    ep = TcEpiArgs();
    ep.status = L->status;
    ep.pdl = 1;
    ep.out = out; ep.ldo = dm.H; ep.residual = ws + w.hg;
    ep.res_scale = 1.0f / kHgScale;  // h from its fp16 copy
    ep.ab_f16 = 1; ep.in_scale = 1.0f / kActScale;
    mark(L, s, "down_residual");
    split(ep);
    ep.pair = pairs(dm.H);
    e = tc_gemm(TC_RESID, 256, ta, ep.pair ? L->ta_wd : L->tm_wd, T, dm.H, dm.I, ep,
                L->sm_count, s);
    if (e != cudaSuccess) return LLAMA_ERR_CUDA;
    ++L->launches;
  } else {
    simt_gemm(b16, EPI_ROWSCALE, x, P + L->pl.wqkv, qkv, T, dm.Nqkv, dm.H, r1,
              nullptr, s);
    simt_rope(b16, qkv, T, dm, pos, cos_t, sin_t, L->status, s);
    simt_attention_prefill(b16, qkv, attn, T, dm, cu, n_seq, seq_len, seq_len, s);
    simt_gemm(b16, EPI_RESIDUAL, attn, P + L->pl.wo, h, T, dm.H, dm.Hq * dm.d,
              nullptr, x, s);
    simt_row_rms(b16, h, T, dm.H, dm.eps, ss2, nullptr, s);
    simt_scale_cols(static_cast<const float*>(h),
                    reinterpret_cast<const float*>(P + L->pl.gpost),
                    reinterpret_cast<float*>(ws + w.hg), T, dm.H, s);
    simt_gemm(b16, EPI_SWIGLU, ws + w.hg, P + L->pl.wgu, act, T, dm.I, dm.H,
              ss2, nullptr, s);
    simt_gemm(b16, EPI_RESIDUAL, act, P + L->pl.wd, out, T, dm.H, dm.I,
              nullptr, h, s);
    L->launches += 8;
  }
  mark(L, s, nullptr);
  return cuda_err(cudaGetLastError());
}

// Backward workspace: the forward's (recomputed) intermediates, then the
// saves and the gradients of the intermediates.
struct BwdLayout {
  WsLayout fw;
  size_t lse, dsum, gu, dout16, dgu, du, dot1, dot2, dh32, dh16, dattn, dqkv, dg_in, dg_post,
      total;
  int np, ng_in, ng_post;  // row-sum slots per row; 32-row groups of W_qkv, W_gate_up
};

BwdLayout bwd_layout(const llama_layer_config& c, int tokens) {
  BwdLayout b;
  b.fw = ws_layout(c, tokens);
  const size_t T = (size_t)(tokens > 0 ? tokens : 0);
  const size_t H = c.hidden, I = c.intermediate, q = (size_t)c.n_heads * c.head_dim;
  const size_t nqkv = (size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  size_t o = b.fw.total;
  b.lse = o; o = align_up(o + T * c.n_heads * 4);
  b.dsum = o; o = align_up(o + T * c.n_heads * 4);
  b.gu = o; o = align_up(o + T * 2 * I * 2);
  b.dout16 = o; o = align_up(o + T * H * 2);
  b.dgu = o; o = align_up(o + T * 2 * I * 2);
  b.du = o; o = align_up(o + T * H * 4);
  b.np = row_sum_slots(c.hidden);
  b.dot1 = o; o = align_up(o + T * 4 * b.np);
  b.dot2 = o; o = align_up(o + T * 4 * b.np);
  b.dh32 = o; o = align_up(o + T * H * 4);
  b.dh16 = o; o = align_up(o + T * H * 2);
  b.dattn = o; o = align_up(o + T * q * 2);
  b.dqkv = o; o = align_up(o + T * nqkv * 2);
  // the norm-weight gradients' column sums per 32-row group of the dW GEMMs,
  // added up in group order at the end: 4 groups per 128-row tile, for every
  // tile the CTA pairs run (an odd tile count gets a partner past the rows,
  // whose groups hold zeros)
  b.ng_in = (int)((nqkv + 255) / 256 * 8);
  b.ng_post = (int)((2 * I + 255) / 256 * 8);
  b.dg_in = o; o = align_up(o + (size_t)b.ng_in * H * 4);
  b.dg_post = o; o = align_up(o + (size_t)b.ng_post * H * 4);
  b.total = o;
  return b;
}

// The forward's activations the backward reads, at their places in the
// backward workspace (the forward's own intermediates sit in its front part).
FwdSaves bwd_saves(const BwdLayout& b, char* ws) {
  FwdSaves sv;
  sv.lse = reinterpret_cast<float*>(ws + b.lse);
  sv.gu = ws + b.gu;
  return sv;
}

// Gradients of the prefill layer: the forward recomputed (keeping the
// attention's softmax denominators and gate / up) unless a training forward
// left them in `ws` (recompute = false), then the chain rule in reverse order
// of the forward's steps ("模型层" 9.6 LlamaForTraining puts this layer under
// a loss; each step is stated in llama_layer.h).
int backward_impl(llama_layer* L, const llama_layer_weights* w, const void* x,
                  const void* dout, void* dx, const llama_layer_grads* gr,
                  const int32_t* pos_in, const int32_t* cu, int n_seq, int seq_len,
                  int T, char* ws, cudaStream_t s, bool recompute) {
  const Dims& dm = L->dm;
  const BwdLayout b = bwd_layout(L->cfg, T);
  int rc = LLAMA_OK;
  if (recompute) {
    const FwdSaves sv = bwd_saves(b, ws);
    rc = forward_impl(L, x, nullptr, pos_in, cu, n_seq, seq_len, T, ws, s, &sv);
    if (rc) return rc;
  } else {
    begin_call(L);
  }
  int launches = L->launches;
  const WsLayout& f = b.fw;
  const char* P = L->packed;
  const int32_t* pos = pos_in ? pos_in : reinterpret_cast<const int32_t*>(ws + f.pos);
  float* dot1 = reinterpret_cast<float*>(ws + b.dot1);
  float* dot2 = reinterpret_cast<float*>(ws + b.dot2);
  float* du = reinterpret_cast<float*>(ws + b.du);
  const int qd = dm.Hq * dm.d;
  const size_t H = dm.H;
  auto fail = [](cudaError_t e) { return e != cudaSuccess; };
  mark(L, s, "bwd_dout_f16");
  if (fail(bwd_dout_f16(dout, ws + b.dout16, T, dm.H, L->sm_count, s)))
    return LLAMA_ERR_CUDA;
  ++launches;
  // K-major [rows, cols] (box 128 rows) and MN-major [K rows, cols] (box 64)
  auto kmaj = [](CUtensorMap* m, const void* p, int rows, int cols) {
    return tc_encode_bf16(m, p, rows, cols, 128);
  };
  auto mnmaj = [](CUtensorMap* m, const void* p, int rows, int cols) {
    return tc_encode_bf16(m, p, rows, cols, 64);
  };
  auto gemm = [&](int epi, const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K,
                  TcEpiArgs ep, const char* name) -> int {
    ep.status = L->status;
    ep.pdl = 1;
    ep.ab_f16 = 1;
    ep.pair = kPairMode;  // CTA pairs (all B maps here are MN-major)
    mark(L, s, name);
    if (tc_gemm(epi, 256, ta, tb, M, N, K, ep, L->sm_count, s) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    ++launches;
    return LLAMA_OK;
  };
  CUtensorMap ta, tb;
  // dW_down = dout^T act (act stored / 16)
  if (!mnmaj(&ta, ws + b.dout16, T, dm.H) || !mnmaj(&tb, ws + f.act, T, dm.I))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = gr->dw_down; ep.ldo = dm.I; ep.in_scale = 1.0f / kActScale; ep.b_const = 0;
    if ((rc = gemm(TC_DW, ta, tb, dm.H, dm.I, T, ep, "bwd_dw_down"))) return rc;
  }
  // d act = dout W_down -> d gate | d up (times 1 / RMS(h)), packed order
  if (!kmaj(&ta, ws + b.dout16, T, dm.H) || !mnmaj(&tb, P + L->pl.wd, dm.H, dm.I))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = ws + b.dgu; ep.ldo = 2 * dm.I; ep.aux_in = ws + b.gu;
    ep.ss_in = reinterpret_cast<const float*>(ws + f.ss2); ep.ss_np = b.np;
    ep.inv_h = 1.0f / dm.H;
    ep.eps = dm.eps;
    if ((rc = gemm(TC_SWIGLU_BWD, ta, tb, T, dm.I, dm.H, ep, "bwd_swiglu"))) return rc;
  }
  // dW_gate_up = dgu^T (h / RMS(h)) g_post, dg_post (h stored / 256)
  if (!mnmaj(&ta, ws + b.dgu, T, 2 * dm.I) || !mnmaj(&tb, ws + f.hg, T, dm.H))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = gr->dw_gate_up; ep.ldo = dm.H; ep.in_scale = 1.0f / kHgScale; ep.b_const = 0;
    ep.colscale = w->g_post; ep.w_orig = w->w_gate_up; ep.inter = dm.I;
    ep.dg = reinterpret_cast<float*>(ws + b.dg_post);
    if ((rc = gemm(TC_DW, ta, tb, 2 * dm.I, dm.H, T, ep, "bwd_dw_gate_up"))) return rc;
  }
  // u2 = dgu W'_gate_up (the gradient of h / RMS(h), times 1 / RMS(h)), sum(u2 h)
  if (!kmaj(&ta, ws + b.dgu, T, 2 * dm.I) || !mnmaj(&tb, P + L->pl.wgu, 2 * dm.I, dm.H))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = du; ep.ldo = dm.H; ep.residual = ws + f.hg; ep.res_scale = 1.0f / kHgScale;
    ep.ss_out = dot2; ep.ss_np = b.np;
    if ((rc = gemm(TC_F32_DOT, ta, tb, T, dm.H, 2 * dm.I, ep, "bwd_dh_mlp"))) return rc;
  }
  mark(L, s, "bwd_norm2");
  if (fail(bwd_norm2(dout, du, ws + f.hg, 1.0f / kHgScale,
                     reinterpret_cast<const float*>(ws + f.ss2), dot2, b.np, dm.eps,
                     reinterpret_cast<float*>(ws + b.dh32), ws + b.dh16, T, dm.H, s)))
    return LLAMA_ERR_CUDA;
  ++launches;
  // dW_o = dh^T attn
  if (!mnmaj(&ta, ws + b.dh16, T, dm.H) || !mnmaj(&tb, ws + f.attn, T, qd))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = gr->dw_o; ep.ldo = qd; ep.b_const = 0;
    if ((rc = gemm(TC_DW, ta, tb, dm.H, qd, T, ep, "bwd_dw_o"))) return rc;
  }
  // d attn = dh W_o, D = rowsum(d attn * attn) per head
  if (!kmaj(&ta, ws + b.dh16, T, dm.H) || !mnmaj(&tb, P + L->pl.wo, dm.H, qd))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = ws + b.dattn; ep.ldo = qd; ep.residual = ws + f.attn;
    ep.aux_out = ws + b.dsum; ep.head_dim = dm.d;
    if ((rc = gemm(TC_DO, ta, tb, T, qd, dm.H, ep, "bwd_dattn"))) return rc;
  }
  // attention backward -> dq | dk | dv (before RoPE)
  {
    AttnBwdArgs ab;
    ab.qkv = reinterpret_cast<const __half*>(ws + f.qkv);
    ab.dout = reinterpret_cast<const __half*>(ws + b.dattn);
    ab.lse = reinterpret_cast<const float*>(ws + b.lse);
    ab.dsum = reinterpret_cast<const float*>(ws + b.dsum);
    ab.dqkv = reinterpret_cast<__half*>(ws + b.dqkv);
    ab.cu = cu; ab.pos = pos;
    ab.cos_t = reinterpret_cast<const float*>(P + L->pl.cos_t);
    ab.sin_t = reinterpret_cast<const float*>(P + L->pl.sin_t);
    ab.tokens = T; ab.seq_len = seq_len; ab.nqkv = dm.Nqkv; ab.n_heads = dm.Hq;
    ab.n_kv_heads = dm.Hkv; ab.head_dim = dm.d; ab.max_pos = dm.max_pos;
    ab.status = L->status;
    ab.sched = L->sched + kSchedDq;  // the dQ pair, then the dK / dV pair
    mark(L, s, "bwd_attention");
    if (attn_backward(ab, n_seq, seq_len, L->sm_count, s) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    launches += 2;
  }
  // dW_qkv = dqkv^T (x / RMS(x)) g_in, dg_in
  if (!mnmaj(&ta, ws + b.dqkv, T, dm.Nqkv) || !mnmaj(&tb, ws + f.xn, T, dm.H))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = gr->dw_qkv; ep.ldo = dm.H; ep.b_const = 0;
    ep.colscale = w->g_in; ep.w_orig = w->w_qkv;
    ep.dg = reinterpret_cast<float*>(ws + b.dg_in);
    if ((rc = gemm(TC_DW, ta, tb, dm.Nqkv, dm.H, T, ep, "bwd_dw_qkv"))) return rc;
  }
  // u1 = dqkv W'_qkv, sum(u1 x)
  if (!kmaj(&ta, ws + b.dqkv, T, dm.Nqkv) || !mnmaj(&tb, P + L->pl.wqkv, dm.Nqkv, dm.H))
    return LLAMA_ERR_CUDA;
  {
    TcEpiArgs ep;
    ep.out = du; ep.ldo = dm.H; ep.residual = x; ep.res_bf16 = 1;
    ep.ss_out = dot1; ep.ss_np = b.np;
    if ((rc = gemm(TC_F32_DOT, ta, tb, T, dm.H, dm.Nqkv, ep, "bwd_dx_attn"))) return rc;
  }
  mark(L, s, "bwd_norm1");
  if (fail(bwd_norm1(reinterpret_cast<const float*>(ws + b.dh32), du, x,
                     reinterpret_cast<const float*>(ws + f.r1), dot1, b.np, dx, T, dm.H, s)))
    return LLAMA_ERR_CUDA;
  ++launches;
  // dg_in, dg_post: the dW GEMMs' row-group sums added up in order
  mark(L, s, "bwd_dg");
  if (fail(bwd_col_sums(reinterpret_cast<const float*>(ws + b.dg_in), b.ng_in, gr->dg_in,
                        reinterpret_cast<const float*>(ws + b.dg_post), b.ng_post,
                        gr->dg_post, dm.H, s)))
    return LLAMA_ERR_CUDA;
  ++launches;
  L->launches = launches;
  mark(L, s, nullptr);
  return cuda_err(cudaGetLastError());
}

constexpr int kDecodeChunk = 256;  // tokens per decode pass (<= GEMM bn)
// Short chunks: the split-KV attention reads each sequence's prefix once per
// group of up to 16 / n_rep new tokens; with more groups than this the
// tensor-core attention over the cache (one read, 128-row tiles mostly
// empty) is faster (8B-shaped layer, 16 sequences, prefixes 512..8191: 4 new
// tokens 74 against 160 us, 8: 124 against 161, 12: 177 against 162).
constexpr int kMaxPrefixReads = 2;

int decode_bn(int B) { return B <= 64 ? 64 : (B <= 128 ? 128 : 256); }

struct DecLayout {
  size_t r1, ss2, xn, qkv, attn, hg, act, part, attn_part, total;
  int bn, max_chunks, rec;
  TcStreamK plan[4];  // QKV, O, GU, DOWN
};

// Decode workspace for B (<= kDecodeChunk) tokens and caches of max_seq rows.
DecLayout dec_layout(const llama_layer* L, int B, int max_seq) {
  const Dims& dm = L->dm;
  const size_t T = (size_t)(B > 0 ? B : 0);
  const size_t es = L->bf16 ? 2 : 4;
  DecLayout w;
  w.bn = decode_bn(B);
  w.plan[DEC_QKV] = tc_streamk_plan(dm.Nqkv, B, dm.H, w.bn, L->sm_count);
  w.plan[DEC_O] = tc_streamk_plan(dm.H, B, dm.Hq * dm.d, w.bn, L->sm_count);
  w.plan[DEC_GU] = tc_streamk_plan(2 * dm.I, B, dm.H, w.bn, L->sm_count);
  w.plan[DEC_DOWN] = tc_streamk_plan(dm.H, B, dm.I, w.bn, L->sm_count);
  size_t part = 0;
  for (const TcStreamK& p : w.plan) {
    size_t n = (size_t)p.tiles * p.slots * 128 * w.bn * sizeof(float);
    if (n > part) part = n;
  }
  w.max_chunks = attn_decode_chunks(max_seq > 0 ? max_seq : 1);
  const int n_rep = dm.Hq / dm.Hkv;
  w.rec = n_rep * (dm.d + 2);
  size_t o = 0;
  w.r1 = o; o = align_up(o + T * 4);
  w.ss2 = o; o = align_up(o + T * 4 * (size_t)((dm.H + 127) / 128));  // per o_proj tile
  w.xn = o; o = align_up(o + T * dm.H * 2);  // fp16 x / RMS(x)
  w.qkv = o; o = align_up(o + T * dm.Nqkv * es);
  w.attn = o; o = align_up(o + T * dm.Hq * dm.d * es);
  w.hg = o; o = align_up(o + T * dm.H * es);
  w.act = o; o = align_up(o + T * dm.I * es);
  w.part = o; o = align_up(o + part);
  w.attn_part = o;
  o = align_up(o + T * dm.Hkv * (size_t)w.max_chunks * w.rec * sizeof(float));
  w.total = o;
  return w;
}

// One pass over token rows row0 .. row0 + B - 1 of a call (x / out point at
// the pass's first row; the cache and start_pos are the whole call's).
int decode_chunk(llama_layer* L, const void* x, void* out, void* ck, void* cv,
                 const int32_t* start_pos, int row0, int seq_tokens, int B,
                 int max_seq, char* ws, cudaStream_t s) {
  const Dims& dm = L->dm;
  const DecLayout w = dec_layout(L, B, max_seq);
  const char* P = L->packed;
  DecodeArgs a;
  a.batch = B; a.bn = w.bn;
  a.row0 = row0; a.seq_tokens = seq_tokens;
  a.hidden = dm.H; a.n_heads = dm.Hq; a.n_kv_heads = dm.Hkv;
  a.head_dim = dm.d; a.inter = dm.I; a.nqkv = dm.Nqkv;
  a.max_seq = max_seq; a.max_pos = dm.max_pos; a.eps = dm.eps;
  a.part = reinterpret_cast<const float*>(ws + w.part);
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.r1 = reinterpret_cast<const float*>(ws + w.r1);
  a.ss2 = reinterpret_cast<float*>(ws + w.ss2);
  a.ss_np = (dm.H + 127) / 128;
  a.start_pos = start_pos;
  a.cos_t = reinterpret_cast<const float*>(P + L->pl.cos_t);
  a.sin_t = reinterpret_cast<const float*>(P + L->pl.sin_t);
  a.qkv = reinterpret_cast<__nv_bfloat16*>(ws + w.qkv);
  a.cache_k = static_cast<__nv_bfloat16*>(ck);
  a.cache_v = static_cast<__nv_bfloat16*>(cv);
  a.attn = reinterpret_cast<__half*>(ws + w.attn);
  a.attn_part = reinterpret_cast<float*>(ws + w.attn_part);
  a.max_chunks = w.max_chunks; a.n_rep_rec = w.rec;
  {
    const int n_rep = dm.Hq / dm.Hkv;  // <= 16 (check_config)
    a.tg = 16 / n_rep < seq_tokens ? 16 / n_rep : seq_tokens;
    a.gps = (seq_tokens + a.tg - 1) / a.tg;
  }
  a.hg = reinterpret_cast<__half*>(ws + w.hg);
  a.act = reinterpret_cast<__half*>(ws + w.act);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = L->status;

  // One projection: stream-K swap-AB GEMM into the partials, then its
  // finalize kernel.
  static const char* const kGemmName[4] = {"qkv_gemm", "o_proj_gemm",
                                            "gate_up_gemm", "down_gemm"};
  static const char* const kFinName[4] = {"qkv_rope_cache_append",
                                          "o_residual", "swiglu",
                                          "down_residual"};
  auto project = [&](int stage, const CUtensorMap& wmap, const void* act_in,
                     int N_out, int K) -> int {
    CUtensorMap tb;
    if (!tc_encode_bf16(&tb, act_in, B, K, w.bn)) return LLAMA_ERR_CUDA;
    TcEpiArgs ep;
    ep.out = ws + w.part;
    ep.pdl = 1;
    ep.part_slots = w.plan[stage].slots;
    ep.status = L->status;
    ep.ab_f16 = 1;  // fp16 weights and activations
    mark(L, s, kGemmName[stage]);
    if (tc_gemm(TC_PARTIAL, w.bn, wmap, tb, N_out, B, K, ep, L->sm_count, s) !=
        cudaSuccess)
      return LLAMA_ERR_CUDA;
    mark(L, s, kFinName[stage]);
    L->launches += 2;
    return decode_finalize(stage, a, w.plan[stage], s) == cudaSuccess
               ? LLAMA_OK : LLAMA_ERR_CUDA;
  };

  // a1: 1/RMS of every new token.
  mark(L, s, "rmsnorm_stats");
  simt_row_norm_f16(x, B, dm.H, dm.eps, const_cast<float*>(a.r1), nullptr, ws + w.xn, s);
  ++L->launches;
  // a2 + a3 + cache append.
  int rc = project(DEC_QKV, L->ta_wqkv, ws + w.xn, dm.Nqkv, dm.H);
  if (rc) return rc;
  // a6: attention over cache rows 0 .. position.  Up to kMaxPrefixReads
  // groups of new tokens per sequence: the split-KV decode attention (each
  // prefix spread over many CTAs, read once per group).  More: the
  // tensor-core prefill attention over the cache, which reads each prefix
  // once per group of query heads.  A pass holds whole sequences.
  mark(L, s, "attention");
  if (a.gps > kMaxPrefixReads && row0 % seq_tokens == 0 && B % seq_tokens == 0) {
    const size_t seq0 = (size_t)(row0 / seq_tokens);
    const size_t cache_seq = (size_t)max_seq * dm.Hkv * dm.d;
    AttnArgs aa;
    aa.qkv = reinterpret_cast<const __half*>(a.qkv);  // bf16 bits: the cache's type
    aa.out = a.attn;
    aa.cu = nullptr;
    aa.tokens = B; aa.seq_len = seq_tokens; aa.nqkv = dm.Nqkv;
    aa.n_heads = dm.Hq; aa.n_kv_heads = dm.Hkv; aa.head_dim = dm.d;
    aa.status = L->status;
    aa.sched = L->sched + kSchedAttn;
    aa.cache_k = a.cache_k + seq0 * cache_seq;
    aa.cache_v = a.cache_v + seq0 * cache_seq;
    aa.start_pos = start_pos + seq0;
    aa.max_seq = max_seq;
    aa.max_pos = dm.max_pos;
    if (attn_prefill_cached(aa, B / seq_tokens, L->sm_count, s) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    L->launches += 1;
  } else {
    if (decode_attention(a, s) != cudaSuccess) return LLAMA_ERR_CUDA;
    L->launches += 2;
  }
  // a7: o_proj + residual (+ sums of h^2).
  if ((rc = project(DEC_O, L->ta_wo, a.attn, dm.H, dm.Hq * dm.d))) return rc;
  // a8: gate_up + SiLU * up.
  if ((rc = project(DEC_GU, L->ta_wgu, a.hg, 2 * dm.I, dm.H))) return rc;
  // a9: down_proj + residual.
  if ((rc = project(DEC_DOWN, L->ta_wd, a.act, dm.H, dm.I))) return rc;
  return cuda_err(cudaGetLastError());
}

// B token rows: seq_tokens consecutive rows per sequence (1 for decode).
int decode_impl(llama_layer* L, const void* x, void* out, void* ck, void* cv,
                const int32_t* start_pos, int B, int max_seq, char* ws,
                cudaStream_t s, int seq_tokens = 1) {
  const llama_layer_config& c = L->cfg;
  const Dims& dm = L->dm;
  const bool b16 = L->bf16;
  begin_call(L);
  if (b16) {
    const size_t es = 2, row = (size_t)dm.H * es;
    // passes of <= kDecodeChunk rows, in order: a pass's rows see the cache
    // rows every earlier pass (and their own) appended; chunks of several
    // tokens pass whole sequences (both attentions take whole chunks)
    const int pass = seq_tokens >= 2 && seq_tokens <= kDecodeChunk
                         ? kDecodeChunk / seq_tokens * seq_tokens : kDecodeChunk;
    for (int b0 = 0; b0 < B; b0 += pass) {
      const int nb = B - b0 < pass ? B - b0 : pass;
      int rc = decode_chunk(L, static_cast<const char*>(x) + b0 * row,
                            static_cast<char*>(out) + b0 * row, ck, cv, start_pos,
                            b0, seq_tokens, nb, max_seq, ws, s);
      if (rc) return rc;
    }
    mark(L, s, nullptr);
    return LLAMA_OK;
  }
  WsLayout w = ws_layout(c, B);
  float* r1 = reinterpret_cast<float*>(ws + w.r1);
  float* r2 = reinterpret_cast<float*>(ws + w.ss2);
  void* qkv = ws + w.qkv;
  void* attn = ws + w.attn;
  void* h = ws + w.h;
  void* act = ws + w.act;
  const char* P = L->packed;
  const float* cos_t = reinterpret_cast<const float*>(P + L->pl.cos_t);
  const float* sin_t = reinterpret_cast<const float*>(P + L->pl.sin_t);

  mark(L, s, "decode_fp32");
  simt_row_rms(b16, x, B, dm.H, dm.eps, r1, nullptr, s);
  simt_gemm(b16, EPI_ROWSCALE, x, P + L->pl.wqkv, qkv, B, dm.Nqkv, dm.H, r1,
            nullptr, s);
  simt_rope(b16, qkv, B, dm, start_pos, cos_t, sin_t, L->status, s);
  simt_cache_append(b16, qkv, ck, cv, start_pos, B, max_seq, dm, L->status, s);
  simt_attention_decode(b16, qkv, ck, cv, attn, start_pos, B, max_seq, dm, s);
  simt_gemm(b16, EPI_RESIDUAL, attn, P + L->pl.wo, h, B, dm.H, dm.Hq * dm.d,
            nullptr, x, s);
  simt_row_rms(b16, h, B, dm.H, dm.eps, r2, nullptr, s);
  simt_scale_cols(static_cast<const float*>(h),
                  reinterpret_cast<const float*>(P + L->pl.gpost),
                  reinterpret_cast<float*>(ws + w.hg), B, dm.H, s);
  simt_gemm(b16, EPI_SWIGLU, ws + w.hg, P + L->pl.wgu, act, B, dm.I, dm.H, r2,
            nullptr, s);
  simt_gemm(b16, EPI_RESIDUAL, act, P + L->pl.wd, out, B, dm.H, dm.I, nullptr,
            h, s);
  L->launches += 10;
  mark(L, s, nullptr);
  return cuda_err(cudaGetLastError());
}

size_t decode_ws_bytes(const llama_layer* L, int batch, int max_seq) {
  if (batch <= 0) return 0;
  if (!L->bf16) return ws_layout(L->cfg, batch).total;
  return dec_layout(L, batch < kDecodeChunk ? batch : kDecodeChunk, max_seq).total;
}

}  // namespace

extern "C" {

int llama_rope_inv_freq(const llama_layer_config* cfg, double* inv_freq) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!inv_freq) return LLAMA_ERR_INVALID_ARG;
  rope_inv_freq(*cfg, inv_freq);
  return LLAMA_OK;
}

int llama_layer_packed_bytes(const llama_layer_config* cfg, size_t* bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!bytes) return LLAMA_ERR_INVALID_ARG;
  *bytes = packed_layout(*cfg).total;
  return LLAMA_OK;
}

int llama_layer_init(const llama_layer_config* cfg,
                     const llama_layer_weights* wts, void* packed,
                     size_t packed_bytes, void* stream, llama_layer_t** out) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!wts || !packed || !out) return LLAMA_ERR_INVALID_ARG;
  const void* ptrs[6] = {wts->w_qkv, wts->w_o, wts->w_gate_up,
                         wts->w_down, wts->g_in, wts->g_post};
  for (const void* p : ptrs)
    if (!p || !aligned(p, 16)) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(packed, kAlign)) return LLAMA_ERR_INVALID_ARG;
  PackedLayout pl = packed_layout(*cfg);
  if (packed_bytes < pl.total) return LLAMA_ERR_WORKSPACE_TOO_SMALL;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LLAMA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return LLAMA_ERR_UNSUPPORTED_DEVICE;

  llama_layer* L = new (std::nothrow) llama_layer();
  if (!L) return LLAMA_ERR_INVALID_ARG;
  L->cfg = *cfg;
  const llama_layer_config& c = *cfg;
  L->dm.H = c.hidden; L->dm.Hq = c.n_heads; L->dm.Hkv = c.n_kv_heads;
  L->dm.d = c.head_dim; L->dm.I = c.intermediate;
  L->dm.Nqkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  L->dm.max_pos = c.max_position; L->dm.eps = c.rms_eps;
  L->bf16 = c.dtype == LLAMA_DTYPE_BF16;
  L->packed = static_cast<char*>(packed);
  L->pl = pl;
  L->status = reinterpret_cast<int*>(L->packed + pl.status);
  L->sk_flag = reinterpret_cast<uint32_t*>(L->packed + pl.skflag);
  L->sched = reinterpret_cast<int*>(L->packed + pl.sched);
  L->sk_epoch = 0;
  L->host_ready = false;
  L->cu_host = nullptr;
  L->cu_cap = 0;
  L->cu_pending = false;
  L->sm_count = sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& dm = L->dm;

  // bf16 layers: every packed weight is fp16, the type of the
  // intermediates it multiplies (x / RMS(x), attn, h, act); fp16 holds bf16
  // weights exactly and W_qkv * g_in within 2^-12.
  const bool f16 = L->bf16;
  launch_pack(L->bf16, wts->w_qkv, wts->g_in, L->packed + pl.wqkv, dm.Nqkv,
              dm.H, 0, f16, s);
  launch_pack(L->bf16, wts->w_o, nullptr, L->packed + pl.wo, dm.H,
              dm.Hq * dm.d, 0, f16, s);
  launch_pack(L->bf16, wts->g_post, nullptr, L->packed + pl.gpost, 1, dm.H, 0,
              false, s);
  // bf16 layers also fold g_post into the columns of W_gate_up (the fp16
  // product of two bf16 values is within 2^-12 of exact), so the MLP input
  // is h itself; the fp32 layer scales h by g_post instead.
  launch_pack(L->bf16, wts->w_gate_up, f16 ? wts->g_post : nullptr,
              L->packed + pl.wgu, 2 * dm.I, dm.H, dm.I, f16, s);
  launch_pack(L->bf16, wts->w_down, nullptr, L->packed + pl.wd, dm.H, dm.I, 0,
              f16, s);

  // RoPE table: cos / sin of p * inv_freq_i in double, stored as fp32.
  const int half = c.head_dim / 2;
  size_t n = (size_t)c.max_position * half;
  float* host = new (std::nothrow) float[2 * n];
  double* f = new (std::nothrow) double[half];
  if (!host || !f) {
    delete[] host;
    delete[] f;
    delete L;
    return LLAMA_ERR_INVALID_ARG;
  }
  rope_inv_freq(c, f);
  for (int p = 0; p < c.max_position; ++p)
    for (int i = 0; i < half; ++i) {
      double a = (double)p * f[i];
      host[(size_t)p * half + i] = (float)cos(a);
      host[n + (size_t)p * half + i] = (float)sin(a);
    }
  cudaError_t e = cudaMemcpyAsync(L->packed + pl.cos_t, host, n * 4,
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(L->packed + pl.sin_t, host + n, n * 4,
                        cudaMemcpyHostToDevice, s);
  // status word and split-tile flags start at zero
  if (e == cudaSuccess)
    e = cudaMemsetAsync(L->packed + pl.status, 0, pl.total - pl.status, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  delete[] host;
  delete[] f;
  if (e != cudaSuccess) {
    delete L;
    return LLAMA_ERR_CUDA;
  }
  if (L->bf16) {
    bool ok = tc_encode_bf16(&L->tm_wqkv, L->packed + pl.wqkv, dm.Nqkv, dm.H, 256) &&
              tc_encode_bf16(&L->tm_wo, L->packed + pl.wo, dm.H, dm.Hq * dm.d, 256) &&
              tc_encode_bf16(&L->tm_wgu, L->packed + pl.wgu, 2 * dm.I, dm.H, 256) &&
              tc_encode_bf16(&L->tm_wd, L->packed + pl.wd, dm.H, dm.I, 256) &&
              tc_encode_bf16(&L->ta_wqkv, L->packed + pl.wqkv, dm.Nqkv, dm.H, 128) &&
              tc_encode_bf16(&L->ta_wo, L->packed + pl.wo, dm.H, dm.Hq * dm.d, 128) &&
              tc_encode_bf16(&L->ta_wgu, L->packed + pl.wgu, 2 * dm.I, dm.H, 128) &&
              tc_encode_bf16(&L->ta_wd, L->packed + pl.wd, dm.H, dm.I, 128);
    if (!ok) {
      delete L;
      return LLAMA_ERR_CUDA;
    }
  }
  *out = L;
  return LLAMA_OK;
}

int llama_layer_workspace_bytes(const llama_layer_t* L, int max_tokens,
                                int decode_batch, int decode_max_seq,
                                size_t* bytes) {
  if (!L || !bytes || max_tokens < 0 || decode_batch < 0 || decode_max_seq < 0)
    return LLAMA_ERR_INVALID_ARG;
  size_t a = max_tokens > 0 ? ws_layout(L->cfg, max_tokens).total : 0;
  size_t b = decode_ws_bytes(L, decode_batch, decode_max_seq);
  *bytes = a > b ? a : b;
  if (*bytes == 0) *bytes = kAlign;
  return LLAMA_OK;
}

int llama_layer_workspace_offsets(const llama_layer_t* L, int tokens, int decode,
                                  size_t offsets[LLAMA_WS_NUM]) {
  if (!L || !offsets || tokens < 0) return LLAMA_ERR_INVALID_ARG;
  if (decode && L->bf16) {
    if (tokens > kDecodeChunk) return LLAMA_ERR_INVALID_ARG;
    DecLayout w = dec_layout(L, tokens, 1);
    offsets[0] = w.qkv;
    offsets[1] = w.attn;
    offsets[2] = w.hg;
    offsets[3] = w.act;
    return LLAMA_OK;
  }
  WsLayout w = ws_layout(L->cfg, tokens);
  offsets[0] = w.qkv;
  offsets[1] = w.attn;
  offsets[2] = L->bf16 ? w.hg : w.h;
  offsets[3] = w.act;
  return LLAMA_OK;
}

int llama_layer_forward(llama_layer_t* L, const void* x, void* out,
                        const int32_t* position_ids, const int32_t* cu_seqlens,
                        int n_seq, int seq_len, int total_tokens,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!L || !x || !out || total_tokens < 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || x == out) return LLAMA_ERR_INVALID_ARG;
  if (position_ids && !aligned(position_ids, 4)) return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens && !aligned(cu_seqlens, 4)) return LLAMA_ERR_INVALID_ARG;
  if (total_tokens == 0) return LLAMA_OK;
  if (n_seq <= 0 || seq_len <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!cu_seqlens && (long)n_seq * seq_len != total_tokens)
    return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens && (long)n_seq > total_tokens) return LLAMA_ERR_INVALID_ARG;
  if (!position_ids && seq_len > L->cfg.max_position) return LLAMA_ERR_INVALID_ARG;
  if ((size_t)seq_len * sizeof(float) > 200 * 1024) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || !aligned(workspace, kAlign)) return LLAMA_ERR_INVALID_ARG;
  if (workspace_bytes < ws_layout(L->cfg, total_tokens).total)
    return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  clobber(L, workspace, workspace_bytes);
  return forward_impl(L, x, out, position_ids, cu_seqlens, n_seq, seq_len,
                      total_tokens, static_cast<char*>(workspace),
                      static_cast<cudaStream_t>(stream));
}

int llama_layer_backward_workspace_bytes(const llama_layer_t* L, int max_tokens,
                                         size_t* bytes) {
  if (!L || !bytes || max_tokens < 0) return LLAMA_ERR_INVALID_ARG;
  if (!L->bf16) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  *bytes = max_tokens > 0 ? bwd_layout(L->cfg, max_tokens).total : kAlign;
  return LLAMA_OK;
}

// Argument checks shared by llama_layer_backward and llama_layer_backward_saved.
static int check_backward(const llama_layer_t* L, const llama_layer_weights* w, const void* x,
                          const void* dout, const void* dx, const llama_layer_grads* gr,
                          const int32_t* position_ids, const int32_t* cu_seqlens, int n_seq,
                          int seq_len, int total_tokens, const void* workspace,
                          size_t workspace_bytes) {
  if (!L || !w || !x || !dout || !dx || !gr || total_tokens < 0) return LLAMA_ERR_INVALID_ARG;
  if (!L->bf16) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  const void* in[7] = {x, dout, dx, w->w_qkv, w->w_gate_up, w->g_in, w->g_post};
  for (const void* p : in)
    if (!p || !aligned(p, 16)) return LLAMA_ERR_INVALID_ARG;
  const void* out[6] = {gr->dw_qkv, gr->dw_o, gr->dw_gate_up, gr->dw_down, gr->dg_in,
                        gr->dg_post};
  for (const void* p : out)
    if (!p || !aligned(p, 16)) return LLAMA_ERR_INVALID_ARG;
  if (dx == x || dx == dout) return LLAMA_ERR_INVALID_ARG;
  if (position_ids && !aligned(position_ids, 4)) return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens && !aligned(cu_seqlens, 4)) return LLAMA_ERR_INVALID_ARG;
  if (total_tokens == 0) return LLAMA_OK;
  if (n_seq <= 0 || seq_len <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!cu_seqlens && (long)n_seq * seq_len != total_tokens) return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens && (long)n_seq > total_tokens) return LLAMA_ERR_INVALID_ARG;
  if (!position_ids && seq_len > L->cfg.max_position) return LLAMA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, kAlign)) return LLAMA_ERR_INVALID_ARG;
  if (workspace_bytes < bwd_layout(L->cfg, total_tokens).total)
    return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  return LLAMA_OK;
}

int llama_layer_backward(llama_layer_t* L, const llama_layer_weights* w, const void* x,
                         const void* dout, void* dx, const llama_layer_grads* gr,
                         const int32_t* position_ids, const int32_t* cu_seqlens, int n_seq,
                         int seq_len, int total_tokens, void* workspace,
                         size_t workspace_bytes, void* stream) {
  int rc = check_backward(L, w, x, dout, dx, gr, position_ids, cu_seqlens, n_seq, seq_len,
                          total_tokens, workspace, workspace_bytes);
  if (rc || total_tokens == 0) return rc;
  clobber(L, workspace, workspace_bytes);
  return backward_impl(L, w, x, dout, dx, gr, position_ids, cu_seqlens, n_seq, seq_len,
                       total_tokens, static_cast<char*>(workspace),
                       static_cast<cudaStream_t>(stream), true);
}

int llama_layer_forward_train(llama_layer_t* L, const void* x, void* out,
                              const int32_t* position_ids, const int32_t* cu_seqlens,
                              int n_seq, int seq_len, int total_tokens, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!L || !x || !out || total_tokens < 0) return LLAMA_ERR_INVALID_ARG;
  if (!L->bf16) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(out, 16) || x == out) return LLAMA_ERR_INVALID_ARG;
  if (position_ids && !aligned(position_ids, 4)) return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens && !aligned(cu_seqlens, 4)) return LLAMA_ERR_INVALID_ARG;
  if (total_tokens == 0) return LLAMA_OK;
  if (n_seq <= 0 || seq_len <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!cu_seqlens && (long)n_seq * seq_len != total_tokens) return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens && (long)n_seq > total_tokens) return LLAMA_ERR_INVALID_ARG;
  if (!position_ids && seq_len > L->cfg.max_position) return LLAMA_ERR_INVALID_ARG;
  if ((size_t)seq_len * sizeof(float) > 200 * 1024) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || !aligned(workspace, kAlign)) return LLAMA_ERR_INVALID_ARG;
  const BwdLayout b = bwd_layout(L->cfg, total_tokens);
  if (workspace_bytes < b.total) return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  clobber(L, workspace, workspace_bytes);
  char* ws = static_cast<char*>(workspace);
  const FwdSaves sv = bwd_saves(b, ws);
  const int rc = forward_impl(L, x, out, position_ids, cu_seqlens, n_seq, seq_len,
                              total_tokens, ws, static_cast<cudaStream_t>(stream), &sv);
  if (rc) return rc;
  L->saved.ws = ws;
  L->saved.bytes = workspace_bytes;
  L->saved.x = x;
  L->saved.pos = position_ids;
  L->saved.cu = cu_seqlens;
  L->saved.n_seq = n_seq;
  L->saved.seq_len = seq_len;
  L->saved.tokens = total_tokens;
  L->saved.valid = true;
  return LLAMA_OK;
}

int llama_layer_backward_saved(llama_layer_t* L, const llama_layer_weights* w, const void* x,
                               const void* dout, void* dx, const llama_layer_grads* gr,
                               const int32_t* position_ids, const int32_t* cu_seqlens,
                               int n_seq, int seq_len, int total_tokens, void* workspace,
                               size_t workspace_bytes, void* stream) {
  int rc = check_backward(L, w, x, dout, dx, gr, position_ids, cu_seqlens, n_seq, seq_len,
                          total_tokens, workspace, workspace_bytes);
  if (rc || total_tokens == 0) return rc;
  const auto& sv = L->saved;
  if (!sv.valid || sv.ws != workspace || sv.x != x || sv.pos != position_ids ||
      sv.cu != cu_seqlens || sv.n_seq != n_seq || sv.seq_len != seq_len ||
      sv.tokens != total_tokens)
    return LLAMA_ERR_INVALID_ARG;
  // the backward writes only past the forward's activations: they stay
  // valid for another backward from the same forward
  return backward_impl(L, w, x, dout, dx, gr, position_ids, cu_seqlens, n_seq, seq_len,
                       total_tokens, static_cast<char*>(workspace),
                       static_cast<cudaStream_t>(stream), false);
}

namespace {

int host_setup(llama_layer* L) {
  if (L->host_ready) return LLAMA_OK;
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&L->h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&L->d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&L->ev_start, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&L->ev_done, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&L->ev_cu, ef) == cudaSuccess;
  for (int c = 0; ok && c < LLAMA_HOST_MAX_CHUNKS; ++c)
    ok = cudaEventCreateWithFlags(&L->ev_in[c], ef) == cudaSuccess &&
         cudaEventCreateWithFlags(&L->ev_comp[c], ef) == cudaSuccess;
  if (!ok) return LLAMA_ERR_CUDA;  // (the few objects made stay until exit)
  L->host_ready = true;
  return LLAMA_OK;
}

}  // namespace

int llama_layer_forward_host(llama_layer_t* L, const void* x_host, void* out_host,
                             void* x_dev, void* out_dev, const int32_t* cu_seqlens,
                             int n_seq, int seq_len, int total_tokens, int chunks,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (!L || !x_host || !out_host || chunks < 0) return LLAMA_ERR_INVALID_ARG;
  if (total_tokens == 0) return LLAMA_OK;
  // the device-side checks are llama_layer_forward's, on the whole batch
  if (!x_dev || !out_dev || total_tokens < 0 || !aligned(x_dev, 16) ||
      !aligned(out_dev, 16) || x_dev == out_dev)
    return LLAMA_ERR_INVALID_ARG;
  if (n_seq <= 0 || seq_len <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!cu_seqlens && (long)n_seq * seq_len != total_tokens) return LLAMA_ERR_INVALID_ARG;
  if (cu_seqlens) {
    // the host copy is checked here, each group's rebased copy again on the
    // device by the forward
    if ((long)n_seq > total_tokens || cu_seqlens[0] != 0 ||
        cu_seqlens[n_seq] != total_tokens)
      return LLAMA_ERR_INVALID_ARG;
    for (int i = 0; i < n_seq; ++i)
      if (cu_seqlens[i + 1] < cu_seqlens[i] || cu_seqlens[i + 1] - cu_seqlens[i] > seq_len)
        return LLAMA_ERR_INVALID_ARG;
  }
  if (seq_len > L->cfg.max_position) return LLAMA_ERR_INVALID_ARG;
  if ((size_t)seq_len * sizeof(float) > 200 * 1024) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || !aligned(workspace, kAlign)) return LLAMA_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(L->cfg, total_tokens);
  if (workspace_bytes < wl.total) return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  clobber(L, workspace, workspace_bytes);
  int rc = host_setup(L);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // groups of whole sequences.  `cut[c]` is the token count before which
  // group c starts (cut at the first sequence that starts at or after it).
  // chunks = 0: a batch of >= 16384 tokens in five groups of 1/16, 3/16,
  // 1/2, 3/16 and 1/16 of its tokens (the first group's copy in and the last
  // group's copy out are the only exposed copies, so they are kept small;
  // each next group's copy in, ~2.4x faster per token than the layer on the
  // 8B shape, hides behind the group before, and the large middle group
  // keeps the GEMMs at full size); a smaller one in groups of >= 2048 tokens
  int nc = chunks;
  long cut[LLAMA_HOST_MAX_CHUNKS + 1];
  const long T = total_tokens;
  if (chunks == 0 && T >= 16384) {
    nc = 5;
    const long sixteenths[6] = {0, 1, 4, 12, 15, 16};
    for (int c = 0; c <= nc; ++c) cut[c] = sixteenths[c] * T / 16;
  } else {
    if (nc == 0) nc = total_tokens / 2048;
    nc = std::max(1, std::min({nc, n_seq, LLAMA_HOST_MAX_CHUNKS}));
    for (int c = 0; c <= nc; ++c) cut[c] = (long)c * T / nc;
  }
  int seq0[LLAMA_HOST_MAX_CHUNKS + 1];
  seq0[0] = 0;
  seq0[nc] = n_seq;
  for (int c = 1; c < nc; ++c) {
    seq0[c] = cu_seqlens ? (int)(std::lower_bound(cu_seqlens, cu_seqlens + n_seq, cut[c]) -
                                 cu_seqlens)
                         : (int)std::min<long>(n_seq, (cut[c] + seq_len - 1) / seq_len);
    seq0[c] = std::max(seq0[c], seq0[c - 1]);
  }
  auto row0 = [&](int c) {
    return cu_seqlens ? (size_t)cu_seqlens[seq0[c]] : (size_t)seq0[c] * seq_len;
  };
  const size_t row = (size_t)L->cfg.hidden * (L->bf16 ? 2 : 4);
  // copies in: the staging buffers are free once earlier work on `stream` is
  if (cudaEventRecord(L->ev_start, s) != cudaSuccess ||
      cudaStreamWaitEvent(L->h2d, L->ev_start, 0) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  int32_t* cu_dev = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + wl.cu);
  if (cu_seqlens) {
    // group c's cu_seqlens, rebased to its first row, at entry seq0[c] + c;
    // the page-locked buffer is rewritten only after the previous call's
    // copy of it has run
    const size_t need = (size_t)n_seq + nc;
    if (L->cu_pending && cudaEventSynchronize(L->ev_cu) != cudaSuccess) return LLAMA_ERR_CUDA;
    L->cu_pending = false;
    if (L->cu_cap < need) {
      if (L->cu_host) cudaFreeHost(L->cu_host);
      L->cu_host = nullptr;
      L->cu_cap = 0;
      const size_t cap = std::max(need, (size_t)1024);
      if (cudaMallocHost(reinterpret_cast<void**>(&L->cu_host), cap * 4) != cudaSuccess)
        return LLAMA_ERR_CUDA;
      L->cu_cap = cap;
    }
    for (int c = 0; c < nc; ++c)
      for (int i = seq0[c]; i <= seq0[c + 1]; ++i)
        L->cu_host[i + c] = cu_seqlens[i] - cu_seqlens[seq0[c]];
    if (cudaMemcpyAsync(cu_dev, L->cu_host, need * 4, cudaMemcpyHostToDevice, L->h2d) !=
            cudaSuccess ||
        cudaEventRecord(L->ev_cu, L->h2d) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    L->cu_pending = true;
  }
  for (int c = 0; c < nc; ++c) {
    const size_t r0 = row0(c), r1 = row0(c + 1);
    if (r1 > r0 &&
        cudaMemcpyAsync(static_cast<char*>(x_dev) + r0 * row,
                        static_cast<const char*>(x_host) + r0 * row, (r1 - r0) * row,
                        cudaMemcpyHostToDevice, L->h2d) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    if (cudaEventRecord(L->ev_in[c], L->h2d) != cudaSuccess) return LLAMA_ERR_CUDA;
  }
  // the layer on each group as soon as its rows are in, each group's rows
  // copied out as soon as it is done (groups without rows are skipped)
  int launches = 0;
  for (int c = 0; c < nc; ++c) {
    const size_t r0 = row0(c), r1 = row0(c + 1);
    if (r1 == r0) continue;
    if (cudaStreamWaitEvent(s, L->ev_in[c], 0) != cudaSuccess) return LLAMA_ERR_CUDA;
    rc = forward_impl(L, static_cast<char*>(x_dev) + r0 * row,
                      static_cast<char*>(out_dev) + r0 * row, nullptr,
                      cu_seqlens ? cu_dev + seq0[c] + c : nullptr, seq0[c + 1] - seq0[c],
                      seq_len, (int)(r1 - r0), static_cast<char*>(workspace), s);
    if (rc) return rc;
    launches += L->launches;
    if (cudaEventRecord(L->ev_comp[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(L->d2h, L->ev_comp[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(out_host) + r0 * row,
                        static_cast<const char*>(out_dev) + r0 * row, (r1 - r0) * row,
                        cudaMemcpyDeviceToHost, L->d2h) != cudaSuccess)
      return LLAMA_ERR_CUDA;
  }
  L->launches = launches;
  // `stream` continues after the last copy out
  if (cudaEventRecord(L->ev_done, L->d2h) != cudaSuccess ||
      cudaStreamWaitEvent(s, L->ev_done, 0) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  return LLAMA_OK;
}

int llama_layer_decode(llama_layer_t* L, const void* x, void* out,
                       void* cache_k, void* cache_v, const int32_t* start_pos,
                       int batch, int max_seq, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!L || !x || !out || batch < 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || x == out) return LLAMA_ERR_INVALID_ARG;
  if (batch == 0) return LLAMA_OK;
  if (!cache_k || !cache_v || !start_pos || max_seq <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(cache_k, 16) || !aligned(cache_v, 16) || !aligned(start_pos, 4) ||
      cache_k == cache_v)
    return LLAMA_ERR_INVALID_ARG;
  if (!L->bf16 && (size_t)max_seq * sizeof(float) > 200 * 1024)
    return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || !aligned(workspace, kAlign)) return LLAMA_ERR_INVALID_ARG;
  if (workspace_bytes < decode_ws_bytes(L, batch, max_seq))
    return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  clobber(L, workspace, workspace_bytes);
  return decode_impl(L, x, out, cache_k, cache_v, start_pos, batch, max_seq,
                     static_cast<char*>(workspace),
                     static_cast<cudaStream_t>(stream));
}

int llama_layer_forward_cached(llama_layer_t* L, const void* x, void* out,
                               void* cache_k, void* cache_v, const int32_t* start_pos,
                               int batch, int seq_tokens, int max_seq, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!L || !x || !out || batch < 0 || seq_tokens <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || x == out) return LLAMA_ERR_INVALID_ARG;
  if (batch == 0) return LLAMA_OK;
  if (!cache_k || !cache_v || !start_pos || max_seq <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(cache_k, 16) || !aligned(cache_v, 16) || !aligned(start_pos, 4) ||
      cache_k == cache_v)
    return LLAMA_ERR_INVALID_ARG;
  if (seq_tokens > max_seq) return LLAMA_ERR_INVALID_ARG;
  if (!L->bf16 && seq_tokens > 1) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  const long rows = (long)batch * seq_tokens;
  if (rows > (1L << 30)) return LLAMA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, kAlign)) return LLAMA_ERR_INVALID_ARG;
  clobber(L, workspace, workspace_bytes);
  if (seq_tokens >= LLAMA_LONG_CHUNK) {
    // the prefill path over the cache: each prefix is read once per head
    // group rather than once per new token
    if ((long)batch * max_seq > (1L << 31) - 1) return LLAMA_ERR_INVALID_ARG;
    if (workspace_bytes < ws_layout(L->cfg, (int)rows).total)
      return LLAMA_ERR_WORKSPACE_TOO_SMALL;
    ChunkArgs ch{cache_k, cache_v, start_pos, max_seq};
    return forward_impl(L, x, out, nullptr, nullptr, batch, seq_tokens, (int)rows,
                        static_cast<char*>(workspace), static_cast<cudaStream_t>(stream),
                        nullptr, &ch);
  }
  if (workspace_bytes < decode_ws_bytes(L, (int)rows, max_seq))
    return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  if (!L->bf16 && (size_t)max_seq * sizeof(float) > 200 * 1024)
    return LLAMA_ERR_UNSUPPORTED_SHAPE;
  return decode_impl(L, x, out, cache_k, cache_v, start_pos, (int)rows, max_seq,
                     static_cast<char*>(workspace), static_cast<cudaStream_t>(stream),
                     seq_tokens);
}

int llama_layer_status(llama_layer_t* L, void* stream) {
  if (!L) return LLAMA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (cudaMemcpy(&word, L->status, sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return LLAMA_ERR_CUDA;
  if (cudaMemset(L->status, 0, sizeof(int)) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (word & ST_TIMEOUT) return LLAMA_ERR_DEVICE_TIMEOUT;
  if (word) return LLAMA_ERR_DEVICE_BAD_INPUT;
  return LLAMA_OK;
}

int llama_layer_set_timing(llama_layer_t* L, int ring) {
  if (!L || ring < 0 || ring > LLAMA_MAX_TIMED_CALLS) return LLAMA_ERR_INVALID_ARG;
  free_timing(L);
  if (ring == 0) return LLAMA_OK;
  const size_t n_ev = (size_t)ring * (LLAMA_MAX_STAGES + 1);
  L->ev = new (std::nothrow) cudaEvent_t[n_ev]();
  L->stage_name = new (std::nothrow) const char*[(size_t)ring * LLAMA_MAX_STAGES]();
  L->n_marks = new (std::nothrow) int[ring]();
  L->ring = ring;
  if (!L->ev || !L->stage_name || !L->n_marks) {
    free_timing(L);
    return LLAMA_ERR_INVALID_ARG;
  }
  for (size_t i = 0; i < n_ev; ++i) {
    if (cudaEventCreate(&L->ev[i]) != cudaSuccess) {
      free_timing(L);
      return LLAMA_ERR_CUDA;
    }
  }
  return LLAMA_OK;
}

int llama_layer_stage_times(llama_layer_t* L, int call, int max_stages,
                            float* ms, const char** names, int* n_stages) {
  if (!L || call < 0 || max_stages < 0 || (max_stages > 0 && !ms))
    return LLAMA_ERR_INVALID_ARG;
  if (n_stages) *n_stages = 0;
  if (!L->ring || call >= L->ring || call >= L->calls) return LLAMA_OK;
  const int c = (L->calls - 1 - call) % L->ring;
  const int n = L->n_marks[c] > 1 ? L->n_marks[c] - 1 : 0;
  if (n_stages) *n_stages = n;
  if (n == 0) return LLAMA_OK;
  const cudaEvent_t* e = L->ev + (size_t)c * (LLAMA_MAX_STAGES + 1);
  if (cudaEventSynchronize(e[n]) != cudaSuccess) return LLAMA_ERR_CUDA;
  for (int i = 0; i < n && i < max_stages; ++i) {
    if (cudaEventElapsedTime(&ms[i], e[i], e[i + 1]) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    if (names) names[i] = L->stage_name[(size_t)c * LLAMA_MAX_STAGES + i];
  }
  return LLAMA_OK;
}

int llama_layer_launch_count(const llama_layer_t* L) {
  return L ? L->launches : LLAMA_ERR_INVALID_ARG;
}

void llama_layer_destroy(llama_layer_t* L) {
  if (L) free_timing(L);
  if (L && L->host_ready) {
    cudaStreamDestroy(L->h2d);
    cudaStreamDestroy(L->d2h);
    if (L->cu_pending) cudaEventSynchronize(L->ev_cu);
    if (L->cu_host) cudaFreeHost(L->cu_host);
    cudaEventDestroy(L->ev_cu);
    cudaEventDestroy(L->ev_start);
    cudaEventDestroy(L->ev_done);
    for (int c = 0; c < LLAMA_HOST_MAX_CHUNKS; ++c) {
      cudaEventDestroy(L->ev_in[c]);
      cudaEventDestroy(L->ev_comp[c]);
    }
  }
  delete L;
}

const char* llama_layer_strerror(int code) {
  switch (code) {
    case LLAMA_OK: return "ok";
    case LLAMA_ERR_INVALID_ARG: return "invalid argument";
    case LLAMA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case LLAMA_ERR_WORKSPACE_TOO_SMALL: return "buffer too small";
    case LLAMA_ERR_CUDA: return "CUDA runtime error";
    case LLAMA_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case LLAMA_ERR_DEVICE_BAD_INPUT: return "bad cu_seqlens / positions / start_pos";
    case LLAMA_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103";
  }
  return "unknown error";
}

int llama_rmsnorm_bf16(const void* x, const void* g, void* out, int rows,
                       int hidden, float eps, void* stream) {
  if (!x || !g || !out || rows < 0 || hidden <= 0 || !(eps > 0.f))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(out, 16) || x == out)
    return LLAMA_ERR_INVALID_ARG;
  if (hidden % 128 != 0) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return LLAMA_OK;
  simt_rmsnorm_bf16(x, g, rows, hidden, eps, out, static_cast<cudaStream_t>(stream));
  return cuda_err(cudaGetLastError());
}

int llama_gemm_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (tc_take_status(&word) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (word & ST_TIMEOUT) return LLAMA_ERR_DEVICE_TIMEOUT;
  if (word) return LLAMA_ERR_DEVICE_BAD_INPUT;
  return LLAMA_OK;
}

int llama_gemm_bf16(const void* A, const void* B, void* D, int M, int N, int K,
                    void* stream) {
  if (!A || !B || !D || M < 0 || N < 0 || K <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16))
    return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 32 != 0) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return LLAMA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LLAMA_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  CUtensorMap ta, tb;
  if (!tc_encode_bf16(&ta, A, M, K, 128) || !tc_encode_bf16(&tb, B, N, K, 256))
    return LLAMA_ERR_CUDA;
  TcEpiArgs ep;
  ep.out = D;
  ep.ldo = N;
  return cuda_err(tc_gemm(TC_STORE, 256, ta, tb, M, N, K, ep, sms,
                          static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
