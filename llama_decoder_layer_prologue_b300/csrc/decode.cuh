// Decode-step kernels: stream-K partial finalizers and split-KV attention.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_tc.cuh"

namespace llama {

enum DecStage : int { DEC_QKV = 0, DEC_O = 1, DEC_GU = 2, DEC_DOWN = 3 };

struct DecodeArgs {
  int batch, bn;  // tokens of this pass; column stride of the GEMM partials
  // token row b of this pass is row row0 + b of the call: sequence
  // (row0 + b) / seq_tokens, position start_pos[that sequence] +
  // (row0 + b) % seq_tokens (seq_tokens = 1: one new token per sequence)
  int row0, seq_tokens;
  int hidden, n_heads, n_kv_heads, head_dim, inter, nqkv;
  int max_seq, max_pos;
  float eps;
  const float* part;  // stream-K partials of the current projection
  const __nv_bfloat16* x;  // [B, H] layer input
  const float* r1;         // [B] 1/RMS(x)
  float* ss2;              // [B, ss_np] sum of h^2 over each o_proj tile's rows
  int ss_np;               // o_proj output tiles (H / 128)
  const int32_t* start_pos;  // [sequences] of the whole call
  const float *cos_t, *sin_t;
  __nv_bfloat16* qkv;      // [B, nqkv]
  __nv_bfloat16 *cache_k, *cache_v;  // [B, max_seq, Hkv, D]
  __half* attn;            // [B, Hq * D] fp16
  float* attn_part;        // split-KV records
  int max_chunks, n_rep_rec;
  // split-KV attention groups: tg consecutive new tokens of one sequence
  // share a CTA's 16-row MMA tile (tg * n_rep <= 16), gps groups per
  // sequence; a pass of seq_tokens > 1 holds whole sequences
  int tg, gps;
  __half* hg;              // [B, H] fp16(h * kHgScale): gate_up operand, residual
  __half* act;             // [B, I] fp16(act * kActScale)
  __nv_bfloat16* out;      // [B, H]
  int* status;
};

// Reduces the partials of projection `stage` and applies its epilogue.
cudaError_t decode_finalize(int stage, const DecodeArgs& a,
                            const TcStreamK& plan, cudaStream_t s);

// Split-KV attention of every new token over cache rows 0 .. its position
// (groups of a.tg tokens of a sequence read each key once), then the
// log-sum-exp combine into a.attn.
cudaError_t decode_attention(const DecodeArgs& a, cudaStream_t s);

// Long chunks of new tokens (the tensor-core prefill attention over the
// cache): positions pos[t] = start_pos[t / S] + t % S (0 and the
// ST_BAD_START_POS bit for a chunk that does not fit the cache or the RoPE
// table), and the chunk's rotated keys and values (qkv, bf16) written into
// cache rows start_pos[b] .. start_pos[b] + S - 1.
cudaError_t chunk_positions(const int32_t* start_pos, int n_seq, int S, int max_seq,
                            int max_pos, int32_t* pos, int* status, cudaStream_t s);
cudaError_t chunk_append(const __nv_bfloat16* qkv, int nqkv, int q_cols, int kv_cols,
                         __nv_bfloat16* ck, __nv_bfloat16* cv, const int32_t* start_pos,
                         int n_seq, int S, int max_seq, int max_pos, int sm_count,
                         cudaStream_t s);

size_t attn_decode_smem(int head_dim);
int attn_decode_chunks(int max_seq);

}  // namespace llama
