// Prefill causal GQA attention (padded batch or packed varlen).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llama {

struct AttnArgs {
  const __half* qkv;         // [tokens, nqkv] fp16: q | k | v, q and k rotated
  __half* out;               // [tokens, n_heads * head_dim] fp16
  const int32_t* cu;         // [n_seq + 1] or null (padded: seq_len each)
  int tokens, seq_len, nqkv, n_heads, n_kv_heads, head_dim;
  int hpc;                   // query heads per tile (set by attn_prefill)
  int* status;               // device status word (bounded waits)
  float* lse = nullptr;      // [tokens, n_heads] or null: log2 of each row's
                             // softmax denominator in the log2(e) / sqrt(d)
                             // scaled domain (softmax = 2^(s * scale - lse))
  // attn_prefill_cached only: the keys and values come from the caller's KV
  // cache [n_seq, max_seq, n_kv_heads, head_dim] (bf16, the chunk's rows
  // already appended); qkv is then bf16 and sequence s's seq_len queries sit
  // at positions start_pos[s] .. start_pos[s] + seq_len - 1
  const __nv_bfloat16* cache_k = nullptr;
  const __nv_bfloat16* cache_v = nullptr;
  const int32_t* start_pos = nullptr;
  int max_seq = 0, max_pos = 0;
  // work-item counter pair {next, done} in device memory, zero between
  // launches (the kernel leaves it so); one pair per kernel that may overlap
  // another under programmatic dependent launch
  int* sched = nullptr;
};

// max_len: longest sequence (padded: seq_len).  Persistent over
// min(work items, sm_count) CTAs taking items dynamically (a.sched).
cudaError_t attn_prefill(const AttnArgs& a, int n_seq, int max_len,
                         int sm_count, cudaStream_t s);

// Chunked prefill against a KV cache ("llama3 结构详解" 3.2, start_pos with
// seqlen > 1): n_seq sequences of a.seq_len new tokens each (qkv rows
// s * seq_len ..), query i of sequence s attends to cache rows
// 0 .. start_pos[s] + i.  A sequence whose chunk does not fit the cache or
// the RoPE table is skipped (its rows are left as they were).
cudaError_t attn_prefill_cached(const AttnArgs& a, int n_seq, int sm_count,
                                cudaStream_t s);

}  // namespace llama
