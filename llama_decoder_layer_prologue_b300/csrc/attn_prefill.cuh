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
};

// max_len: longest sequence (padded: seq_len).  Persistent over
// min(work items, sm_count) CTAs.
cudaError_t attn_prefill(const AttnArgs& a, int n_seq, int max_len,
                         int sm_count, cudaStream_t s);

}  // namespace llama
