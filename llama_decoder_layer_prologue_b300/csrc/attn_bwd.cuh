// Backward pass of the prefill causal GQA attention (padded batch or packed
// varlen).  Host interface.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llama {

struct AttnBwdArgs {
  const __half* qkv;     // [tokens, nqkv] fp16: q | k | v of the forward, q and k rotated
  const __half* dout;    // [tokens, n_heads * head_dim] fp16: gradient of the attention output
  const float* lse;      // [tokens, n_heads]: the forward's log2 softmax denominators
  const float* dsum;     // [tokens, n_heads]: sum over d of dout * attention output
  __half* dqkv;          // [tokens, nqkv] fp16 out: dq | dk | dv before RoPE
  const int32_t* cu;     // [n_seq + 1] or null (padded: seq_len each)
  const int32_t* pos;    // [tokens] the forward's positions (RoPE)
  const float* cos_t;    // [max_pos, d/2]
  const float* sin_t;
  int tokens, seq_len, nqkv, n_heads, n_kv_heads, head_dim, max_pos;
  int hpc;               // query heads per tile (set by attn_backward)
  int* status;           // device status word (bounded waits)
  // work-item counter pairs {next, done} of the dQ and the dK / dV kernel
  // (sched[0..1], sched[2..3]), zero between launches (the kernels leave
  // them so): items are taken in order, longest range first
  int* sched = nullptr;
};

// dq (from the query tiles' side) and dk, dv (from the key tiles' side, the
// n_rep query heads of a kv head summed), each rotated back by RoPE^T and
// written into dqkv.  max_len: longest sequence.  Two persistent launches
// over min(work items, sm_count) CTAs taking items dynamically (a.sched).
cudaError_t attn_backward(const AttnBwdArgs& a, int n_seq, int max_len, int sm_count,
                          cudaStream_t s);

}  // namespace llama
