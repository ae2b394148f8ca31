// Internal launch interface between the C ABI (llama_layer.cu) and the kernel
// files.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llama {

// Scales of the fp16 intermediates of the bf16 layer (powers of two, so
// exact): the gate_up operand h (g_post lives in the packed W_gate_up) is
// stored times kHgScale and the SwiGLU output act times kActScale, leaving
// fp16 headroom for large hidden states; the consuming epilogues multiply
// back.
constexpr float kHgScale = 1.0f / 256.0f;
constexpr float kActScale = 1.0f / 16.0f;

struct Dims {
  int H, Hq, Hkv, d, I, Nqkv, max_pos;
  float eps;
};

// ----------------------------------------------------------------- simt.cu
// Element type T is float or __nv_bfloat16 (tag: is_bf16).
// r[row] = 1 / sqrt(mean(x[row]^2) + eps) for `rows` rows of width H; also
// zeroes zero[row] when zero is not null.
void simt_row_rms(bool is_bf16, const void* x, int rows, int H, float eps,
                  float* r, float* zero, cudaStream_t s);

// bf16 rows of width H (a multiple of 128): out = bf16(x / RMS(x) * g).
void simt_rmsnorm_bf16(const void* x, const void* g, int rows, int H, float eps,
                       void* out, cudaStream_t s);

// bf16 rows of width H (a multiple of 128): r and zero as simt_row_rms, and
// xn[row] = fp16(x[row] * r[row]).
void simt_row_norm_f16(const void* x, int rows, int H, float eps, float* r,
                       float* zero, void* xn, cudaStream_t s);

// Positions and sequence checks: pos[t] = t - start of t's sequence (when
// fill_pos), validates cu_seqlens (device) when given, else padded seq_len.
void launch_positions(const int32_t* cu, int n_seq, int seq_len, int T,
                      int32_t* pos, bool fill_pos, int* status,
                      cudaStream_t s);

// Plain GEMM-with-epilogue, fp32 accumulate, one output element per thread
// slot.  D[M, N] = A[M, K] . B[N, K]^T then:
//   EPI_ROWSCALE: out = r[m] * acc
//   EPI_RESIDUAL: out = res[m, n] + acc
//   EPI_SWIGLU:   B rows are gate/up interleaved in blocks of 128; output
//                 column j = silu(r[m] * gate_j) * (r[m] * up_j), N = I.
enum { EPI_ROWSCALE = 1, EPI_RESIDUAL = 2, EPI_SWIGLU = 3 };
void simt_gemm(bool is_bf16, int epi, const void* A, const void* B, void* out,
               int M, int N, int K, const float* rowscale,
               const void* residual, cudaStream_t s);

// out[r, c] = in[r, c] * g[c] for `rows` rows of width `cols` (fp32 path).
void simt_scale_cols(const float* in, const float* g, float* out, int rows,
                     int cols, cudaStream_t s);

// In-place RoPE on the q and k heads of qkv rows [T, Nqkv].
void simt_rope(bool is_bf16, void* qkv, int T, const Dims& dm,
               const int32_t* pos, const float* cos_t, const float* sin_t,
               int* status, cudaStream_t s);

// Prefill attention, one block per (token, q head).
void simt_attention_prefill(bool is_bf16, const void* qkv, void* attn, int T,
                            const Dims& dm, const int32_t* cu, int n_seq,
                            int seq_len, int max_keys, cudaStream_t s);

// Decode: copy k', v of every sequence into its cache row start_pos[b].
void simt_cache_append(bool is_bf16, const void* qkv, void* cache_k,
                       void* cache_v, const int32_t* start_pos, int B,
                       int max_seq, const Dims& dm, int* status,
                       cudaStream_t s);

// Decode attention over cache rows 0..start_pos[b], one block per (b, head).
void simt_attention_decode(bool is_bf16, const void* qkv, const void* cache_k,
                           const void* cache_v, void* attn,
                           const int32_t* start_pos, int B, int max_seq,
                           const Dims& dm, cudaStream_t s);

// ----------------------------------------------------------------- bwd_rows.cu
// Row passes of the backward pass (bf16 layers; H a multiple of 8):
// out = fp16(dout) [rows, H].
cudaError_t bwd_dout_f16(const void* dout, void* out, int rows, int H, int sm_count,
                         cudaStream_t s);
// dh = dout + u - h r2^2 dot / H with h = hg_scale * hg (fp16), r2 from the
// row's sum of squares: dh32 fp32 and dh16 fp16 [rows, H].  ss and dot hold
// np fixed-order slots per row, added in slot order.
cudaError_t bwd_norm2(const void* dout, const float* u, const void* hg, float hg_scale,
                      const float* ss, const float* dot, int np, float eps, float* dh32,
                      void* dh16, int rows, int H, cudaStream_t s);
// dx = bf16(dh + r1 u - x r1^3 dot / H) [rows, H] (dot: np slots per row).
cudaError_t bwd_norm1(const float* dh, const float* u, const void* x, const float* r1,
                      const float* dot, int np, void* dx, int rows, int H, cudaStream_t s);
// out_k[c] = sum over g < ng_k of part_k[g * N + c], in order, for k = 0, 1.
cudaError_t bwd_col_sums(const float* part0, int ng0, float* out0, const float* part1,
                         int ng1, float* out1, int N, cudaStream_t s);

// ----------------------------------------------------------------- pack.cu
// out[n, k] = W[src(n), k] * (g ? g[k] : 1), src(n) = n, or the gate/up
// interleave in blocks of 128 when interleave_inter > 0.  out_f16 (bf16
// input only): the packed copy is fp16 (exact for bf16 values in fp16's
// normal range).
void launch_pack(bool is_bf16, const void* W, const void* g, void* out,
                 int rows, int cols, int interleave_inter, bool out_f16,
                 cudaStream_t s);

}  // namespace llama
