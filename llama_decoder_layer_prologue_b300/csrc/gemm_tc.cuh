// tcgen05 / TMEM GEMM fed by TMA: D = A[M, K] . B[N, K]^T, bf16 operands,
// fp32 accumulation in tensor memory, fused epilogues.  Host interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llama {

enum TcEpi : int {
  TC_STORE = 0,     // out = acc (bf16)
  TC_QKV = 1,       // out = r1[m] * acc, RoPE on q / k head columns
  TC_RESID_SS = 2,  // out = res + acc; ss_out[m] += sum over row of out^2
  TC_SWIGLU = 3,    // gate|up interleaved by 128: out = silu(r2 g) * (r2 u)
  TC_RESID = 4,     // out = res + acc
  TC_PARTIAL = 5,   // fp32 split-K partial: part[split][m][n] = acc
};

struct TcEpiArgs {
  void* out = nullptr;  // bf16 [M, ldo] (TC_SWIGLU: [M, N/2]); fp32 partials
  int ldo = 0;
  const void* residual = nullptr;  // bf16 [M, ldo]
  const float* rowscale = nullptr; // r1 [M]
  const float* ss_in = nullptr;    // sum of squares of h [M] (TC_SWIGLU)
  float* ss_out = nullptr;         // TC_RESID_SS
  float inv_h = 0.f, eps = 0.f;
  const int32_t* pos = nullptr;    // TC_QKV: position of every row
  const float* cos_t = nullptr;    // [max_pos, d/2]
  const float* sin_t = nullptr;
  int head_dim = 0, rope_cols = 0, max_pos = 0;  // rope on columns < rope_cols
  int* status = nullptr;
};

// Encodes a 2-D bf16 tensor map over a row-major [rows, cols] matrix with a
// box of box_rows x 64 elements and the 128-byte swizzle.  false on failure.
bool tc_encode_bf16(CUtensorMap* map, const void* ptr, uint64_t rows,
                    uint64_t cols, uint32_t box_rows);

// Launches the persistent GEMM.  bn in {64, 128, 256}; splits >= 1 splits K
// (TC_PARTIAL only).  Returns cudaSuccess or the launch error.
cudaError_t tc_gemm(int epi, int bn, const CUtensorMap& ta,
                    const CUtensorMap& tb, int M, int N, int K, int splits,
                    const TcEpiArgs& ep, int grid_limit, cudaStream_t s);

}  // namespace llama
