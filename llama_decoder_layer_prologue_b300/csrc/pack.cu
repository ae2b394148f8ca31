// Weight repacking at init: fold an RMSNorm weight into the columns of the
// following projection and interleave gate / up rows for the fused SwiGLU
// epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace llama {
namespace {

// Packed row n of a gate|up weight with `inter` rows per half: blocks of 256
// packed rows hold 128 gate rows then the 128 matching up rows.
__device__ __forceinline__ int gate_up_source_row(int n, int inter) {
  int blk = n / 256, w = n % 256;
  return w < 128 ? blk * 128 + w : inter + blk * 128 + (w - 128);
}

template <typename T, typename TO>
__global__ void pack_kernel(const T* __restrict__ W, const T* __restrict__ g,
                            TO* __restrict__ out, int rows, int cols,
                            int inter) {
  size_t total = (size_t)rows * cols;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    int n = (int)(i / cols), k = (int)(i % cols);
    int src = inter > 0 ? gate_up_source_row(n, inter) : n;
    float v = Elem<T>::load(W + (size_t)src * cols + k);
    if (g) v *= Elem<T>::load(g + k);
    Elem<TO>::store(out + i, v);
  }
}

}  // namespace

void launch_pack(bool is_bf16, const void* W, const void* g, void* out,
                 int rows, int cols, int interleave_inter, bool out_f16,
                 cudaStream_t s) {
  int blocks = 148 * 8;
  if (is_bf16 && out_f16)
    pack_kernel<__nv_bfloat16, __half><<<blocks, 256, 0, s>>>(
        (const __nv_bfloat16*)W, (const __nv_bfloat16*)g, (__half*)out, rows,
        cols, interleave_inter);
  else if (is_bf16)
    pack_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, 256, 0, s>>>(
        (const __nv_bfloat16*)W, (const __nv_bfloat16*)g,
        (__nv_bfloat16*)out, rows, cols, interleave_inter);
  else
    pack_kernel<float, float><<<blocks, 256, 0, s>>>(
        (const float*)W, (const float*)g, (float*)out, rows, cols,
        interleave_inter);
}

}  // namespace llama
