// Row passes of the layer's backward pass: the fp16 copy of the incoming
// gradient, and the two RMSNorm backward steps that close the residual
// branches ("模型层" 9.5 DecoderLayer: out = h + mlp(norm(h)),
// h = x + attn(norm(x)); "llama3 结构详解" 3.1 RMSNorm y = a / RMS(a) * g).
// For y = (a r) W'^T with r = (mean(a^2) + eps)^(-1/2) and the norm weight
// folded into W', the gradient u = dL/d(a r) = dy W' gives
//   da = r u - a r^3 mean(u a)            (per row),
// the GEMM epilogue that produces u also gives dot = sum(u a), as
// fixed-order slots per row (partial sums over column halves of its tiles)
// that these kernels add in slot order, like the sums of squares of h.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;

// 8 consecutive bf16 / fp16 / fp32 values.
__device__ __forceinline__ void load8_bf16(const bf16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack_bf16x2(w[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8_f16(const __half* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack_f16x2(w[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8_f32(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__global__ void dout_f16_kernel(const bf16* __restrict__ dout, __half* __restrict__ out,
                                size_t n8) {
  pdl_trigger();
  pdl_wait();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += stride) {
    float v[8];
    load8_bf16(dout + 8 * i, v);
    *reinterpret_cast<uint4*>(out + 8 * i) =
        make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                   pack_f16x2(v[6], v[7]));
  }
}

// Sum of a row's np slots, in slot order (lane-invariant).
__device__ __forceinline__ float slot_sum(const float* __restrict__ p, int np) {
  float s = 0.f;
  for (int i = 0; i < np; ++i) s += p[i];
  return s;
}

// One warp per row: dh = dout + u - h r2^2 dot / H (u already carries one
// factor r2; h = hg_scale * hg).
__global__ void norm2_bwd_kernel(const bf16* __restrict__ dout, const float* __restrict__ u,
                                 const __half* __restrict__ hg, float hg_scale,
                                 const float* __restrict__ ss, const float* __restrict__ dot,
                                 int np, float inv_h, float eps, float* __restrict__ dh32,
                                 __half* __restrict__ dh16, int rows, int H) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float r2 = rsqrtf(slot_sum(ss + (size_t)row * np, np) * inv_h + eps);
  const float c = r2 * r2 * slot_sum(dot + (size_t)row * np, np) * inv_h * hg_scale;
  const size_t base = (size_t)row * H;
  for (int col = lane * 8; col < H; col += 256) {
    float d[8], g[8], h[8];
    load8_bf16(dout + base + col, d);
    load8_f32(u + base + col, g);
    load8_f16(hg + base + col, h);
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = d[i] + g[i] - h[i] * c;
    *reinterpret_cast<float4*>(dh32 + base + col) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(dh32 + base + col + 4) = make_float4(o[4], o[5], o[6], o[7]);
    *reinterpret_cast<uint4*>(dh16 + base + col) =
        make_uint4(pack_f16x2(o[0], o[1]), pack_f16x2(o[2], o[3]), pack_f16x2(o[4], o[5]),
                   pack_f16x2(o[6], o[7]));
  }
}

// One warp per row: dx = dh + r1 u - x r1^3 dot / H.
__global__ void norm1_bwd_kernel(const float* __restrict__ dh, const float* __restrict__ u,
                                 const bf16* __restrict__ x, const float* __restrict__ r1,
                                 const float* __restrict__ dot, int np, float inv_h,
                                 bf16* __restrict__ dx, int rows, int H) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float r = r1[row];
  const float c = r * r * r * slot_sum(dot + (size_t)row * np, np) * inv_h;
  const size_t base = (size_t)row * H;
  for (int col = lane * 8; col < H; col += 256) {
    float d[8], g[8], a[8];
    load8_f32(dh + base + col, d);
    load8_f32(u + base + col, g);
    load8_bf16(x + base + col, a);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = pack_bf16x2(d[2 * i] + r * g[2 * i] - a[2 * i] * c,
                         d[2 * i + 1] + r * g[2 * i + 1] - a[2 * i + 1] * c);
    *reinterpret_cast<uint4*>(dx + base + col) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// out[c] = sum over the ng row groups of part[g * N + c] (the norm-weight
// gradients from the dW GEMMs' per-warp column sums) in a fixed order: a
// block takes 32 columns (lane = column), warp w adds groups w, w + 16, ...
// in order, and the 16 warp sums are added in warp order.  Two independent
// reductions, blockIdx.y picking one.
struct ColSums {
  const float* part[2];
  float* out[2];
  int ng[2];
};

constexpr int kColWarps = 16;

__global__ void __launch_bounds__(kColWarps * 32) col_sums_kernel(ColSums a, int N) {
  __shared__ float ws[kColWarps][32];
  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.y, warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  float s0 = 0.f, s1 = 0.f;  // alternate groups: two chains, a fixed pairing
  if (c < N) {
    const float* p = a.part[k] + c;
    int g = warp;
    for (; g + kColWarps < a.ng[k]; g += 2 * kColWarps) {
      s0 += p[(size_t)g * N];
      s1 += p[(size_t)(g + kColWarps) * N];
    }
    if (g < a.ng[k]) s0 += p[(size_t)g * N];
  }
  ws[warp][lane] = s0 + s1;
  __syncthreads();
  if (warp == 0 && c < N) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kColWarps; ++w) t += ws[w][lane];
    a.out[k][c] = t;
  }
}

}  // namespace

cudaError_t bwd_dout_f16(const void* dout, void* out, int rows, int H, int sm_count,
                         cudaStream_t s) {
  const size_t n8 = (size_t)rows * H / 8;
  return launch_pdl(dout_f16_kernel, dim3(sm_count * 4), dim3(256), 0, s,
                    static_cast<const bf16*>(dout), static_cast<__half*>(out), n8);
}

cudaError_t bwd_norm2(const void* dout, const float* u, const void* hg, float hg_scale,
                      const float* ss, const float* dot, int np, float eps, float* dh32,
                      void* dh16, int rows, int H, cudaStream_t s) {
  return launch_pdl(norm2_bwd_kernel, dim3((rows + 7) / 8), dim3(256), 0, s,
                    static_cast<const bf16*>(dout), u, static_cast<const __half*>(hg), hg_scale,
                    ss, dot, np, 1.0f / H, eps, dh32, static_cast<__half*>(dh16), rows, H);
}

cudaError_t bwd_norm1(const float* dh, const float* u, const void* x, const float* r1,
                      const float* dot, int np, void* dx, int rows, int H, cudaStream_t s) {
  return launch_pdl(norm1_bwd_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, dh, u,
                    static_cast<const bf16*>(x), r1, dot, np, 1.0f / H, static_cast<bf16*>(dx),
                    rows, H);
}

cudaError_t bwd_col_sums(const float* part0, int ng0, float* out0, const float* part1, int ng1,
                         float* out1, int N, cudaStream_t s) {
  ColSums a;
  a.part[0] = part0; a.part[1] = part1;
  a.out[0] = out0; a.out[1] = out1;
  a.ng[0] = ng0; a.ng[1] = ng1;
  return launch_pdl(col_sums_kernel, dim3((N + 31) / 32, 2), dim3(kColWarps * 32), 0, s, a,
                    N);
}

}  // namespace llama
