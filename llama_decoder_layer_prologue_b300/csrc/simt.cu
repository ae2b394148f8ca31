// Plain SIMT kernels for every stage of the layer, fp32 accumulation.
// They carry the fp32 workload (where tf32 tensor cores would not meet a
// 1e-4 error bound) and the shapes no tensor-core kernel covers.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;

// ----------------------------------------------------------------- RMSNorm
// "llama3 结构详解" 3.1: RMS(a) = sqrt(mean(a^2) + eps); one warp per row.
// Each lane reads 4 consecutive elements per step (8 or 16 bytes), 4 steps
// in flight; H is a multiple of 128.
__device__ __forceinline__ float sumsq4(const float* p) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  return v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
}
__device__ __forceinline__ float sumsq4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y);
  return a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y;
}

template <typename T>
__global__ void row_rms_kernel(const T* __restrict__ x, int rows, int H,
                               float eps, float* __restrict__ r,
                               float* __restrict__ zero) {
  pdl_trigger();
  pdl_wait();
  int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* xr = x + (size_t)row * H + lane * 4;
  float ss[4] = {0.f, 0.f, 0.f, 0.f};
  int j = 0;
  for (; j + 512 <= H; j += 512) {
#pragma unroll
    for (int u = 0; u < 4; ++u) ss[u] += sumsq4(xr + j + u * 128);
  }
  for (; j < H; j += 128) ss[0] += sumsq4(xr + j);
  float sum = warp_sum((ss[0] + ss[1]) + (ss[2] + ss[3]));
  float& ssum = sum;
  if (lane == 0) {
    r[row] = rsqrtf(ssum / (float)H + eps);
    if (zero) zero[row] = 0.f;
  }
}

// bf16 rows: r[row] = 1/RMS as above, zero[row] = 0, and the normalised row
// xn = fp16(x * r) (the operand of the QKV projection, whose packed weights
// hold g_in).  One warp per row; the second pass re-reads the row the warp
// has just read (L1).
__global__ void row_norm_f16_kernel(const __nv_bfloat16* __restrict__ x, int rows,
                                    int H, float eps, float* __restrict__ r,
                                    float* __restrict__ zero,
                                    __half* __restrict__ xn) {
  pdl_trigger();
  pdl_wait();
  int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat16* xr = x + (size_t)row * H + lane * 4;
  float ss[4] = {0.f, 0.f, 0.f, 0.f};
  int j = 0;
  for (; j + 512 <= H; j += 512) {
#pragma unroll
    for (int u = 0; u < 4; ++u) ss[u] += sumsq4(xr + j + u * 128);
  }
  for (; j < H; j += 128) ss[0] += sumsq4(xr + j);
  const float rs = rsqrtf(warp_sum((ss[0] + ss[1]) + (ss[2] + ss[3])) / (float)H + eps);
  if (lane == 0) {
    r[row] = rs;
    if (zero) zero[row] = 0.f;
  }
  __half* out = xn + (size_t)row * H + lane * 4;
  for (j = 0; j < H; j += 128) {
    const uint2 u = *reinterpret_cast<const uint2*>(xr + j);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    __half2 lo = __floats2half2_rn(a.x * rs, a.y * rs);
    __half2 hi = __floats2half2_rn(b.x * rs, b.y * rs);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + j) = o;
  }
}

// bf16 rows: out = bf16(x / RMS(x) * g), the model's final RMSNorm ("模型层"
// 9.5 / the model.py walkthrough 5: the norm before the output projection).
// One warp per row; fp32 statistics and product, one rounding.
__global__ void rmsnorm_bf16_kernel(const __nv_bfloat16* __restrict__ x,
                                    const __nv_bfloat16* __restrict__ g, int rows,
                                    int H, float eps, __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat16* xr = x + (size_t)row * H + lane * 4;
  float ss[4] = {0.f, 0.f, 0.f, 0.f};
  int j = 0;
  for (; j + 512 <= H; j += 512) {
#pragma unroll
    for (int u = 0; u < 4; ++u) ss[u] += sumsq4(xr + j + u * 128);
  }
  for (; j < H; j += 128) ss[0] += sumsq4(xr + j);
  const float rs = rsqrtf(warp_sum((ss[0] + ss[1]) + (ss[2] + ss[3])) / (float)H + eps);
  __nv_bfloat16* o = out + (size_t)row * H + lane * 4;
  const __nv_bfloat16* gl = g + lane * 4;
  for (j = 0; j < H; j += 128) {
    const uint2 u = *reinterpret_cast<const uint2*>(xr + j);
    const uint2 w = *reinterpret_cast<const uint2*>(gl + j);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    const float2 ga = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 gb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * rs * ga.x, a.y * rs * ga.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(b.x * rs * gb.x, b.y * rs * gb.y);
    uint2 r;
    r.x = *reinterpret_cast<uint32_t*>(&lo);
    r.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(o + j) = r;
  }
}

// ----------------------------------------------------------------- positions
// One block per sequence.  Checks the prefix sums; writes pos[t] = t - start.
__global__ void positions_kernel(const int32_t* __restrict__ cu, int n_seq,
                                 int seq_len, int T, int32_t* __restrict__ pos,
                                 int fill_pos, int* status) {
  pdl_trigger();
  pdl_wait();
  int s = blockIdx.x;
  int a, b;
  if (cu) {
    a = cu[s];
    b = cu[s + 1];
    bool bad = a < 0 || b < a || b > T || b - a > seq_len ||
               (s == 0 && a != 0) || (s == n_seq - 1 && b != T);
    if (bad) {
      if (threadIdx.x == 0) set_status(status, ST_BAD_SEQLENS);
      return;
    }
  } else {
    a = s * seq_len;
    b = a + seq_len;
  }
  if (!fill_pos) return;
  for (int t = a + threadIdx.x; t < b; t += blockDim.x) pos[t] = t - a;
}

// ----------------------------------------------------------------- GEMM
// 64 x 64 output tile per block, 16 x 16 threads, 4 x 4 outputs each.
constexpr int GT = 64, GK = 16;

__device__ __forceinline__ float silu_f(float x) {
  return x / (1.0f + __expf(-x));
}

template <typename T, int EPI>
__global__ void __launch_bounds__(256) gemm_kernel(
    const T* __restrict__ A, const T* __restrict__ B, T* __restrict__ out,
    int M, int N, int K, const float* __restrict__ rowscale,
    const T* __restrict__ residual) {
  __shared__ float As[GK][GT + 1];
  __shared__ float Bs[2][GK][GT + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
  constexpr int NB = EPI == EPI_SWIGLU ? 2 : 1;
  float acc[NB][4][4] = {};
  for (int k0 = 0; k0 < K; k0 += GK) {
    for (int i = threadIdx.x; i < GT * GK; i += 256) {
      int r = i / GK, c = i % GK;
      int m = m0 + r, k = k0 + c;
      As[c][r] = (m < M && k < K) ? Elem<T>::load(A + (size_t)m * K + k) : 0.f;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        int n = n0 + r;
        int brow = n;
        if (EPI == EPI_SWIGLU) brow = (n / 128) * 256 + nb * 128 + (n % 128);
        Bs[nb][c][r] = (n < N && k < K)
                           ? Elem<T>::load(B + (size_t)brow * K + k)
                           : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < GK; ++c) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[c][ty * 4 + i];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float bv = Bs[nb][c][tx * 4 + j];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[nb][i][j] = fmaf(a[i], bv, acc[nb][i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v;
      if (EPI == EPI_ROWSCALE) {
        v = rowscale[m] * acc[0][i][j];
      } else if (EPI == EPI_RESIDUAL) {
        v = Elem<T>::load(residual + (size_t)m * N + n) + acc[0][i][j];
      } else {
        float g = rowscale[m] * acc[0][i][j];
        float u = rowscale[m] * acc[NB - 1][i][j];
        v = silu_f(g) * u;
      }
      Elem<T>::store(out + (size_t)m * N + n, v);
    }
  }
}

__global__ void scale_cols_kernel(const float* __restrict__ in,
                                  const float* __restrict__ g,
                                  float* __restrict__ out, size_t n, int cols) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = in[i] * g[i % cols];
}

// ----------------------------------------------------------------- RoPE
// "RoPE高效实现": y = x cos + rotate_half(x) sin on the (i, i + d/2) pairs.
template <typename T>
__global__ void rope_kernel(T* __restrict__ qkv, int T_, Dims dm,
                            const int32_t* __restrict__ pos,
                            const float* __restrict__ cos_t,
                            const float* __restrict__ sin_t, int* status) {
  int t = blockIdx.x;
  int half = dm.d / 2;
  int p = pos[t];
  if (p < 0 || p >= dm.max_pos) {
    if (threadIdx.x == 0) set_status(status, ST_BAD_POSITION);
    p = 0;
  }
  T* row = qkv + (size_t)t * dm.Nqkv;
  int heads = dm.Hq + dm.Hkv;  // q heads then k heads
  for (int idx = threadIdx.x; idx < heads * half; idx += blockDim.x) {
    int h = idx / half, i = idx % half;
    T* x = row + h * dm.d;
    float c = cos_t[(size_t)p * half + i], s = sin_t[(size_t)p * half + i];
    float x1 = Elem<T>::load(x + i), x2 = Elem<T>::load(x + i + half);
    Elem<T>::store(x + i, x1 * c - x2 * s);
    Elem<T>::store(x + i + half, x2 * c + x1 * s);
  }
}

// ----------------------------------------------------------------- attention
__device__ float block_reduce(float v, float* red, bool is_max) {
  int lane = threadIdx.x & 31, w = threadIdx.x / 32, nw = blockDim.x / 32;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < nw; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// softmax(q k_u / sqrt(d)) v_u over n keys; keys / values `stride` elements
// apart.  Scores live in dynamic shared memory.
template <typename T>
__device__ void attend(const T* q, const T* k, const T* v, size_t stride,
                       int n, int d, T* out) {
  extern __shared__ float sc[];
  __shared__ float red[32];
  const float scale = rsqrtf((float)d);
  int lane = threadIdx.x & 31, w = threadIdx.x / 32, nw = blockDim.x / 32;
  for (int u = w; u < n; u += nw) {
    float acc = 0.f;
    for (int i = lane; i < d; i += 32)
      acc = fmaf(Elem<T>::load(q + i), Elem<T>::load(k + u * stride + i), acc);
    acc = warp_sum(acc);
    if (lane == 0) sc[u] = acc * scale;
  }
  __syncthreads();
  float m = -INFINITY;
  for (int u = threadIdx.x; u < n; u += blockDim.x) m = fmaxf(m, sc[u]);
  m = block_reduce(m, red, true);
  float l = 0.f;
  for (int u = threadIdx.x; u < n; u += blockDim.x) {
    float e = __expf(sc[u] - m);
    sc[u] = e;
    l += e;
  }
  l = block_reduce(l, red, false);
  __syncthreads();
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float acc = 0.f;
    for (int u = 0; u < n; ++u)
      acc = fmaf(sc[u], Elem<T>::load(v + u * stride + i), acc);
    Elem<T>::store(out + i, acc / l);
  }
}

template <typename T>
__global__ void attn_prefill_kernel(const T* __restrict__ qkv, T* __restrict__ attn,
                                    int T_, Dims dm, const int32_t* __restrict__ cu,
                                    int n_seq, int seq_len) {
  int t = blockIdx.x, h = blockIdx.y;
  int a;
  if (cu) {  // last sequence start <= t (binary search), clamped into [0, t]
    int lo = 0, hi = n_seq;
    while (hi - lo > 1) {
      int mid = (lo + hi) / 2;
      if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    a = min(max(cu[lo], 0), t);
  } else {
    a = (t / seq_len) * seq_len;
  }
  int g = h / (dm.Hq / dm.Hkv);
  const T* q = qkv + (size_t)t * dm.Nqkv + h * dm.d;
  const T* k = qkv + (size_t)a * dm.Nqkv + (dm.Hq + g) * dm.d;
  const T* v = qkv + (size_t)a * dm.Nqkv + (dm.Hq + dm.Hkv + g) * dm.d;
  attend(q, k, v, (size_t)dm.Nqkv, t - a + 1, dm.d,
         attn + (size_t)t * dm.Hq * dm.d + h * dm.d);
}

template <typename T>
__global__ void cache_append_kernel(const T* __restrict__ qkv, T* cache_k,
                                    T* cache_v, const int32_t* start_pos,
                                    int max_seq, Dims dm, int* status) {
  int b = blockIdx.x;
  int sp = start_pos[b];
  if (sp < 0 || sp >= max_seq || sp >= dm.max_pos) {
    if (threadIdx.x == 0) set_status(status, ST_BAD_START_POS);
    return;
  }
  int kv = dm.Hkv * dm.d;
  const T* row = qkv + (size_t)b * dm.Nqkv + dm.Hq * dm.d;
  size_t dst = ((size_t)b * max_seq + sp) * kv;
  for (int i = threadIdx.x; i < kv; i += blockDim.x) {
    cache_k[dst + i] = row[i];
    cache_v[dst + i] = row[kv + i];
  }
}

template <typename T>
__global__ void attn_decode_kernel(const T* __restrict__ qkv,
                                   const T* __restrict__ cache_k,
                                   const T* __restrict__ cache_v,
                                   T* __restrict__ attn,
                                   const int32_t* start_pos, int max_seq,
                                   Dims dm) {
  int b = blockIdx.x, h = blockIdx.y;
  int sp = start_pos[b];
  T* o = attn + (size_t)b * dm.Hq * dm.d + h * dm.d;
  if (sp < 0 || sp >= max_seq || sp >= dm.max_pos) {  // flagged by append
    for (int i = threadIdx.x; i < dm.d; i += blockDim.x) Elem<T>::store(o + i, 0.f);
    return;
  }
  int g = h / (dm.Hq / dm.Hkv);
  size_t base = (size_t)b * max_seq * dm.Hkv * dm.d + g * dm.d;
  attend(qkv + (size_t)b * dm.Nqkv + h * dm.d, cache_k + base, cache_v + base,
         (size_t)dm.Hkv * dm.d, sp + 1, dm.d, o);
}

template <typename T>
void set_smem(const void* fn, size_t bytes) {
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)bytes);
}

}  // namespace

#define DISPATCH(is_bf16, ...)          \
  do {                                  \
    if (is_bf16) {                      \
      using T = bf16;                   \
      __VA_ARGS__;                      \
    } else {                            \
      using T = float;                  \
      __VA_ARGS__;                      \
    }                                   \
  } while (0)

void simt_row_rms(bool is_bf16, const void* x, int rows, int H, float eps,
                  float* r, float* zero, cudaStream_t s) {
  if (rows <= 0) return;
  DISPATCH(is_bf16, launch_pdl(row_rms_kernel<T>, dim3((rows + 7) / 8), dim3(256), 0,
                               s, (const T*)x, rows, H, eps, r, zero));
}

// The same for rows of exactly 128 * STEPS elements, held in registers: every
// load of a lane is in flight at once and the row is read once.
template <int STEPS>
__global__ void row_norm_f16_reg_kernel(const __nv_bfloat16* __restrict__ x,
                                        int rows, float eps, float* __restrict__ r,
                                        float* __restrict__ zero,
                                        __half* __restrict__ xn) {
  pdl_trigger();
  pdl_wait();
  constexpr int H = 128 * STEPS;
  int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat16* xr = x + (size_t)row * H + lane * 4;
  uint2 u[STEPS];
#pragma unroll
  for (int j = 0; j < STEPS; ++j) u[j] = __ldg(reinterpret_cast<const uint2*>(xr + 128 * j));
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < STEPS; ++j) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j].x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j].y));
    ss = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(b.x, b.x, fmaf(b.y, b.y, ss))));
  }
  const float rs = rsqrtf(warp_sum(ss) / (float)H + eps);
  if (lane == 0) {
    r[row] = rs;
    if (zero) zero[row] = 0.f;
  }
  __half* out = xn + (size_t)row * H + lane * 4;
#pragma unroll
  for (int j = 0; j < STEPS; ++j) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j].x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j].y));
    __half2 lo = __floats2half2_rn(a.x * rs, a.y * rs);
    __half2 hi = __floats2half2_rn(b.x * rs, b.y * rs);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + 128 * j) = o;
  }
}

void simt_row_norm_f16(const void* x, int rows, int H, float eps, float* r,
                       float* zero, void* xn, cudaStream_t s) {
  if (rows <= 0) return;
  const dim3 grid((rows + 7) / 8), block(256);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* o = static_cast<__half*>(xn);
  switch (H) {
    case 1024: launch_pdl(row_norm_f16_reg_kernel<8>, grid, block, 0, s, xb, rows, eps, r, zero, o); return;
    case 2048: launch_pdl(row_norm_f16_reg_kernel<16>, grid, block, 0, s, xb, rows, eps, r, zero, o); return;
    case 3072: launch_pdl(row_norm_f16_reg_kernel<24>, grid, block, 0, s, xb, rows, eps, r, zero, o); return;
    case 4096: launch_pdl(row_norm_f16_reg_kernel<32>, grid, block, 0, s, xb, rows, eps, r, zero, o); return;
    case 5120: launch_pdl(row_norm_f16_reg_kernel<40>, grid, block, 0, s, xb, rows, eps, r, zero, o); return;
    default:
      launch_pdl(row_norm_f16_kernel, grid, block, 0, s, xb, rows, H, eps, r, zero, o);
  }
}

void simt_rmsnorm_bf16(const void* x, const void* g, int rows, int H, float eps,
                       void* out, cudaStream_t s) {
  if (rows <= 0) return;
  launch_pdl(rmsnorm_bf16_kernel, dim3((rows + 7) / 8), dim3(256), 0, s,
             static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(g),
             rows, H, eps, static_cast<__nv_bfloat16*>(out));
}

void launch_positions(const int32_t* cu, int n_seq, int seq_len, int T,
                      int32_t* pos, bool fill_pos, int* status,
                      cudaStream_t s) {
  if (n_seq <= 0) return;
  launch_pdl(positions_kernel, dim3(n_seq), dim3(256), 0, s, cu, n_seq, seq_len, T,
             pos, fill_pos ? 1 : 0, status);
}

void simt_gemm(bool is_bf16, int epi, const void* A, const void* B, void* out,
               int M, int N, int K, const float* rowscale,
               const void* residual, cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  dim3 grid((N + GT - 1) / GT, (M + GT - 1) / GT);
  DISPATCH(is_bf16, {
    if (epi == EPI_ROWSCALE)
      gemm_kernel<T, EPI_ROWSCALE><<<grid, 256, 0, s>>>(
          (const T*)A, (const T*)B, (T*)out, M, N, K, rowscale,
          (const T*)residual);
    else if (epi == EPI_RESIDUAL)
      gemm_kernel<T, EPI_RESIDUAL><<<grid, 256, 0, s>>>(
          (const T*)A, (const T*)B, (T*)out, M, N, K, rowscale,
          (const T*)residual);
    else
      gemm_kernel<T, EPI_SWIGLU><<<grid, 256, 0, s>>>(
          (const T*)A, (const T*)B, (T*)out, M, N, K, rowscale,
          (const T*)residual);
  });
}

void simt_scale_cols(const float* in, const float* g, float* out, int rows,
                     int cols, cudaStream_t s) {
  if (rows <= 0) return;
  scale_cols_kernel<<<148 * 4, 256, 0, s>>>(in, g, out, (size_t)rows * cols,
                                            cols);
}

void simt_rope(bool is_bf16, void* qkv, int ntok, const Dims& dm,
               const int32_t* pos, const float* cos_t, const float* sin_t,
               int* status, cudaStream_t s) {
  if (ntok <= 0) return;
  DISPATCH(is_bf16, rope_kernel<T><<<ntok, 256, 0, s>>>(
                        (T*)qkv, ntok, dm, pos, cos_t, sin_t, status));
}

void simt_attention_prefill(bool is_bf16, const void* qkv, void* attn,
                            int ntok, const Dims& dm, const int32_t* cu,
                            int n_seq, int seq_len, int max_keys,
                            cudaStream_t s) {
  if (ntok <= 0) return;
  size_t smem = (size_t)max_keys * sizeof(float);
  dim3 grid(ntok, dm.Hq);
  DISPATCH(is_bf16, {
    set_smem<T>((const void*)attn_prefill_kernel<T>, smem);
    attn_prefill_kernel<T><<<grid, 128, smem, s>>>(
        (const T*)qkv, (T*)attn, ntok, dm, cu, n_seq, seq_len);
  });
}

void simt_cache_append(bool is_bf16, const void* qkv, void* cache_k,
                       void* cache_v, const int32_t* start_pos, int B,
                       int max_seq, const Dims& dm, int* status,
                       cudaStream_t s) {
  if (B <= 0) return;
  DISPATCH(is_bf16, cache_append_kernel<T><<<B, 256, 0, s>>>(
                        (const T*)qkv, (T*)cache_k, (T*)cache_v, start_pos,
                        max_seq, dm, status));
}

void simt_attention_decode(bool is_bf16, const void* qkv, const void* cache_k,
                           const void* cache_v, void* attn,
                           const int32_t* start_pos, int B, int max_seq,
                           const Dims& dm, cudaStream_t s) {
  if (B <= 0) return;
  size_t smem = (size_t)max_seq * sizeof(float);
  dim3 grid(B, dm.Hq);
  DISPATCH(is_bf16, {
    set_smem<T>((const void*)attn_decode_kernel<T>, smem);
    attn_decode_kernel<T><<<grid, 128, smem, s>>>(
        (const T*)qkv, (const T*)cache_k, (const T*)cache_v, (T*)attn,
        start_pos, max_seq, dm);
  });
}

}  // namespace llama
