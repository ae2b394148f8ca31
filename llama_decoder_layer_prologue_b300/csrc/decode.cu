// KV-cache decode: one new token per sequence ("llama3 结构详解" 3.2; Llama-3
// model.py walkthrough 3).  The four projections run swap-AB on the tcgen05
// GEMM (weight rows are the 128-row MMA operand, the tokens the N side) with
// a stream-K schedule; the kernels here reduce their fp32 partials and apply
// each stage's epilogue, and run the split-KV attention over the cache.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "decode.cuh"
#include "kernels.h"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;

// The finalizers reduce the stream-K partials of one 128-row tile for a chunk
// of FB tokens into shared memory (reads run along the tokens of one row,
// i.e. along memory), then apply the stage's epilogue with the output row as
// the fastest thread index (writes run along the token-major outputs).
constexpr int FB = 16;   // tokens per block
constexpr int FT = 256;  // threads per block
constexpr int FS = FB + 1;  // padded smem row: conflict-free column reads
constexpr int EPT = 128 * FB / FT;  // elements per thread

__device__ __forceinline__ bool start_ok(int sp, const DecodeArgs& a) {
  return sp >= 0 && sp < a.max_seq && sp < a.max_pos;
}

// s[r * FS + j] = sum over tile t's slots of partial (row r, token b0 + j).
// Slot-outer so that every thread has EPT independent loads in flight.
__device__ __forceinline__ void gather_tile(const DecodeArgs& a,
                                            const TcStreamK& plan, int t, int b0,
                                            float* s) {
  const float* base = a.part + (size_t)t * plan.slots * 128 * a.bn + b0;
  const int nseg = tc_streamk_segments(plan, t);
  const int nb = min(FB, a.batch - b0);
  float acc[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) acc[i] = 0.f;
  for (int k = 0; k < nseg; ++k) {
    const float* src = base + (size_t)k * 128 * a.bn;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const int e = threadIdx.x + i * FT, r = e / FB, j = e - r * FB;
      if (j < nb) acc[i] += src[(size_t)r * a.bn + j];
    }
  }
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int e = threadIdx.x + i * FT, r = e / FB, j = e - r * FB;
    s[r * FS + j] = acc[i];
  }
}

// q, k, v of the new tokens: row scale 1/RMS, RoPE at start_pos on q and k,
// all three -> qkv[b, :], k and v also -> cache row start_pos[b].
__global__ void __launch_bounds__(FT) finalize_qkv_kernel(DecodeArgs a,
                                                          TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s[128 * FS];
  const int t = blockIdx.x, b0 = blockIdx.y * FB;
  gather_tile(a, plan, t, b0, s);
  __syncthreads();
  const int D = a.head_dim, half = D / 2;
  const int hq = a.n_heads, hkv = a.n_kv_heads;
  const int nb = min(FB, a.batch - b0);
  for (int e = threadIdx.x; e < 128 * FB; e += FT) {
    const int r = e & 127, j = e >> 7;
    if (j >= nb) continue;
    const int b = b0 + j, n = t * 128 + r;
    if (n >= a.nqkv) continue;  // last tile of a width that is not 128-aligned
    const int head = n / D, i = n - head * D;
    const int sp = a.start_pos[b];
    if (!start_ok(sp, a)) {
      if (t == 0 && r == 0) set_status(a.status, ST_BAD_START_POS);
      continue;
    }
    const float r1 = a.r1[b];
    float x = r1 * s[r * FS + j];
    if (head < hq + hkv) {
      const int pr = i < half ? r + half : r - half;
      const float y = r1 * s[pr * FS + j];
      const float c = a.cos_t[(size_t)sp * half + (i % half)];
      const float sn = a.sin_t[(size_t)sp * half + (i % half)];
      x = i < half ? x * c - y * sn : x * c + y * sn;
    }
    const bf16 v = __float2bfloat16_rn(x);
    a.qkv[(size_t)b * a.nqkv + n] = v;
    if (head >= hq) {
      const int g = head < hq + hkv ? head - hq : head - hq - hkv;
      bf16* cache = head < hq + hkv ? a.cache_k : a.cache_v;
      cache[(((size_t)b * a.max_seq + sp) * hkv + g) * D + i] = v;
    }
  }
}

// h = x + o_proj: fp32 copy (residual of the down projection), bf16 copy of
// h * g_post (operand of gate_up) and the row sums of h^2.
__global__ void __launch_bounds__(FT) finalize_o_kernel(DecodeArgs a,
                                                        TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s[128 * FS];
  const int t = blockIdx.x, b0 = blockIdx.y * FB;
  gather_tile(a, plan, t, b0, s);
  __syncthreads();
  const int H = a.hidden;
  const int nb = min(FB, a.batch - b0);
  for (int e = threadIdx.x; e < 128 * FB; e += FT) {
    const int r = e & 127, j = e >> 7;  // a warp: 32 rows of one token
    if (j >= nb) continue;
    const int b = b0 + j, n = t * 128 + r;
    const float h = __bfloat162float(a.x[(size_t)b * H + n]) + s[r * FS + j];
    a.h32[(size_t)b * H + n] = h;
    a.hg[(size_t)b * H + n] =
        __float2half_rn(h * __bfloat162float(a.g_post[n]) * kHgScale);
    const float ss = warp_sum(h * h);
    if ((threadIdx.x & 31) == 0) atomicAdd(a.ss2 + b, ss);
  }
}

// act = silu(r2 gate) * (r2 up); packed tiles 2k / 2k+1 are the gate / up
// rows of act columns [128 k, 128 k + 128).
__global__ void __launch_bounds__(FT) finalize_gu_kernel(DecodeArgs a,
                                                         TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sg[128 * FS];
  __shared__ float su[128 * FS];
  const int k = blockIdx.x, b0 = blockIdx.y * FB;
  gather_tile(a, plan, 2 * k, b0, sg);
  gather_tile(a, plan, 2 * k + 1, b0, su);
  __syncthreads();
  const float inv_h = 1.0f / a.hidden;
  const int nb = min(FB, a.batch - b0);
  for (int e = threadIdx.x; e < 128 * FB; e += FT) {
    const int r = e & 127, j = e >> 7;
    if (j >= nb) continue;
    const int b = b0 + j;
    const float r2 = rsqrtf(a.ss2[b] * inv_h + a.eps) / kHgScale;
    const float g = r2 * sg[r * FS + j], u = r2 * su[r * FS + j];
    a.act[(size_t)b * a.inter + k * 128 + r] =
        __float2half_rn(g / (1.0f + __expf(-g)) * u * kActScale);
  }
}

// out = h + down_proj.
__global__ void __launch_bounds__(FT) finalize_down_kernel(DecodeArgs a,
                                                           TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s[128 * FS];
  const int t = blockIdx.x, b0 = blockIdx.y * FB;
  gather_tile(a, plan, t, b0, s);
  __syncthreads();
  const int H = a.hidden;
  const int nb = min(FB, a.batch - b0);
  for (int e = threadIdx.x; e < 128 * FB; e += FT) {
    const int r = e & 127, j = e >> 7;
    if (j >= nb) continue;
    const int b = b0 + j, n = t * 128 + r;
    a.out[(size_t)b * H + n] = __float2bfloat16_rn(
        fmaf(s[r * FS + j], 1.0f / kActScale, a.h32[(size_t)b * H + n]));
  }
}

// ------------------------------------------------------------ attention
// Split-KV: CTA (split c, kv head g, sequence b) takes cache rows
// [KS c, min(KS c + KS, start_pos + 1)) and the n_rep query heads of g (the
// rows of one 16-row MMA tile).  The rows stream through a 3-stage cp.async
// ring of 64-key tiles; each of the 4 warps scores 16 keys of a tile with
// mma.sync (S = Q K^T), keeps its own online softmax (log2 domain) and P V
// accumulator, and the warps merge at the end into one (O, m, l) record.
constexpr int KS = 512;  // keys per split
constexpr int KT = 64;   // keys per tile
constexpr int NST = 3;   // ring stages

template <int D>
__global__ void __launch_bounds__(128) attn_decode_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int P = D + 8;  // padded row (bf16 elements): conflict-free ldmatrix
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + 16 * P;            // [NST][KT][P]
  bf16* sV = sK + NST * KT * P;      // [NST][KT][P]
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int sp = a.start_pos[b];
  if (!start_ok(sp, a)) return;
  const int n_keys = sp + 1, k0 = c * KS;
  if (k0 >= n_keys) return;
  const int k1 = min(k0 + KS, n_keys);
  const int n_tiles = (k1 - k0 + KT - 1) / KT;
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;

  // ---- Q rows (zero beyond n_rep), part of the first cp.async group
  for (int idx = tid; idx < 16 * CH; idx += 128) {
    const int row = idx / CH, ch = idx % CH;
    const bf16* src = a.qkv + (size_t)b * a.nqkv +
                      (g * n_rep + (row < n_rep ? row : 0)) * D + ch * 8;
    cp_async16(smem_u32(sQ + row * P + ch * 8), src, row < n_rep ? 16 : 0);
  }
  const size_t row_stride = (size_t)a.n_kv_heads * D;
  const bf16* kbase = a.cache_k + (size_t)b * a.max_seq * row_stride + g * D;
  const bf16* vbase = a.cache_v + (size_t)b * a.max_seq * row_stride + g * D;
  auto load_tile = [&](int j, int st) {
    bf16* dk = sK + st * KT * P;
    bf16* dv = sV + st * KT * P;
    for (int idx = tid; idx < KT * CH; idx += 128) {
      const int row = idx / CH, ch = idx % CH;
      const int key = k0 + j * KT + row;
      const bool ok = key < k1;
      const size_t off = (ok ? (size_t)key * row_stride : 0) + ch * 8;
      cp_async16(smem_u32(dk + row * P + ch * 8), kbase + off, ok ? 16 : 0);
      cp_async16(smem_u32(dv + row * P + ch * 8), vbase + off, ok ? 16 : 0);
    }
  };
#pragma unroll
  for (int st = 0; st < NST - 1; ++st) {
    if (st < n_tiles) load_tile(st, st);
    cp_async_commit();
  }

  const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
  float oacc[D / 8][4] = {};
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
  for (int j = 0; j < n_tiles; ++j) {
    if (j + NST - 1 < n_tiles) load_tile(j + NST - 1, (j + NST - 1) % NST);
    cp_async_commit();
    cp_async_wait<NST - 1>();
    __syncthreads();
    const bf16* tk = sK + (j % NST) * KT * P;
    const bf16* tv = sV + (j % NST) * KT * P;
    // S = Q K^T for this warp's 16 keys (2 n-tiles of 8)
    float sacc[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t af[4], bfr[4];
      ldsm_x4(af, smem_u32(sQ + (lane % 16) * P + kk * 16 + (lane / 16) * 8));
      const int krow = warp * 16 + (lane / 16) * 8 + (lane % 8);
      ldsm_x4(bfr, smem_u32(tk + krow * P + kk * 16 + ((lane / 8) % 2) * 8));
      mma_16816(sacc[0], af, bfr[0], bfr[1]);
      mma_16816(sacc[1], af, bfr[2], bfr[3]);
    }
    // scale, mask, online softmax (rows lane/4 and lane/4 + 8)
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k0 + j * KT + warp * 16 + nt * 8 + 2 * (lane % 4) + (e & 1);
        float v = sacc[nt][e] * scale;
        if (key >= k1) v = -INFINITY;
        sacc[nt][e] = v;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
      }
    float alpha[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      tmax[hr] = fmaxf(tmax[hr], __shfl_xor_sync(0xffffffffu, tmax[hr], 1));
      tmax[hr] = fmaxf(tmax[hr], __shfl_xor_sync(0xffffffffu, tmax[hr], 2));
      const float mnew = fmaxf(mrow[hr], tmax[hr]);
      const float mref = mnew == -INFINITY ? 0.f : mnew;
      alpha[hr] = exp2f(mrow[hr] - mref);
      mrow[hr] = mnew;
      lrow[hr] *= alpha[hr];
      tmax[hr] = mref;
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = exp2f(sacc[nt][e] - tmax[e >> 1]);
        sacc[nt][e] = p;
        lrow[e >> 1] += p;
      }
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      oacc[dt][0] *= alpha[0];
      oacc[dt][1] *= alpha[0];
      oacc[dt][2] *= alpha[1];
      oacc[dt][3] *= alpha[1];
    }
    // O += P V over the warp's 16 keys
    uint32_t pf[4];
    pf[0] = pack_bf16x2(sacc[0][0], sacc[0][1]);
    pf[1] = pack_bf16x2(sacc[0][2], sacc[0][3]);
    pf[2] = pack_bf16x2(sacc[1][0], sacc[1][1]);
    pf[3] = pack_bf16x2(sacc[1][2], sacc[1][3]);
#pragma unroll
    for (int dt = 0; dt < D / 8; dt += 2) {
      uint32_t vf[4];
      const int vrow = warp * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
      ldsm_x4_t(vf, smem_u32(tv + vrow * P + dt * 8 + (lane / 16) * 8));
      mma_16816(oacc[dt], pf, vf[0], vf[1]);
      mma_16816(oacc[dt + 1], pf, vf[2], vf[3]);
    }
    __syncthreads();  // stage j % NST is refilled by iteration j + 1
  }
  cp_async_wait<0>();
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
  }
  // ---- merge the 4 warps (rows < n_rep only) through shared memory
  __syncthreads();
  float* sO = reinterpret_cast<float*>(sK);  // [4 warps][16 rows][D]
  float* sM = sO + 4 * 16 * D;               // [4][16]
  float* sL = sM + 4 * 16;                   // [4][16]
  const int r0 = lane / 4;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + 2 * (lane % 4);
    sO[(warp * 16 + r0) * D + col] = oacc[dt][0];
    sO[(warp * 16 + r0) * D + col + 1] = oacc[dt][1];
    sO[(warp * 16 + r0 + 8) * D + col] = oacc[dt][2];
    sO[(warp * 16 + r0 + 8) * D + col + 1] = oacc[dt][3];
  }
  if (lane % 4 == 0) {
    sM[warp * 16 + r0] = mrow[0];
    sM[warp * 16 + r0 + 8] = mrow[1];
    sL[warp * 16 + r0] = lrow[0];
    sL[warp * 16 + r0 + 8] = lrow[1];
  }
  __syncthreads();
  const int rec = a.n_rep_rec;  // floats per record: n_rep * (D + 2)
  float* outp = a.attn_part +
                (((size_t)b * a.n_kv_heads + g) * a.max_chunks + c) * rec;
  for (int idx = tid; idx < n_rep * D; idx += 128) {
    const int row = idx / D, col = idx % D;
    float m = -INFINITY;
    for (int w = 0; w < 4; ++w) m = fmaxf(m, sM[w * 16 + row]);
    const float mr = m == -INFINITY ? 0.f : m;
    float o = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float mw = sM[w * 16 + row];
      const float mwr = mw == -INFINITY ? 0.f : mw;
      o += exp2f(mwr - mr) * sO[(w * 16 + row) * D + col];
    }
    outp[row * D + col] = o;
    if (col == 0) {
      float l = 0.f;
      for (int w = 0; w < 4; ++w) {
        const float mw = sM[w * 16 + row];
        const float mwr = mw == -INFINITY ? 0.f : mw;
        l += exp2f(mwr - mr) * sL[w * 16 + row];
      }
      outp[n_rep * D + row] = mr;
      outp[n_rep * D + n_rep + row] = l;
    }
  }
}

// attn[b, h] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the splits.
__global__ void attn_combine_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  const int D = a.head_dim;
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int g = h / n_rep, row = h % n_rep;
  __half* o = a.attn + (size_t)b * a.n_heads * D + h * D;
  const int sp = a.start_pos[b];
  if (!start_ok(sp, a)) {
    for (int i = threadIdx.x; i < D; i += blockDim.x) o[i] = __float2half_rn(0.f);
    return;
  }
  const int nc = (sp + 1 + KS - 1) / KS;
  const float* base =
      a.attn_part + ((size_t)b * a.n_kv_heads + g) * a.max_chunks * a.n_rep_rec;
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c)
    M = fmaxf(M, base[(size_t)c * a.n_rep_rec + n_rep * D + row]);
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int c = 0; c < nc; ++c) {
      const float* rec = base + (size_t)c * a.n_rep_rec;
      const float w = exp2f(rec[n_rep * D + row] - M);
      num += w * rec[row * D + i];
      den += w * rec[n_rep * D + n_rep + row];
    }
    o[i] = __float2half_rn(num / den);
  }
}

}  // namespace

size_t attn_decode_smem(int head_dim) {
  const size_t P = head_dim + 8;
  size_t load = (16 + 2 * NST * KT) * P * sizeof(bf16);
  size_t merge = 16 * P * 2 + (size_t)4 * 16 * head_dim * 4 + 2 * 4 * 16 * 4;
  return load > merge ? load : merge;
}

int attn_decode_chunks(int max_seq) { return (max_seq + KS - 1) / KS; }

cudaError_t decode_finalize(int stage, const DecodeArgs& a,
                            const TcStreamK& plan, cudaStream_t s) {
  const int chunks = (a.batch + FB - 1) / FB;
  switch (stage) {
    case DEC_QKV:
      return launch_pdl(finalize_qkv_kernel, dim3(plan.tiles, chunks), dim3(FT), 0, s, a, plan);
    case DEC_O:
      return launch_pdl(finalize_o_kernel, dim3(plan.tiles, chunks), dim3(FT), 0, s, a, plan);
    case DEC_GU:
      return launch_pdl(finalize_gu_kernel, dim3(plan.tiles / 2, chunks), dim3(FT), 0, s, a,
                        plan);
    case DEC_DOWN:
      return launch_pdl(finalize_down_kernel, dim3(plan.tiles, chunks), dim3(FT), 0, s, a,
                        plan);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t decode_attention(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.max_chunks, a.n_kv_heads, a.batch);
  size_t smem = attn_decode_smem(a.head_dim);
  if (a.head_dim == 128) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_decode_kernel<128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set = true;
    }
    cudaError_t e = launch_pdl(attn_decode_kernel<128>, grid, dim3(128), smem, s, a);
    if (e != cudaSuccess) return e;
  } else {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_decode_kernel<64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set = true;
    }
    cudaError_t e = launch_pdl(attn_decode_kernel<64>, grid, dim3(128), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel, dim3(a.n_heads, a.batch), dim3(128), 0, s, a);
}

}  // namespace llama
