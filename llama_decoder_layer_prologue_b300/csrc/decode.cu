// KV-cache decode: one new token per sequence ("llama3 结构详解" 3.2; Llama-3
// model.py walkthrough 3).  The four projections run swap-AB on the tcgen05
// GEMM (weight rows are the 128-row MMA operand, the tokens the N side) with
// a stream-K schedule; the kernels here reduce their fp32 partials and apply
// each stage's epilogue, and run the split-KV attention over the cache.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "decode.cuh"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;

// Sum over the stream-K slots of partial (output row 128 t + r, token b).
struct Partials {
  const float* base;
  int nseg, bn;
  __device__ Partials(const float* part, const TcStreamK& plan, int t, int bn_)
      : base(part + (size_t)t * plan.slots * 128 * bn_),
        nseg(tc_streamk_segments(plan, t)), bn(bn_) {}
  __device__ __forceinline__ float operator()(int r, int b) const {
    float acc = 0.f;
    for (int j = 0; j < nseg; ++j) acc += base[((size_t)j * 128 + r) * bn + b];
    return acc;
  }
};

__device__ __forceinline__ bool start_ok(int sp, const DecodeArgs& a) {
  return sp >= 0 && sp < a.max_seq && sp < a.max_pos;
}

// q, k, v of the new tokens: row scale 1/RMS, RoPE at start_pos on q and k,
// all three -> qkv[b, :], k and v also -> cache row start_pos[b].
__global__ void __launch_bounds__(128) finalize_qkv_kernel(DecodeArgs a,
                                                           TcStreamK plan) {
  const int t = blockIdx.x, r = threadIdx.x, n = t * 128 + r;
  const int D = a.head_dim, half = D / 2;
  const Partials P(a.part, plan, t, a.bn);
  const int head = n / D, i = n - head * D;
  const int hq = a.n_heads, hkv = a.n_kv_heads;
  const bool rope = head < hq + hkv;
  const int partner = i < half ? r + half : r - half;
  for (int b = 0; b < a.batch; ++b) {
    const int sp = a.start_pos[b];
    if (!start_ok(sp, a)) {
      if (t == 0 && r == 0) set_status(a.status, ST_BAD_START_POS);
      continue;
    }
    const float r1 = a.r1[b];
    float x = r1 * P(r, b);
    if (rope) {
      const float c = a.cos_t[(size_t)sp * half + (i % half)];
      const float sn = a.sin_t[(size_t)sp * half + (i % half)];
      const float y = r1 * P(partner, b);
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
__global__ void __launch_bounds__(128) finalize_o_kernel(DecodeArgs a,
                                                         TcStreamK plan) {
  const int t = blockIdx.x, r = threadIdx.x, n = t * 128 + r;
  const int H = a.hidden;
  const Partials P(a.part, plan, t, a.bn);
  for (int b = 0; b < a.batch; ++b) {
    const float h = __bfloat162float(a.x[(size_t)b * H + n]) + P(r, b);
    a.h32[(size_t)b * H + n] = h;
    a.hg[(size_t)b * H + n] =
        __float2bfloat16_rn(h * __bfloat162float(a.g_post[n]));
    const float ss = warp_sum(h * h);
    if ((threadIdx.x & 31) == 0) atomicAdd(a.ss2 + b, ss);
  }
}

// act = silu(r2 gate) * (r2 up); packed tiles 2k / 2k+1 are the gate / up
// rows of act columns [128 k, 128 k + 128).
__global__ void __launch_bounds__(128) finalize_gu_kernel(DecodeArgs a,
                                                          TcStreamK plan) {
  const int k = blockIdx.x, r = threadIdx.x;
  const Partials G(a.part, plan, 2 * k, a.bn), U(a.part, plan, 2 * k + 1, a.bn);
  const float inv_h = 1.0f / a.hidden;
  for (int b = 0; b < a.batch; ++b) {
    const float r2 = rsqrtf(a.ss2[b] * inv_h + a.eps);
    const float g = r2 * G(r, b), u = r2 * U(r, b);
    a.act[(size_t)b * a.inter + k * 128 + r] =
        __float2bfloat16_rn(g / (1.0f + __expf(-g)) * u);
  }
}

// out = h + down_proj.
__global__ void __launch_bounds__(128) finalize_down_kernel(DecodeArgs a,
                                                            TcStreamK plan) {
  const int t = blockIdx.x, r = threadIdx.x, n = t * 128 + r;
  const int H = a.hidden;
  const Partials P(a.part, plan, t, a.bn);
  for (int b = 0; b < a.batch; ++b)
    a.out[(size_t)b * H + n] =
        __float2bfloat16_rn(a.h32[(size_t)b * H + n] + P(r, b));
}

// ------------------------------------------------------------ attention
// Split-KV: CTA (chunk c, kv head g, sequence b) takes cache rows
// [128 c, min(128 c + 128, start_pos + 1)) and the n_rep query heads of g
// (rows of one 16-row MMA tile).  Each of the 4 warps scores 32 keys with
// mma.sync (S = Q K^T), takes exp2 against its own row maxima, accumulates
// P V, and the warps merge; the CTA writes (O, m, l) for the chunk.
constexpr int KC = 128;  // keys per chunk

template <int D>
__global__ void __launch_bounds__(128) attn_decode_kernel(DecodeArgs a) {
  constexpr int P = D + 8;  // padded row (bf16 elements): conflict-free ldmatrix
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + 16 * P;
  bf16* sV = sK + KC * P;
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int sp = a.start_pos[b];
  if (!start_ok(sp, a)) return;
  const int n_keys = sp + 1, k0 = c * KC;
  if (k0 >= n_keys) return;
  const int nk = min(KC, n_keys - k0);
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;

  // ---- loads: Q rows (zero beyond n_rep), K / V rows (zero beyond nk)
  constexpr int CH = D / 8;  // 16-byte chunks per row
  for (int idx = tid; idx < 16 * CH; idx += 128) {
    const int row = idx / CH, ch = idx % CH;
    const bf16* src = a.qkv + (size_t)b * a.nqkv +
                      (g * n_rep + (row < n_rep ? row : 0)) * D + ch * 8;
    cp_async16(smem_u32(sQ + row * P + ch * 8), src, row < n_rep ? 16 : 0);
  }
  const size_t row_stride = (size_t)a.n_kv_heads * D;
  const bf16* kbase = a.cache_k + ((size_t)b * a.max_seq + k0) * row_stride + g * D;
  const bf16* vbase = a.cache_v + ((size_t)b * a.max_seq + k0) * row_stride + g * D;
  for (int idx = tid; idx < KC * CH; idx += 128) {
    const int row = idx / CH, ch = idx % CH;
    const bool ok = row < nk;
    const size_t off = (ok ? (size_t)row * row_stride : 0) + ch * 8;
    cp_async16(smem_u32(sK + row * P + ch * 8), kbase + off, ok ? 16 : 0);
    cp_async16(smem_u32(sV + row * P + ch * 8), vbase + off, ok ? 16 : 0);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  // ---- S = Q K^T for this warp's 32 keys (4 n-tiles of 8)
  const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
  float sacc[4][4] = {};
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t af[4];
    ldsm_x4(af, smem_u32(sQ + (lane % 16) * P + kk * 16 + (lane / 16) * 8));
#pragma unroll
    for (int nt = 0; nt < 4; nt += 2) {
      uint32_t bf[4];
      const int krow = warp * 32 + (nt + lane / 16) * 8 + (lane % 8);
      ldsm_x4(bf, smem_u32(sK + krow * P + kk * 16 + ((lane / 8) % 2) * 8));
      mma_16816(sacc[nt], af, bf[0], bf[1]);
      mma_16816(sacc[nt + 1], af, bf[2], bf[3]);
    }
  }
  // ---- scale, mask, row max / exp2 / row sum (rows lane/4 and lane/4 + 8)
  float mrow[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = warp * 32 + nt * 8 + 2 * (lane % 4) + (e & 1);
      float v = sacc[nt][e] * scale;
      if (key >= nk) v = -INFINITY;
      sacc[nt][e] = v;
      mrow[e >> 1] = fmaxf(mrow[e >> 1], v);
    }
  float lrow[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mrow[h] = fmaxf(mrow[h], __shfl_xor_sync(0xffffffffu, mrow[h], 1));
    mrow[h] = fmaxf(mrow[h], __shfl_xor_sync(0xffffffffu, mrow[h], 2));
  }
  const float mref[2] = {mrow[0] == -INFINITY ? 0.f : mrow[0],
                         mrow[1] == -INFINITY ? 0.f : mrow[1]};
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float p = exp2f(sacc[nt][e] - mref[e >> 1]);
      sacc[nt][e] = p;
      lrow[e >> 1] += p;
    }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
  }
  // ---- O = P V (P as the A operand straight from the S accumulators)
  float oacc[D / 8][4] = {};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t pf[4];
    pf[0] = pack_bf16x2(sacc[2 * j][0], sacc[2 * j][1]);
    pf[1] = pack_bf16x2(sacc[2 * j][2], sacc[2 * j][3]);
    pf[2] = pack_bf16x2(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
    pf[3] = pack_bf16x2(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
#pragma unroll
    for (int dt = 0; dt < D / 8; dt += 2) {
      uint32_t vf[4];
      const int vrow = warp * 32 + j * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
      ldsm_x4_t(vf, smem_u32(sV + vrow * P + dt * 8 + (lane / 16) * 8));
      mma_16816(oacc[dt], pf, vf[0], vf[1]);
      mma_16816(oacc[dt + 1], pf, vf[2], vf[3]);
    }
  }
  // ---- merge the 4 warps (rows < n_rep only) through shared memory
  __syncthreads();  // K / V no longer needed: reuse them
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

// attn[b, h] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the chunks.
__global__ void attn_combine_kernel(DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int D = a.head_dim;
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int g = h / n_rep, row = h % n_rep;
  bf16* o = a.attn + (size_t)b * a.n_heads * D + h * D;
  const int sp = a.start_pos[b];
  if (!start_ok(sp, a)) {
    for (int i = threadIdx.x; i < D; i += blockDim.x) o[i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int nc = (sp + 1 + KC - 1) / KC;
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
    o[i] = __float2bfloat16_rn(num / den);
  }
}

}  // namespace

size_t attn_decode_smem(int head_dim) {
  const size_t P = head_dim + 8;
  size_t load = (16 + 2 * KC) * P * sizeof(bf16);
  size_t merge = (size_t)4 * 16 * head_dim * 4 + 2 * 4 * 16 * 4 + 16 * P * 2;
  return load > merge ? load : merge;
}

int attn_decode_chunks(int max_seq) { return (max_seq + KC - 1) / KC; }

cudaError_t decode_finalize(int stage, const DecodeArgs& a,
                            const TcStreamK& plan, cudaStream_t s) {
  switch (stage) {
    case DEC_QKV: finalize_qkv_kernel<<<plan.tiles, 128, 0, s>>>(a, plan); break;
    case DEC_O: finalize_o_kernel<<<plan.tiles, 128, 0, s>>>(a, plan); break;
    case DEC_GU: finalize_gu_kernel<<<plan.tiles / 2, 128, 0, s>>>(a, plan); break;
    case DEC_DOWN: finalize_down_kernel<<<plan.tiles, 128, 0, s>>>(a, plan); break;
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
    attn_decode_kernel<128><<<grid, 128, smem, s>>>(a);
  } else {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_decode_kernel<64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set = true;
    }
    attn_decode_kernel<64><<<grid, 128, smem, s>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3(a.n_heads, a.batch), 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace llama
