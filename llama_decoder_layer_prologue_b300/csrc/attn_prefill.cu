// Causal grouped-query attention for prefill, padded or packed varlen
// ("模型层" 9.3 CausalSelfAttention; "parallel_attention.py" 2 step 4 and 3
// flash_attn_varlen_func): o = softmax(q k^T / sqrt(d) + causal mask) v within
// each sequence, query head h reading kv head h / n_rep.
//
// One CTA = 8 warps = 128 query rows: `hpc` query heads of one kv group x
// 128 / hpc positions (16 rows per warp, all of one head).  The group's K / V
// tiles (64 keys) stream through a double-buffered cp.async ring and are
// shared by every head of the CTA (repeat_kv is never materialised).  Scores
// and P V run on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with an online
// softmax in the log2 domain; q and k arrive already rotated by the QKV GEMM
// epilogue.  CTAs are launched longest causal block first.
#include <cuda_bf16.h>
#include <math.h>

#include "attn_prefill.cuh"
#include "common.cuh"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;
constexpr int BKV = 64;  // keys per tile

template <int D>
__global__ void __launch_bounds__(256, 1) attn_prefill_kernel(AttnArgs a) {
  constexpr int P = D + 8;  // padded smem row (bf16): conflict-free ldmatrix
  constexpr int CH = D / 8;
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);  // [128][P]
  bf16* sK = sQ + 128 * P;                   // [2][BKV][P]
  bf16* sV = sK + 2 * BKV * P;               // [2][BKV][P]

  const int hpc = a.hpc, wph = 8 / hpc, BP = 16 * wph;
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest causal block first
  const int h0 = blockIdx.y * hpc;
  const int g = h0 / n_rep;
  const int s = blockIdx.z;
  int a0, L;
  if (a.cu) {
    a0 = a.cu[s];
    const int a1 = a.cu[s + 1];
    if (a0 < 0 || a1 < a0 || a1 > a.tokens) return;  // flagged by the host
    L = a1 - a0;                                      // side's check kernel
  } else {
    a0 = s * a.seq_len;
    L = a.seq_len;
  }
  const int q0 = qb * BP;
  if (q0 >= L) return;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int head = h0 + warp / wph;
  const int wp0 = q0 + (warp % wph) * 16;           // warp's first position
  const int wp_last = min(wp0 + 15, L - 1);         // last valid position
  const size_t ld = a.nqkv;
  const bf16* qkv = a.qkv;

  // ---- Q rows of the CTA (zero beyond the sequence)
  for (int idx = tid; idx < 128 * CH; idx += 256) {
    const int row = idx / CH, ch = idx % CH;
    const int rw = row / 16;
    const int hh = h0 + rw / wph, pos = q0 + (rw % wph) * 16 + (row % 16);
    const bool ok = pos < L;
    const bf16* src = qkv + (size_t)(a0 + (ok ? pos : 0)) * ld + hh * D + ch * 8;
    cp_async16(smem_u32(sQ + row * P + ch * 8), src, ok ? 16 : 0);
  }
  const bf16* kbase = qkv + (size_t)a0 * ld + (a.n_heads + g) * D;
  const bf16* vbase = qkv + (size_t)a0 * ld + (a.n_heads + a.n_kv_heads + g) * D;
  auto load_kv = [&](int j, int buf) {
    bf16* dk = sK + buf * BKV * P;
    bf16* dv = sV + buf * BKV * P;
    for (int idx = tid; idx < BKV * CH; idx += 256) {
      const int row = idx / CH, ch = idx % CH;
      const int key = j * BKV + row;
      const bool ok = key < L;
      const size_t off = (size_t)(ok ? key : 0) * ld + ch * 8;
      cp_async16(smem_u32(dk + row * P + ch * 8), kbase + off, ok ? 16 : 0);
      cp_async16(smem_u32(dv + row * P + ch * 8), vbase + off, ok ? 16 : 0);
    }
  };
  const int n_tiles = (min(q0 + BP, L) + BKV - 1) / BKV;
  load_kv(0, 0);
  cp_async_commit();

  const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
  float oacc[D / 8][4] = {};
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
  const int prow[2] = {wp0 + lane / 4, wp0 + lane / 4 + 8};

  for (int j = 0; j < n_tiles; ++j) {
    const int buf = j & 1;
    if (j + 1 < n_tiles) {
      load_kv(j + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (wp0 < L && j * BKV <= wp_last) {
      const bf16* tk = sK + buf * BKV * P;
      const bf16* tv = sV + buf * BKV * P;
      // S = Q K^T over 64 keys (8 n-tiles)
      float sacc[8][4] = {};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(af, smem_u32(sQ + (warp * 16 + (lane % 16)) * P + kk * 16 +
                             (lane / 16) * 8));
#pragma unroll
        for (int nt = 0; nt < 8; nt += 2) {
          uint32_t bfr[4];
          const int krow = (nt + lane / 16) * 8 + (lane % 8);
          ldsm_x4(bfr, smem_u32(tk + krow * P + kk * 16 + ((lane / 8) % 2) * 8));
          mma_16816(sacc[nt], af, bfr[0], bfr[1]);
          mma_16816(sacc[nt + 1], af, bfr[2], bfr[3]);
        }
      }
      // scale + causal mask + online softmax (rows prow[0], prow[1])
      const bool diag = j * BKV + BKV - 1 > wp0;  // some key above a row
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = sacc[nt][e] * scale;
          if (diag) {
            const int key = j * BKV + nt * 8 + 2 * (lane % 4) + (e & 1);
            if (key > prow[e >> 1]) v = -INFINITY;
          }
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
      for (int nt = 0; nt < 8; ++nt)
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
      // O += P V (P straight from the S accumulators as the A operand)
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk) {
        uint32_t pf[4];
        pf[0] = pack_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1]);
        pf[1] = pack_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3]);
        pf[2] = pack_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        pf[3] = pack_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int dt = 0; dt < D / 8; dt += 2) {
          uint32_t vf[4];
          const int vrow = kk * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
          ldsm_x4_t(vf, smem_u32(tv + vrow * P + dt * 8 + (lane / 16) * 8));
          mma_16816(oacc[dt], pf, vf[0], vf[1]);
          mma_16816(oacc[dt + 1], pf, vf[2], vf[3]);
        }
      }
    }
    __syncthreads();  // buffer `buf` is refilled by the next iteration
  }

  // ---- normalise and store (rows inside the sequence only)
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
  }
  const size_t ldo = (size_t)a.n_heads * D;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int pos = prow[hr];
    if (pos >= L) continue;
    const float inv = 1.0f / lrow[hr];
    bf16* o = a.out + (size_t)(a0 + pos) * ldo + head * D + 2 * (lane % 4);
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      *reinterpret_cast<uint32_t*>(o + dt * 8) =
          pack_bf16x2(oacc[dt][2 * hr] * inv, oacc[dt][2 * hr + 1] * inv);
    }
  }
}

int heads_per_cta(int n_rep) {
  int h = 8;
  while (h > 1 && n_rep % h != 0) h >>= 1;
  return h;
}

}  // namespace

cudaError_t attn_prefill(const AttnArgs& args, int n_seq, int max_len,
                         cudaStream_t s) {
  AttnArgs a = args;
  const int n_rep = a.n_heads / a.n_kv_heads;
  a.hpc = heads_per_cta(n_rep);
  const int BP = 16 * (8 / a.hpc);
  dim3 grid((max_len + BP - 1) / BP, a.n_heads / a.hpc, n_seq);
  if (grid.x == 0 || n_seq <= 0) return cudaSuccess;
  const size_t smem = (size_t)(128 + 4 * BKV) * (a.head_dim + 8) * sizeof(bf16);
  if (a.head_dim == 128) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_prefill_kernel<128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set = true;
    }
    attn_prefill_kernel<128><<<grid, 256, smem, s>>>(a);
  } else {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_prefill_kernel<64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set = true;
    }
    attn_prefill_kernel<64><<<grid, 256, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace llama
