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

// The finalizers read the stream-K partials token-major (part[tile][slot]
// [token][128]): a warp takes one token and the 128 rows of a tile, a lane
// rows 4 lane .. 4 lane + 3, so every partial load is a 512-byte warp-wide
// float4 read and every output store runs along the token's row.  All loads
// of a thread (up to FMAXS slots, plus the epilogue's inputs) are issued
// before the first use: the kernels are latency-bound, and this keeps them
// at one or two memory round trips.
constexpr int FT = 256;            // threads per block
constexpr int FB = FT / 32;        // tokens per block (one per warp)
constexpr int FMAXS = 8;           // slots loaded per round trip

__device__ __forceinline__ bool start_ok(int sp, const DecodeArgs& a) {
  return sp >= 0 && sp < a.max_seq && sp < a.max_pos;
}

// Sequence and position of token row b of this pass.
__device__ __forceinline__ void row_seq_pos(const DecodeArgs& a, int b, int& seq,
                                            int& sp) {
  const int r = a.row0 + b;
  seq = r / a.seq_tokens;
  const int p0 = a.start_pos[seq];
  sp = p0 < 0 ? -1 : p0 + (r - seq * a.seq_tokens);  // negative stays invalid
}

// Sum over tile t's slots of rows 4 lane .. 4 lane + 3 of token b.
__device__ __forceinline__ float4 gather_rows(const DecodeArgs& a,
                                              const TcStreamK& plan, int t,
                                              int b) {
  const int nseg = tc_streamk_segments(plan, t);
  const float* src = a.part + ((size_t)t * plan.slots * a.bn + b) * 128 +
                     (threadIdx.x & 31) * 4;
  const size_t slot_stride = (size_t)a.bn * 128;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nseg; k0 += FMAXS) {
    float4 v[FMAXS];
#pragma unroll
    for (int k = 0; k < FMAXS; ++k)
      v[k] = k0 + k < nseg
                 ? __ldcg(reinterpret_cast<const float4*>(src + (k0 + k) * slot_stride))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < FMAXS; ++k) {
      acc.x += v[k].x; acc.y += v[k].y; acc.z += v[k].z; acc.w += v[k].w;
    }
  }
  return acc;
}

__device__ __forceinline__ float4 ld_bf16x4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ void st_bf16x4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ void st_f16x4(__half* p, float4 v) {
  __half2 lo = __floats2half2_rn(v.x, v.y);
  __half2 hi = __floats2half2_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// q, k, v of the new tokens (the GEMM's operand is already x / RMS(x)): RoPE
// at start_pos on q and k,
// all three -> qkv[b, :], k and v also -> cache row sp of the token's
// sequence (row_seq_pos).  Head
// boundaries fall on 4-row groups and head_dim divides 128, so the RoPE
// partner rows i +- D/2 sit D/8 lanes away in the same warp.
__global__ void __launch_bounds__(FT) finalize_qkv_kernel(DecodeArgs a,
                                                          TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, b = blockIdx.y * FB + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.batch) return;
  int seq, sp;
  row_seq_pos(a, b, seq, sp);
  float4 x = gather_rows(a, plan, t, b);
  if (!start_ok(sp, a)) {
    if (lane == 0) set_status(a.status, ST_BAD_START_POS);
    return;
  }
  const int D = a.head_dim, half = D / 2;
  const int hq = a.n_heads, hkv = a.n_kv_heads;
  const int n = t * 128 + lane * 4;
  const int head = n / D, i = n - head * D;
  const int dl = half / 4;  // partner lane offset
  float4 y;
  y.x = __shfl_xor_sync(0xffffffffu, x.x, dl);
  y.y = __shfl_xor_sync(0xffffffffu, x.y, dl);
  y.z = __shfl_xor_sync(0xffffffffu, x.z, dl);
  y.w = __shfl_xor_sync(0xffffffffu, x.w, dl);
  if (n >= a.nqkv) return;  // last tile of a width that is not 128-aligned
  if (head < hq + hkv) {
    const int ci = i < half ? i : i - half;
    const float4 c = __ldg(reinterpret_cast<const float4*>(a.cos_t + (size_t)sp * half + ci));
    const float4 sn = __ldg(reinterpret_cast<const float4*>(a.sin_t + (size_t)sp * half + ci));
    const float sg = i < half ? -1.f : 1.f;  // x c - y s (first half), x c + y s
    x = make_float4(fmaf(sg * y.x, sn.x, x.x * c.x), fmaf(sg * y.y, sn.y, x.y * c.y),
                    fmaf(sg * y.z, sn.z, x.z * c.z), fmaf(sg * y.w, sn.w, x.w * c.w));
  }
  st_bf16x4(a.qkv + (size_t)b * a.nqkv + n, x);
  if (head >= hq) {
    const int g = head < hq + hkv ? head - hq : head - hq - hkv;
    __nv_bfloat16* cache = head < hq + hkv ? a.cache_k : a.cache_v;
    st_bf16x4(cache + (((size_t)seq * a.max_seq + sp) * hkv + g) * D + i, x);
  }
}

// h = x + o_proj: fp16 copy h / 256 (operand of gate_up, whose packed
// weights hold g_post, and residual of the down projection) and the row sums
// of h^2.
__global__ void __launch_bounds__(FT) finalize_o_kernel(DecodeArgs a,
                                                        TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, b = blockIdx.y * FB + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.batch) return;
  const int H = a.hidden, n = t * 128 + lane * 4;
  const float4 xv = ld_bf16x4(a.x + (size_t)b * H + n);
  const float4 o = gather_rows(a, plan, t, b);
  const float4 h = make_float4(xv.x + o.x, xv.y + o.y, xv.z + o.z, xv.w + o.w);
  st_f16x4(a.hg + (size_t)b * H + n,
           make_float4(h.x * kHgScale, h.y * kHgScale, h.z * kHgScale, h.w * kHgScale));
  const float ss = warp_sum(h.x * h.x + h.y * h.y + h.z * h.z + h.w * h.w);
  if (lane == 0) a.ss2[(size_t)b * a.ss_np + t] = ss;  // this tile's slot
}

// act = silu(r2 gate) * (r2 up); packed tiles 2k / 2k+1 are the gate / up
// rows of act columns [128 k, 128 k + 128).
__global__ void __launch_bounds__(FT) finalize_gu_kernel(DecodeArgs a,
                                                         TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.x, b = blockIdx.y * FB + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.batch) return;
  float ss = 0.f;  // the o_proj tiles' slots, in tile order
  for (int i = 0; i < a.ss_np; ++i) ss += a.ss2[(size_t)b * a.ss_np + i];
  const float4 gs = gather_rows(a, plan, 2 * k, b);
  const float4 us = gather_rows(a, plan, 2 * k + 1, b);
  const float r2 = rsqrtf(ss * (1.0f / a.hidden) + a.eps) / kHgScale;
  float gv[4] = {gs.x, gs.y, gs.z, gs.w}, uv[4] = {us.x, us.y, us.z, us.w};
  float av[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float g = r2 * gv[q], u = r2 * uv[q];
    av[q] = g / (1.0f + __expf(-g)) * u * kActScale;
  }
  st_f16x4(a.act + (size_t)b * a.inter + k * 128 + lane * 4,
           make_float4(av[0], av[1], av[2], av[3]));
}

// out = h + down_proj, h from its fp16 copy.
__global__ void __launch_bounds__(FT) finalize_down_kernel(DecodeArgs a,
                                                           TcStreamK plan) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, b = blockIdx.y * FB + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.batch) return;
  const int H = a.hidden, n = t * 128 + lane * 4;
  const uint2 hu = __ldcg(reinterpret_cast<const uint2*>(a.hg + (size_t)b * H + n));
  const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&hu.x));
  const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&hu.y));
  constexpr float hs = 1.0f / kHgScale;
  const float4 h = make_float4(hs * h01.x, hs * h01.y, hs * h23.x, hs * h23.y);
  const float4 d = gather_rows(a, plan, t, b);
  constexpr float is = 1.0f / kActScale;
  st_bf16x4(a.out + (size_t)b * H + n,
            make_float4(fmaf(d.x, is, h.x), fmaf(d.y, is, h.y), fmaf(d.z, is, h.z),
                        fmaf(d.w, is, h.w)));
}

// ------------------------------------------------------------ attention
// Split-KV: CTA (split c, kv head g, group z) takes a.tg consecutive new
// tokens of one sequence (positions sp0 .. sp0 + ntok - 1, row_seq_pos) and
// the n_rep query heads of g for each: row R = t n_rep + r of one 16-row MMA
// tile is token t, head r.  It reads cache rows [KS c, min(KS c + KS,
// last position + 1)) of the sequence once for all of them; row R sees the
// keys up to its own token's position (the chunk's later keys are masked).
// The rows stream through a 3-stage cp.async ring of 64-key tiles; each of
// the 4 warps scores 16 keys of a tile with mma.sync (S = Q K^T), keeps its
// own online softmax (log2 domain) and P V accumulator, and the warps merge
// at the end into one (O, m, l) record per token.
constexpr int KS = 512;  // keys per split
constexpr int KT = 64;   // keys per tile
constexpr int NST = 3;   // ring stages

// Shared memory of the split-KV kernel: NST stages of K and V tiles (D / 64
// swizzle atoms of KT rows x 128 bytes each, as TMA writes them with the
// 128-byte swizzle), then the 16 padded Q rows and the stages' mbarriers.
template <int D>
struct DecSmem {
  static constexpr uint32_t TILE = KT * D * 2;  // one K or V tile
  static constexpr uint32_t P = D + 8;          // padded Q row (bf16 elements)
  static constexpr uint32_t K_OFF = 0, V_OFF = NST * TILE, Q_OFF = 2 * NST * TILE;
  static constexpr uint32_t BAR_OFF = Q_OFF + 16 * P * 2;
  static constexpr uint32_t TOTAL = BAR_OFF + 64 + 1024;  // + alignment slack
  // the warps' merge reuses the K stages: [4][16][D] fp32 O, [4][16] m, l
  static_assert(4 * 16 * D * 4 + 2 * 4 * 16 * 4 <= NST * TILE, "merge space");
};

// Byte offset of 16-byte chunk c (of the row's D / 8) of row r in a tile.
template <int D>
__device__ __forceinline__ uint32_t dec_tile_off(int r, int c) {
  return (uint32_t)((c / 8) * (KT * 128) + r * 128 + (((c % 8) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(128) attn_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                          const __grid_constant__ CUtensorMap tmV,
                                                          DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  using L = DecSmem<D>;
  constexpr int P = L::P;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + L::K_OFF;  // [NST][TILE]
  uint8_t* sV = smem + L::V_OFF;  // [NST][TILE]
  bf16* sQ = reinterpret_cast<bf16*>(smem + L::Q_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);  // [NST]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + NST);
  const int c = blockIdx.x, g = blockIdx.y, z = blockIdx.z;
  // the group's tokens: rows b0 .. b0 + ntok - 1 of the pass
  const int sq = z / a.gps, t0 = (z - sq * a.gps) * a.tg;
  const int b0 = sq * a.seq_tokens + t0;
  int seq, sp0;
  row_seq_pos(a, b0, seq, sp0);
  if (!start_ok(sp0, a)) return;
  // tokens whose positions fit the cache and the RoPE table (the rest are
  // left to the combine kernel, which writes zeros for them)
  int ntok = min(a.tg, a.seq_tokens - t0);
  while (ntok > 1 && !start_ok(sp0 + ntok - 1, a)) --ntok;
  const int n_keys = sp0 + ntok, k0 = c * KS;
  if (k0 >= n_keys) return;
  const int k1 = min(k0 + KS, n_keys);
  const int n_tiles = (k1 - k0 + KT - 1) / KT;
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int rows = ntok * n_rep;  // <= 16
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(&full[st], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // ---- Q rows (zero beyond rows)
  for (int idx = tid; idx < 16 * CH; idx += 128) {
    const int row = idx / CH, ch = idx % CH;
    const int rr = row < rows ? row : 0;
    const bf16* src = a.qkv + (size_t)(b0 + rr / n_rep) * a.nqkv +
                      (g * n_rep + rr % n_rep) * D + ch * 8;
    cp_async16(smem_u32(sQ + row * P + ch * 8), src, row < rows ? 16 : 0);
  }
  cp_async_commit();
  __syncthreads();  // the barriers are initialised
  // K / V tile j: cache rows seq * max_seq + k0 + KT j .. of kv head g, one
  // TMA box per 64 columns (rows past the tensor come back as zeros)
  const int crow = seq * a.max_seq + k0;
  auto issue = [&](int j) {
    const int st = j % NST;
    mbar_arrive_expect_tx(&full[st], 2 * L::TILE);
#pragma unroll
    for (int at = 0; at < D / 64; ++at) {
      tma_load_2d(sK + st * L::TILE + at * (KT * 128), &tmK, &full[st], g * D + at * 64,
                  crow + j * KT);
      tma_load_2d(sV + st * L::TILE + at * (KT * 128), &tmV, &full[st], g * D + at * 64,
                  crow + j * KT);
    }
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int j = 0; j < NST - 1 && j < n_tiles; ++j) issue(j);
  }
  // the last key each of this thread's two accumulator rows sees (-1: an
  // empty row)
  int lim[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int R = lane / 4 + 8 * hr;
    lim[hr] = R < rows ? sp0 + R / n_rep : -1;
  }
  cp_async_wait<0>();

  const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
  float oacc[D / 8][4] = {};
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
  bool ok = true;
  int j = 0;
  for (; j < n_tiles; ++j) {
    // stage (j - 1) % NST was released by the barrier that ended iteration j - 1
    if (tid == 0 && j + NST - 1 < n_tiles) issue(j + NST - 1);
    ok = __syncthreads_and(mbar_wait(&full[j % NST], (j / NST) & 1, a.status, abort_flag));
    if (!ok) break;
    const uint32_t tk = smem_u32(sK + (j % NST) * L::TILE);
    const uint32_t tv = smem_u32(sV + (j % NST) * L::TILE);
    if (k0 + (j + 1) * KT > k1) {
      // the split's last tile: V rows past its last key hold whatever the
      // cache holds there (P is 0 for them, but 0 * NaN would not be)
      uint8_t* vz = sV + (j % NST) * L::TILE;
      const int r0 = k1 - (k0 + j * KT);
      for (int idx = tid; idx < (KT - r0) * CH; idx += 128) {
        const int r = r0 + idx / CH, ch = idx % CH;
        *reinterpret_cast<uint4*>(vz + dec_tile_off<D>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }
    // S = Q K^T for this warp's 16 keys (2 n-tiles of 8)
    float sacc[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t af[4], bfr[4];
      ldsm_x4(af, smem_u32(sQ + (lane % 16) * P + kk * 16 + (lane / 16) * 8));
      const int krow = warp * 16 + (lane / 16) * 8 + (lane % 8);
      ldsm_x4(bfr, tk + dec_tile_off<D>(krow, kk * 2 + (lane / 8) % 2));
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
        if (key >= k1 || key > lim[e >> 1]) v = -INFINITY;
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
      ldsm_x4_t(vf, tv + dec_tile_off<D>(vrow, dt + lane / 16));
      mma_16816(oacc[dt], pf, vf[0], vf[1]);
      mma_16816(oacc[dt + 1], pf, vf[2], vf[3]);
    }
    __syncthreads();  // stage j % NST is refilled by iteration j + 1
  }
  if (!ok) {
    // a load that never landed (status already set): let the other copies
    // issued into this block's shared memory land (bounded), then leave
    if (tid == 0) {
      volatile int own = 0;
      for (int jj = j + 1; jj < n_tiles && jj < j + NST; ++jj)
        mbar_wait(&full[jj % NST], (jj / NST) & 1, a.status, &own);
    }
    __syncthreads();
    return;
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
  }
  // ---- merge the 4 warps (the group's rows only) through shared memory
  __syncthreads();
  float* sO = reinterpret_cast<float*>(sK);  // [4 warps][16 rows][D] over the K stages
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
  for (int idx = tid; idx < rows * D; idx += 128) {
    const int R = idx / D, col = idx % D;  // tile row R: token R / n_rep, head row
    const int row = R % n_rep;
    float* outp = a.attn_part +
                  (((size_t)(b0 + R / n_rep) * a.n_kv_heads + g) * a.max_chunks + c) * rec;
    float m = -INFINITY;
    for (int w = 0; w < 4; ++w) m = fmaxf(m, sM[w * 16 + R]);
    const float mr = m == -INFINITY ? 0.f : m;
    float o = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float mw = sM[w * 16 + R];
      const float mwr = mw == -INFINITY ? 0.f : mw;
      o += exp2f(mwr - mr) * sO[(w * 16 + R) * D + col];
    }
    outp[row * D + col] = o;
    if (col == 0) {
      float l = 0.f;
      for (int w = 0; w < 4; ++w) {
        const float mw = sM[w * 16 + R];
        const float mwr = mw == -INFINITY ? 0.f : mw;
        l += exp2f(mwr - mr) * sL[w * 16 + R];
      }
      outp[n_rep * D + row] = mr;
      outp[n_rep * D + n_rep + row] = l;
    }
  }
}

// attn[b, h] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the splits.
// The split weights go through shared memory (one load of every (m, l) by
// the block), then each thread's O loads over the splits are issued
// together, so the kernel costs two memory round trips for up to 8 splits.
constexpr int CT = 128;  // combine threads
__global__ void __launch_bounds__(CT) attn_combine_kernel(DecodeArgs a) {
  extern __shared__ float wsplit[];  // a.max_chunks split weights
  __shared__ float red[CT / 32];
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  const int D = a.head_dim;
  const int n_rep = a.n_heads / a.n_kv_heads;
  const int g = h / n_rep, row = h % n_rep;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __half* o = a.attn + (size_t)b * a.n_heads * D + h * D;
  int seq, sp;
  row_seq_pos(a, b, seq, sp);
  if (!start_ok(sp, a)) {
    for (int i = threadIdx.x; i < D; i += CT) o[i] = __float2half_rn(0.f);
    return;
  }
  const int nc = (sp + 1 + KS - 1) / KS;
  const float* base =
      a.attn_part + ((size_t)b * a.n_kv_heads + g) * a.max_chunks * a.n_rep_rec;
  const int moff = n_rep * D + row, loff = n_rep * D + n_rep + row;
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < nc; c += CT)
    mx = fmaxf(mx, __ldcg(base + (size_t)c * a.n_rep_rec + moff));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < CT / 32; ++w) M = fmaxf(M, red[w]);
  float den = 0.f;
  for (int c = threadIdx.x; c < nc; c += CT) {
    const float* rec = base + (size_t)c * a.n_rep_rec;
    const float w = exp2f(__ldcg(rec + moff) - M);
    wsplit[c] = w;
    den += w * __ldcg(rec + loff);
  }
  den = warp_sum(den);
  __syncthreads();  // every warp has read red[] (M) and written wsplit[]
  if (lane == 0) red[warp] = den;
  __syncthreads();
  den = red[0];
#pragma unroll
  for (int w = 1; w < CT / 32; ++w) den += red[w];
  const float inv = 1.0f / den;
  for (int i = threadIdx.x; i < D; i += CT) {
    const float* src = base + row * D + i;
    float num = 0.f;
    for (int c0 = 0; c0 < nc; c0 += 8) {
      float v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        v[c] = c0 + c < nc ? __ldcg(src + (size_t)(c0 + c) * a.n_rep_rec) : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c0 + c < nc) num = fmaf(wsplit[c0 + c], v[c], num);
    }
    o[i] = __float2half_rn(num * inv);
  }
}

}  // namespace

size_t attn_decode_smem(int head_dim) {
  return head_dim == 128 ? DecSmem<128>::TOTAL : DecSmem<64>::TOTAL;
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
  // a pass of several tokens per sequence holds whole sequences
  if (a.tg < 1 || a.gps < 1 || a.batch % a.seq_tokens != 0) return cudaErrorInvalidValue;
  dim3 grid(a.max_chunks, a.n_kv_heads, (a.batch / a.seq_tokens) * a.gps);
  // the caches as [sequences x max_seq rows, kv heads x D] bf16, up to the
  // pass's last sequence; tiles of 64 rows x 64 columns
  const uint64_t n_seq = (uint64_t)(a.row0 + a.batch - 1) / a.seq_tokens + 1;
  CUtensorMap tk, tv;
  if (!tc_encode_bf16(&tk, a.cache_k, n_seq * a.max_seq, (uint64_t)a.n_kv_heads * a.head_dim,
                      KT) ||
      !tc_encode_bf16(&tv, a.cache_v, n_seq * a.max_seq, (uint64_t)a.n_kv_heads * a.head_dim,
                      KT))
    return cudaErrorInvalidValue;
  const size_t smem = attn_decode_smem(a.head_dim);
  if (a.head_dim == 128) {
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = ensure_smem_attr(attn_decode_kernel<128>, (int)smem, attr_done);
        e != cudaSuccess)
      return e;
    cudaError_t e = launch_pdl(attn_decode_kernel<128>, grid, dim3(128), smem, s, tk, tv, a);
    if (e != cudaSuccess) return e;
  } else {
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = ensure_smem_attr(attn_decode_kernel<64>, (int)smem, attr_done);
        e != cudaSuccess)
      return e;
    cudaError_t e = launch_pdl(attn_decode_kernel<64>, grid, dim3(128), smem, s, tk, tv, a);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel, dim3(a.n_heads, a.batch), dim3(CT),
                    (size_t)a.max_chunks * sizeof(float), s, a);
}

}  // namespace llama

// ------------------------------------------------------------ long chunks
namespace llama {
namespace {

__device__ __forceinline__ bool chunk_fits(int sp, int S, int max_seq, int max_pos) {
  return sp >= 0 && sp <= max_seq - S && sp <= max_pos - S;
}

__global__ void chunk_positions_kernel(const int32_t* __restrict__ start_pos, int n_seq,
                                       int S, int max_seq, int max_pos,
                                       int32_t* __restrict__ pos, int* status) {
  pdl_trigger();
  pdl_wait();
  const int T = n_seq * S;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    const int b = t / S, i = t - b * S;
    const int sp = start_pos[b];
    const bool ok = chunk_fits(sp, S, max_seq, max_pos);
    if (!ok && i == 0) set_status(status, ST_BAD_START_POS);
    pos[t] = ok ? sp + i : 0;
  }
}

// One 16-byte piece of a row of k or v per thread: cache[b, start_pos[b] + i]
// = qkv[b * S + i, k | v columns].
__global__ void chunk_append_kernel(const __nv_bfloat16* __restrict__ qkv, int nqkv,
                                    int q_cols, int kv_cols,
                                    __nv_bfloat16* __restrict__ ck,
                                    __nv_bfloat16* __restrict__ cv,
                                    const int32_t* __restrict__ start_pos, int n_seq, int S,
                                    int max_seq, int max_pos) {
  pdl_trigger();
  pdl_wait();
  const int per_row = 2 * kv_cols / 8;
  const long long total = (long long)n_seq * S * per_row;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / per_row), w = (int)(e - (long long)t * per_row);
    const int b = t / S, i = t - b * S;
    const int sp = start_pos[b];
    if (!chunk_fits(sp, S, max_seq, max_pos)) continue;
    const bool is_v = w >= kv_cols / 8;
    const int c = (is_v ? w - kv_cols / 8 : w) * 8;
    const uint4 val = *reinterpret_cast<const uint4*>(qkv + (size_t)t * nqkv + q_cols +
                                                      (is_v ? kv_cols : 0) + c);
    __nv_bfloat16* dst = (is_v ? cv : ck) + ((size_t)b * max_seq + sp + i) * kv_cols + c;
    *reinterpret_cast<uint4*>(dst) = val;
  }
}

}  // namespace

cudaError_t chunk_positions(const int32_t* start_pos, int n_seq, int S, int max_seq,
                            int max_pos, int32_t* pos, int* status, cudaStream_t s) {
  const int T = n_seq * S;
  const int blocks = (T + 255) / 256 < 1184 ? (T + 255) / 256 : 1184;
  return launch_pdl(chunk_positions_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, s,
                    start_pos, n_seq, S, max_seq, max_pos, pos, status);
}

cudaError_t chunk_append(const __nv_bfloat16* qkv, int nqkv, int q_cols, int kv_cols,
                         __nv_bfloat16* ck, __nv_bfloat16* cv, const int32_t* start_pos,
                         int n_seq, int S, int max_seq, int max_pos, int sm_count,
                         cudaStream_t s) {
  return launch_pdl(chunk_append_kernel, dim3(sm_count * 4), dim3(256), 0, s, qkv, nqkv,
                    q_cols, kv_cols, ck, cv, start_pos, n_seq, S, max_seq, max_pos);
}

}  // namespace llama
