// Persistent tcgen05 GEMM for sm_103a.
//
// One CTA per SM, 10 warps:
//   warp 0      TMA producer: A / B K-slices (64 bf16 = one 128-byte swizzle
//               row) into a STAGES-deep shared-memory ring (mbarrier full /
//               empty pairs).
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               (M = 128, N = BN, K = 16) into one of two TMEM accumulators
//               and commits each ring slot back to the producer.
//   warps 2..9  epilogue: tcgen05.ld of their 32 TMEM lanes (one output row
//               per thread; two warps per lane quadrant, each taking half of
//               the tile's columns), fused epilogue, stores.  The two
//               accumulators let the epilogue of tile i overlap the main loop
//               of tile i + 1.
// The layer's GEMMs run as CTA pairs (clusters of 2, CG2 below): rank 0's
// MMA thread issues one M = 256 tcgen05.mma.cta_group::2 per K step over
// both CTAs' shared memory and tensor memory.  Tiles are visited in bands of
// M-tiles sized by L2 (tc_group_m) so that a wave of CTAs shares A and B
// slices in L2.  Every wait is bounded (see mbar_wait).
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "gemm_tc.cuh"

namespace llama {
namespace {

constexpr int BM = 128, BK = 64;
// warp 0 producer, warp 1 MMA, warps 2..9 epilogue (two per TMEM lane
// quadrant, each on half of the tile's columns)
constexpr int kEpiWarps = 8, kGemmThreads = 64 + 32 * kEpiWarps;

// Status word of the GEMMs launched without a layer (llama_gemm_bf16,
// llama_gemm_bf16_streamk_static), one per device; read and cleared by
// tc_take_status.
__device__ int g_tc_status;

// HALF_B: each CTA of a cta_group::2 pair holds BN / 2 rows of the B slice.
template <int BN, int STAGES, bool HALF_B = false>
struct Layout {
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = (HALF_B ? BN / 2 : BN) * BK * 2;
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t BAR_OFF = STAGES * STAGE;
  static constexpr uint32_t TOTAL = BAR_OFF + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

// Tile t of a whole-tile schedule visited in bands of group_m M-tiles (all
// N-tiles of a band before the next band).
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int group_m,
                                            int& m, int& n) {
  int group = group_m * n_tiles;
  int g = t / group;
  int first_m = g * group_m;
  int gm = min(m_tiles - first_m, group_m);
  int w = t - g * group;
  m = first_m + w % gm;
  n = w / gm;
}

// 256-bit global accesses (sm_100 and later): a lane moves one whole
// 32-byte sector, so a warp's 32 row-accesses of one chunk are 32 full
// sectors.  The 128-bit forms serve pointers that are only 16-byte aligned.
// Both are volatile so that they keep their place relative to the mbarrier
// waits and TMEM loads (a load issued before a wait overlaps it).
__device__ __forceinline__ void ld_v8(const void* p, uint32_t* u) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]),
                 "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
               : "l"(p));
}

__device__ __forceinline__ void ld_v4(const void* p, uint32_t* u) {
  asm volatile("ld.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3])
               : "l"(p));
}

__device__ __forceinline__ void st_v8(void* p, const uint32_t* u) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
               "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]),
               "r"(u[6]), "r"(u[7])
               : "memory");
}

__device__ __forceinline__ void st_v4(void* p, const uint32_t* u) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(u[0]),
               "r"(u[1]), "r"(u[2]), "r"(u[3])
               : "memory");
}

// `words` (a multiple of 8) 32-bit words at p, 32-byte or 16-byte accesses.
template <int WORDS>
__device__ __forceinline__ void ld_words(const void* p, uint32_t* u, bool v8) {
  const char* c = static_cast<const char*>(p);
  if (v8) {
#pragma unroll
    for (int i = 0; i < WORDS / 8; ++i) ld_v8(c + 32 * i, u + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < WORDS / 4; ++i) ld_v4(c + 16 * i, u + 4 * i);
  }
}

template <int WORDS>
__device__ __forceinline__ void st_words(void* p, const uint32_t* u, bool v8) {
  char* c = static_cast<char*>(p);
  if (v8) {
#pragma unroll
    for (int i = 0; i < WORDS / 8; ++i) st_v8(c + 32 * i, u + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < WORDS / 4; ++i) st_v4(c + 16 * i, u + 4 * i);
  }
}

// 32 values as 16-bit elements (fp16 or bf16) at element offset `off` of p.
__device__ __forceinline__ void store_16x32(void* p, size_t off, const float* v,
                                            bool f16, bool v8) {
  uint32_t u[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    u[i] = f16 ? pack_f16x2(v[2 * i], v[2 * i + 1]) : pack_bf16x2(v[2 * i], v[2 * i + 1]);
  st_words<16>(static_cast<char*>(p) + 2 * off, u, v8);
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

// Residual words (16-bit pairs) per 32-column chunk; every chunk of the
// part is loaded before the accumulator wait.
constexpr int kResidWords = 16;

// Inputs of one tile's epilogue that do not depend on the accumulator,
// loaded before waiting for it: the residual of the first column chunk, the
// row's RMS statistics, its RoPE position and cos / sin of the first chunk.
struct EpiPre {
  uint32_t w[64];           // residual chunks (bf16 / fp16 pairs)
  uint32_t cs[32], sn[32];  // TC_QKV: cos / sin (fp32 bits) of frequencies 0..31
  float f;               // TC_QKV: 1/RMS; TC_SWIGLU: sum of h^2
  int p;                 // TC_QKV: position
};

// Column chunks of 32 that this epilogue warp covers: [c_begin, c_end).
template <int BN>
__device__ __forceinline__ int chunk_begin(int part) { return part * (BN / 64); }

template <int BN, int EPI>
__device__ __forceinline__ void epilogue_prefetch(EpiPre& pre, int row, bool valid,
                                                  int n0, int N, int part,
                                                  const TcEpiArgs& ep) {
  if (!valid) return;
  if constexpr (EPI == TC_RESID_SS || EPI == TC_RESID || EPI == TC_F32_DOT ||
                EPI == TC_DO) {
    // every chunk of the part's 16-bit residual (bf16 x for TC_RESID_SS,
    // the fp16 copy of h for TC_RESID, h or x for TC_F32_DOT, the attention
    // output for TC_DO)
    constexpr int RW = kResidWords;
    const int cb = chunk_begin<BN>(part);
#pragma unroll
    for (int k = 0; k < BN / 64; ++k) {
      const int col = n0 + (cb + k) * 32;
      if (col >= N) break;
      const size_t off = (size_t)row * ep.ldo + col;
      ld_words<RW>(static_cast<const uint16_t*>(ep.residual) + off, pre.w + k * RW,
                   EPI == TC_RESID ? true : ep.vec32 != 0);
    }
  } else if constexpr (EPI == TC_QKV) {
    pre.f = ep.rowscale ? ep.rowscale[row] : 1.f;
    int p = ep.pos[row];
    if (p < 0 || p >= ep.max_pos) {
      set_status(ep.status, ST_BAD_POSITION);
      p = 0;
    }
    pre.p = p;
    const int half = ep.head_dim / 2;
    ld_words<32>(ep.cos_t + (size_t)p * half, pre.cs, true);
    ld_words<32>(ep.sin_t + (size_t)p * half, pre.sn, true);
  } else if constexpr (EPI == TC_SWIGLU || EPI == TC_SWIGLU_BWD) {
    // the row's sum of squares from its slots, added in slot order
    const float* sp = ep.ss_in + (size_t)row * ep.ss_np;
    float sum = 0.f;
    for (int i = 0; i < ep.ss_np; ++i) sum += sp[i];
    pre.f = sum;
  }
}

// Column sums over the 32 rows of a warp: v[j] holds lane's value of column
// j; afterwards v[0] of lane l holds the sum over all lanes of column l
// (recursive halving: each step trades half of the remaining columns with
// the lane `off` away, 31 shuffles in all).
__device__ __forceinline__ void warp_column_sums(float* v, int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

// Source row of packed gate|up row n (blocks of 256 packed rows: 128 gate
// rows, then the 128 matching up rows).
__device__ __forceinline__ int gate_up_row(int n, int inter) {
  const int blk = n / 256, w = n % 256;
  return w < 128 ? blk * 128 + w : inter + blk * 128 + (w - 128);
}

// Adds the other piece of a split tile (fp32 row `fin`) into this thread's
// TMEM row before the epilogue reads it: exactly the 32-column chunks that
// this warp's epilogue reads (TC_SWIGLU: gate chunks 2 part, 2 part + 1 and
// the matching up chunks 4 + 2 part, 5 + 2 part; otherwise the part's four
// chunks), so no other warp's reads depend on it.
template <int BN, int EPI>
__device__ __forceinline__ void add_partial_tmem(uint32_t t_row, const float* fin,
                                                 int part) {
#pragma unroll 1
  for (int k = 0; k < BN / 64; ++k) {
    const int c = EPI == TC_SWIGLU ? (k < 2 ? 2 * part + k : 4 + 2 * part + (k - 2))
                                   : part * (BN / 64) + k;
    uint32_t u[32];
    ld_words<32>(fin + c * 32, u, true);
    float v[32];
    tmem_ld32(t_row + c * 32, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += __uint_as_float(u[j]);
    tmem_st32(t_row + c * 32, v);  // waits for the store
  }
}

// Epilogue of one accumulator row (TMEM lane) over column half `part` (0 or
// 1) of the tile (two warps share each lane quadrant, one per half).
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(uint32_t t_row, int row, bool valid,
                                              int n0, int M, int N, int part,
                                              const TcEpiArgs& ep, EpiPre& pre,
                                              int lane) {
  if constexpr (EPI == TC_STORE || EPI == TC_RESID || EPI == TC_RESID_SS) {
    // unrolled over the part's chunks so that the residual registers of
    // every chunk stay in place (no copies that would wait on the loads)
    constexpr int RW = kResidWords;
    float ss = 0.f;
    const int cb = chunk_begin<BN>(part);
#pragma unroll
    for (int k = 0; k < BN / 64; ++k) {
      const int c = cb + k;
      const int col = n0 + c * 32;
      const bool live = valid && col < N;
      const size_t off = (size_t)row * ep.ldo + col;
      float v[32];
      tmem_ld32(t_row + c * 32, v);
      if (live) {
        if constexpr (EPI == TC_RESID_SS) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 r = unpack_bf16x2(pre.w[k * RW + j]);
            v[2 * j] += r.x;
            v[2 * j + 1] += r.y;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            ss = fmaf(v[j], v[j], ss);
            v[j] *= ep.out_scale;
          }
          store_16x32(ep.out, off, v, ep.out_f16, true);
        } else if constexpr (EPI == TC_RESID) {
          const float sc = ep.in_scale, rsc = ep.res_scale;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 r = unpack_f16x2(pre.w[k * RW + j]);
            v[2 * j] = fmaf(sc, v[2 * j], rsc * r.x);
            v[2 * j + 1] = fmaf(sc, v[2 * j + 1], rsc * r.y);
          }
          store_16x32(ep.out, off, v, false, ep.vec32);
        } else {
          store_16x32(ep.out, off, v, false, ep.vec32);
        }
      }
    }
    if constexpr (EPI == TC_RESID_SS) {
      if (valid) ep.ss_out[(size_t)row * ep.ss_np + (n0 / BN) * 2 + part] = ss;
    }
  } else if constexpr (EPI == TC_QKV) {
    const int d = ep.head_dim, half = d / 2;
    const float rs = valid ? pre.f : 0.f;
#pragma unroll 1
    for (int hb = part * (BN / 2); hb < (part + 1) * (BN / 2); hb += d) {
      const int hc = n0 + hb;
      const bool rope = hc < ep.rope_cols;
#pragma unroll 1
      for (int c = 0; c < half; c += 32) {
        // frequencies 32..63 (head_dim 128: one head block per part, so
        // the prefetched 0..31 are not needed again)
        if (c > 0 && valid) {
          ld_words<32>(ep.cos_t + (size_t)pre.p * half + c, pre.cs, true);
          ld_words<32>(ep.sin_t + (size_t)pre.p * half + c, pre.sn, true);
        }
        float x1[32], x2[32];
        tmem_ld32_nowait(t_row + hb + c, x1);
        tmem_ld32_nowait(t_row + hb + half + c, x2);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          tmem_pin(x1[j]);
          tmem_pin(x2[j]);
        }
        if (valid && hc < N) {
          if (rope) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float a = rs * x1[j], b = rs * x2[j];
              const float cj = __uint_as_float(pre.cs[j]), sj = __uint_as_float(pre.sn[j]);
              x1[j] = a * cj - b * sj;
              x2[j] = b * cj + a * sj;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              x1[j] *= rs;
              x2[j] *= rs;
            }
          }
          const size_t o = (size_t)row * ep.ldo + hc + c;
          store_16x32(ep.out, o, x1, ep.out_f16, true);
          store_16x32(ep.out, o + half, x2, ep.out_f16, true);
        }
      }
    }
  } else if constexpr (EPI == TC_SWIGLU) {
    static_assert(BN == 256, "gate/up interleave is 128 + 128");
    const float r2 = valid ? ep.in_scale * rsqrtf(pre.f * ep.inv_h + ep.eps) : 0.f;
#pragma unroll 1
    for (int c = part * 2; c < part * 2 + 2; ++c) {
      float g[32], u[32];
      tmem_ld32_nowait(t_row + c * 32, g);
      tmem_ld32_nowait(t_row + 128 + c * 32, u);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        tmem_pin(g[j]);
        tmem_pin(u[j]);
      }
      int col = n0 / 2 + c * 32;
      if (valid && n0 < N) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] *= r2;
          u[j] *= r2;
        }
        if (ep.aux_out) {  // gate and up themselves, for the backward pass
          const size_t o = (size_t)row * N + n0 + c * 32;
          store_16x32(ep.aux_out, o, g, true, true);
          store_16x32(ep.aux_out, o + 128, u, true, true);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) g[j] = silu(g[j]) * u[j] * ep.out_scale;
        store_16x32(ep.out, (size_t)row * ep.ldo + col, g, ep.out_f16, true);
      }
    }
  } else if constexpr (EPI == TC_SWIGLU_BWD) {
    // this part's 128 columns of d act are one packed gate|up block
    const float r2 = valid ? rsqrtf(pre.f * ep.inv_h + ep.eps) : 0.f;
    const int i0 = n0 + part * (BN / 2);
    const int pb = (i0 / 128) * 256;  // first packed column of the block
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      float da[32];
      tmem_ld32(t_row + part * (BN / 2) + c * 32, da);
      if (!valid || i0 >= N) continue;
      const size_t o = (size_t)row * 2 * N + pb + c * 32;
      uint32_t gw[16], uw[16];
      ld_words<16>(static_cast<const __half*>(ep.aux_in) + o, gw, true);
      ld_words<16>(static_cast<const __half*>(ep.aux_in) + o + 128, uw, true);
      float dg_[32], du_[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 g2 = unpack_f16x2(gw[j]), u2 = unpack_f16x2(uw[j]);
        const float gg[2] = {g2.x, g2.y}, uu[2] = {u2.x, u2.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float sg = 1.0f / (1.0f + __expf(-gg[e]));
          const float a = da[2 * j + e] * ep.in_scale * r2 * ep.out_scale;
          du_[2 * j + e] = a * gg[e] * sg;                                // silu(g)
          dg_[2 * j + e] = a * uu[e] * sg * (1.0f + gg[e] * (1.0f - sg));  // silu'(g)
        }
      }
      store_16x32(ep.out, o, dg_, true, true);
      store_16x32(ep.out, o + 128, du_, true, true);
    }
  } else if constexpr (EPI == TC_F32_DOT) {
    constexpr int RW = kResidWords;
    float dot = 0.f;
    const int cb = chunk_begin<BN>(part);
#pragma unroll
    for (int k = 0; k < BN / 64; ++k) {
      const int c = cb + k;
      const int col = n0 + c * 32;
      float v[32];
      tmem_ld32(t_row + c * 32, v);
      if (valid && col < N) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 r = ep.res_bf16 ? unpack_bf16x2(pre.w[k * RW + j])
                                       : unpack_f16x2(pre.w[k * RW + j]);
          v[2 * j] *= ep.in_scale;
          v[2 * j + 1] *= ep.in_scale;
          dot = fmaf(v[2 * j], r.x, dot);
          dot = fmaf(v[2 * j + 1], r.y, dot);
        }
        uint32_t u[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(v[j]);
        st_words<32>(static_cast<float*>(ep.out) + (size_t)row * ep.ldo + col, u,
                     ep.vec32 != 0);
      }
    }
    if (valid) ep.ss_out[(size_t)row * ep.ss_np + (n0 / BN) * 2 + part] = dot * ep.res_scale;
  } else if constexpr (EPI == TC_DO) {
    constexpr int RW = kResidWords;
    const int cb = chunk_begin<BN>(part);
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < BN / 64; ++k) {
      const int c = cb + k;
      const int col = n0 + c * 32;
      float v[32];
      tmem_ld32(t_row + c * 32, v);
      if (valid && col < N) {
        uint32_t u[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          u[j] = pack_f16x2(v[2 * j] * ep.in_scale, v[2 * j + 1] * ep.in_scale);
          const float2 d2 = unpack_f16x2(u[j]), o2 = unpack_f16x2(pre.w[k * RW + j]);
          dot = fmaf(d2.x, o2.x, fmaf(d2.y, o2.y, dot));
        }
        st_words<16>(static_cast<__half*>(ep.out) + (size_t)row * ep.ldo + col, u, true);
        if ((col + 32) % ep.head_dim == 0) {  // the head's last chunk
          static_cast<float*>(ep.aux_out)[(size_t)row * (N / ep.head_dim) +
                                          col / ep.head_dim] = dot;
          dot = 0.f;
        }
      }
    }
  } else if constexpr (EPI == TC_DW) {
    const int src = ep.inter > 0 ? gate_up_row(row, ep.inter) : row;
    const int cb = chunk_begin<BN>(part);
#pragma unroll 1
    for (int k = 0; k < BN / 64; ++k) {
      const int col = n0 + (cb + k) * 32;
      float v[32];
      tmem_ld32(t_row + (cb + k) * 32, v);
      if (col >= N) continue;  // the same for every lane of the warp
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= ep.in_scale;
      if (ep.dg) {
        float p[32];
        if (valid) {
          uint32_t w[16];
          ld_words<16>(static_cast<const __nv_bfloat16*>(ep.w_orig) +
                           (size_t)src * ep.ldo + col, w, false);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 w2 = unpack_bf16x2(w[j]);
            p[2 * j] = w2.x * v[2 * j];
            p[2 * j + 1] = w2.y * v[2 * j + 1];
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) p[j] = 0.f;
        }
        warp_column_sums(p, lane);
        ep.dg[(size_t)(row / 32) * N + col + lane] = p[0];  // this warp's 32 rows
      }
      if (valid) {
        if (ep.colscale) {
          uint32_t gsc[16];
          ld_words<16>(static_cast<const __nv_bfloat16*>(ep.colscale) + col, gsc, false);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 g2 = unpack_bf16x2(gsc[j]);
            v[2 * j] *= g2.x;
            v[2 * j + 1] *= g2.y;
          }
        }
        uint32_t u[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(v[j]);
        st_words<32>(static_cast<float*>(ep.out) + (size_t)src * ep.ldo + col, u,
                     ep.vec32 != 0);
      }
    }
  }
}

// Work of one CTA as a sequence of segments (tile, K-blocks [kb0, kb1), slot).
//   tile-stride mode: whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...,
//                     visited in bands of group_m M-tiles (tc_group_m).
//   split phase:      before those, the first sk_tiles tiles (in the same
//                     order) are shared by K-block: the CTA owns units
//                     [c W / G, (c + 1) W / G) of W = sk_tiles * kb_total, at
//                     least one tile's worth, so a tile is cut at most once;
//                     the tile-stride tiles then start at sk_tiles.
//   stream-K mode:    (TC_PARTIAL) the CTA owns the global K-block range
//                     [c W / G, (c + 1) W / G) of W = tiles * kb_total; each
//                     run inside one tile is a segment whose fp32 partial goes
//                     to slot (c - first CTA of that tile).
struct Sched {
  int m_tiles, n_tiles, kb_total, num_tiles, grid, cta, group_m;
  int pair;  // CTA pairs: this CTA's rank (tiles 2 m + pair), else -1
  bool stream_k;
  long long W, g, g_end;
  int next_tile;

  // pr >= 0: the grid runs as CTA pairs (clusters of 2) over pair tiles
  // (M-tiles 2 m and 2 m + 1 of one N-tile); this CTA takes M-tile 2 m + pr.
  __device__ Sched(int M, int N, int K, int bn, bool sk, int sk_tiles, int gm,
                   int pr = -1) {
    group_m = gm;
    pair = pr;
    m_tiles = (M + BM - 1) / BM;
    if (pr >= 0) m_tiles = (m_tiles + 1) / 2;
    n_tiles = (N + bn - 1) / bn;
    kb_total = (K + BK - 1) / BK;
    num_tiles = m_tiles * n_tiles;
    grid = pr >= 0 ? gridDim.x / 2 : gridDim.x;
    cta = pr >= 0 ? blockIdx.x / 2 : blockIdx.x;
    stream_k = sk;
    const int split = sk ? num_tiles : sk_tiles;
    W = (long long)split * kb_total;
    g = (long long)cta * W / grid;
    g_end = (long long)(cta + 1) * W / grid;
    next_tile = sk ? num_tiles : split + cta;
  }

  __device__ bool next(int& mt, int& nt, int& kb0, int& kb1, int& tile,
                       int& slot) {
    if (g < g_end) {
      tile = (int)(g / kb_total);
      kb0 = (int)(g - (long long)tile * kb_total);
      long long left = g_end - g;
      kb1 = (int)(kb0 + left < kb_total ? kb0 + left : kb_total);
      g += kb1 - kb0;
      if (stream_k) {
        long long gs = (long long)tile * kb_total;
        int first = (int)(((gs + 1) * grid - 1) / W);
        slot = cta - first;
        mt = tile / n_tiles;
        nt = tile - mt * n_tiles;
      } else {
        slot = 0;
        tile_coords(tile, m_tiles, n_tiles, group_m, mt, nt);
      }
      return true;
    }
    if (next_tile >= num_tiles) return false;
    tile = next_tile;
    tile_coords(tile, m_tiles, n_tiles, group_m, mt, nt);
    if (pair >= 0) mt = 2 * mt + pair;
    kb0 = 0;
    kb1 = kb_total;
    slot = 0;
    next_tile += grid;
    return true;
  }
};

// Shared-memory image of one operand K-slice (64 K values): K-major, one TMA
// box of R rows x 128 bytes; MN-major (AMN / BMN), R / 64 boxes of 64 K-rows
// x 64 MN values (128 bytes), 8 KB apart.  The matching descriptors: K-major
// steps 32 bytes per K step of 16; MN-major steps 16 rows (2048 bytes) and
// finds the next 64-wide MN block 8 KB away.
template <bool MN, int R>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* m,
                                             uint64_t* bar, int kb, int r0) {
  if constexpr (MN) {
#pragma unroll
    for (int i = 0; i < R / 64; ++i)
      tma_load_2d(dst + i * 8192, m, bar, r0 + 64 * i, kb * BK);
  } else {
    tma_load_2d(dst, m, bar, kb * BK, r0);
  }
}

// B K-slice of a CTA pair: this CTA loads its half (rank r: N rows
// n0 + R/2 r .., or 64-wide MN blocks 2 r, 2 r + 1) and multicasts it into the
// same place of both CTAs' shared memory; the peer does the other half.  The
// K-major map has an R/2-row box.
template <bool MN, int R>
__device__ __forceinline__ void load_b_pair(uint8_t* dst, const CUtensorMap* m,
                                            uint64_t* bar, int kb, int n0, int rank) {
  if constexpr (MN) {
#pragma unroll
    for (int i = 0; i < R / 128; ++i) {
      const int blk = rank * (R / 128) + i;
      tma_load_2d_mc(dst + blk * 8192, m, bar, n0 + 64 * blk, kb * BK, 0x3);
    }
  } else {
    tma_load_2d_mc(dst + rank * (R / 2) * 128, m, bar, kb * BK, n0 + rank * (R / 2), 0x3);
  }
}

// load_operand for a cta_group::2 pair: R rows (K-major) or R / 64 MN blocks
// of this CTA's own operand share, into its own shared memory, completing on
// the mbarrier at shared::cluster address `bar` (rank 0's).
template <bool MN, int R>
__device__ __forceinline__ void load_operand_pair(uint8_t* dst, const CUtensorMap* m,
                                                  uint32_t bar, int kb, int r0) {
  if constexpr (MN) {
#pragma unroll
    for (int i = 0; i < R / 64; ++i)
      tma_load_2d_pair(dst + i * 8192, m, bar, r0 + 64 * i, kb * BK);
  } else {
    tma_load_2d_pair(dst, m, bar, kb * BK, r0);
  }
}

template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr) {
  return MN ? sdesc_mn128(addr, 8192) : sdesc_k128(addr);
}

template <bool MN>
__device__ __forceinline__ uint64_t operand_kstep(int k) {
  return MN ? (uint64_t)(k * (2048 >> 4)) : (uint64_t)(2 * k);
}

// MC: the grid runs as CTA pairs (clusters of 2) on pair tiles sharing
// their B tile, each CTA loading half of every B K-slice and multicasting it
// to both; a stage is free once both CTAs' MMAs are done with it (empty
// barriers count a multicast commit from each).
// CG2 (with MC): the pair runs one M = 256 tcgen05.mma
// (cta_group::2) per K step instead of two M = 128 ones.  Each CTA loads its
// own A rows and its half of the B slice (no multicast), both completing on
// rank 0's full barrier; rank 0's thread issues every MMA and commits each
// stage to both CTAs' empty barriers and each tile to both CTAs' acc_full;
// both CTAs' epilogues release an accumulator on rank 0's acc_empty.  Per
// K step each SM's tensor core reads 16 KB of operands from its shared
// memory instead of 24 KB, and a stage holds 32 KB instead of 48.
template <int BN, int STAGES, int EPI, bool AMN = false, bool BMN = false, bool MC = false,
          bool CG2 = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
                   TcEpiArgs ep) {
  static_assert(!CG2 || (MC && EPI != TC_PARTIAL), "cta_group::2 runs as CTA pairs");
  using L = Layout<BN, STAGES, CG2>;
  constexpr bool kStreamK = EPI == TC_PARTIAL;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // arrivals of the epilogue threads at the split tiles' flags
  int* sk_count = const_cast<int*>(abort_flag) + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MC && !CG2 ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], CG2 ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    sk_count[0] = sk_count[1] = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if constexpr (CG2)
      tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
    else
      tmem_alloc(tmem_slot, L::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the peer's barriers are initialised before anything is multicast to it
  uint32_t rank = 0;
  if constexpr (MC) {
    rank = cluster_ctarank();
    cluster_sync();
  }

  Sched sched(M, N, K, BN, kStreamK, ep.sk_tiles, ep.group_m, MC ? (int)rank : -1);
  int mt, nt, kb0, kb1, tile, slot;

  pdl_trigger();
  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      // The weights (A of the swap-AB stream-K GEMM, B otherwise) never
      // depend on the previous kernel: their first STAGES K-slices are
      // requested before waiting for it.
      constexpr bool kWeightsA = EPI == TC_PARTIAL;
      // cta_group::2: every copy of the pair completes on rank 0's full
      // barrier, which rank 0 arms for both CTAs' bytes
      const bool arm = !CG2 || rank == 0;
      constexpr uint32_t kArmBytes = CG2 ? 2 * L::STAGE : L::STAGE;
      uint32_t pre = 0;
      if (kWeightsA || ep.b_const) {
        Sched s2 = sched;
        int pm, pn, pk0, pk1, pt, ps;
        if (s2.next(pm, pn, pk0, pk1, pt, ps)) {
          for (int kb = pk0; kb < pk1 && pre < (uint32_t)STAGES; ++kb, ++pre) {
            uint8_t* sa = smem + pre * L::STAGE;
            if (arm) mbar_arrive_expect_tx(&full[pre], kArmBytes);
            if (kWeightsA)
              load_operand<AMN, BM>(sa, &tmA, &full[pre], kb, pm * BM);
            else if constexpr (CG2)
              load_operand_pair<BMN, BN / 2>(sa + L::A_BYTES, &tmB, mapa_rank(&full[pre], 0),
                                             kb, pn * BN + (int)rank * (BN / 2));
            else if constexpr (MC)
              load_b_pair<BMN, BN>(sa + L::A_BYTES, &tmB, &full[pre], kb, pn * BN, rank);
            else
              load_operand<BMN, BN>(sa + L::A_BYTES, &tmB, &full[pre], kb, pn * BN);
          }
        }
      }
      pdl_wait();
      while (ok && sched.next(mt, nt, kb0, kb1, tile, slot)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, ep.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * L::STAGE;
          if constexpr (CG2) {
            const uint32_t fb = mapa_rank(&full[stage], 0);
            if (issued >= pre && arm) mbar_arrive_expect_tx(&full[stage], kArmBytes);
            load_operand_pair<AMN, BM>(sa, &tmA, fb, kb, mt * BM);
            if (issued >= pre)
              load_operand_pair<BMN, BN / 2>(sa + L::A_BYTES, &tmB, fb, kb,
                                             nt * BN + (int)rank * (BN / 2));
          } else if (issued < pre) {  // weights already requested, tx already armed
            if (kWeightsA)
              load_operand<BMN, BN>(sa + L::A_BYTES, &tmB, &full[stage], kb, nt * BN);
            else
              load_operand<AMN, BM>(sa, &tmA, &full[stage], kb, mt * BM);
          } else {
            mbar_arrive_expect_tx(&full[stage], L::STAGE);
            load_operand<AMN, BM>(sa, &tmA, &full[stage], kb, mt * BM);
            if constexpr (MC)
              load_b_pair<BMN, BN>(sa + L::A_BYTES, &tmB, &full[stage], kb, nt * BN, rank);
            else
              load_operand<BMN, BN>(sa + L::A_BYTES, &tmB, &full[stage], kb, nt * BN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && CG2 && rank != 0) {
        // this CTA's copies complete on rank 0's barriers, which rank 0's
        // producer drains before the pair's closing cluster barrier
      } else if (!ok) {  // let the copies already issued land before leaving
        volatile int own = 0;
        if (issued < pre) issued = pre;  // prefetched stages are in flight too
        uint32_t n = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
        for (uint32_t j = 1; j <= n; ++j) {
          uint32_t idx = issued - j;
          mbar_wait(&full[idx % STAGES], (idx / STAGES) & 1, ep.status, &own);
        }
      } else if constexpr (MC) {
        // the peer's MMA commits to this CTA's empty barriers (its last ones
        // included) have landed before this CTA may leave
        uint32_t n = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
        for (uint32_t j = 1; j <= n; ++j) {
          uint32_t idx = issued - j;
          mbar_wait(&empty[idx % STAGES], (idx / STAGES) & 1, ep.status, abort_flag);
        }
      }
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0 && (!CG2 || rank == 0)) {
      constexpr int kMmaM = CG2 ? 2 * BM : BM;
      const uint32_t idesc = (ep.ab_f16 ? idesc_f16(kMmaM, BN) : idesc_bf16(kMmaM, BN)) |
                             (AMN ? 1u << 15 : 0u) | (BMN ? 1u << 16 : 0u);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t local = 0;
      bool ok = true;
      bool issued_any = false;
      while (ok && sched.next(mt, nt, kb0, kb1, tile, slot)) {
        const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
        ++local;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, ep.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, ep.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * L::STAGE);
          const uint64_t ad = operand_desc<AMN>(sa),
                         bd = operand_desc<BMN>(sa + L::A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            if constexpr (CG2)
              tc_mma_pair_nc(d_tmem, ad + operand_kstep<AMN>(k), bd + operand_kstep<BMN>(k),
                             idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            else
              tc_mma_bf16_nc(d_tmem, ad + operand_kstep<AMN>(k), bd + operand_kstep<BMN>(k),
                             idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          issued_any = true;
          if constexpr (CG2)
            tc_commit_pair(&empty[stage], 0x3);  // the stage is free in both CTAs
          else if constexpr (MC)
            tc_commit_mc(&empty[stage], 0x3);  // both CTAs read this stage's B
          else
            tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) {
          if constexpr (CG2)
            tc_commit_pair(&acc_full[acc], 0x3);  // both CTAs' halves of the tile
          else
            tc_commit(&acc_full[acc]);
        }
      }
      if (!ok && issued_any) {  // wait for the MMAs in flight
        volatile int own = 0;
        if constexpr (CG2)
          tc_commit_pair(drain, 0x1);
        else
          tc_commit(drain);
        mbar_wait(drain, 0, ep.status, &own);
      }
    }
  } else {
    pdl_wait();
    const int quad = warp & 3;            // TMEM lane quadrant of this warp
    const int part = (warp - 2) / 4;      // column half of the tile
    uint32_t local = 0;
    while (sched.next(mt, nt, kb0, kb1, tile, slot)) {
      const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
      ++local;
      const int r = quad * 32 + lane;
      EpiPre pre;
      if constexpr (EPI != TC_PARTIAL)
        epilogue_prefetch<BN, EPI>(pre, mt * BM + r, mt * BM + r < M, nt * BN, N, part, ep);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&acc_full[acc], acc_phase, ep.status, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
      if constexpr (EPI == TC_PARTIAL) {
        // token-major slot: column c of the tile is 128 consecutive floats,
        // so a warp's 32 rows of one column are one 128-byte store
        float* o = static_cast<float*>(ep.out) +
                   ((size_t)tile * ep.part_slots + slot) * BN * BM + r;
#pragma unroll 1
        for (int c = part * (BN / 64); c < (part + 1) * (BN / 64); ++c) {
          float v[32];
          tmem_ld32(t_row + c * 32, v);
#pragma unroll
          for (int q = 0; q < 32; ++q) o[(size_t)(c * 32 + q) * BM] = v[q];
        }
      } else if (kb0 > 0) {
        // the later K-blocks of a split tile, computed first: hand the fp32
        // sums to the CTA that finishes the tile (blockIdx.x - 1)
        float* dst = ep.sk_part + ((size_t)blockIdx.x * BM + r) * BN;
#pragma unroll 1
        for (int c = part * (BN / 64); c < (part + 1) * (BN / 64); ++c) {
          float v[32];
          tmem_ld32(t_row + c * 32, v);
          uint32_t u[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(v[j]);
          st_words<32>(dst + c * 32, u, true);
        }
        __threadfence();
        if (atomicAdd(&sk_count[0], 1) == kEpiWarps * 32 - 1)
          st_release_gpu(ep.sk_flag + blockIdx.x, ep.sk_epoch);
      } else {
        const int row = mt * BM + r;
        const bool split = kb1 < sched.kb_total;  // the rest comes from CTA + 1
        if (split && flag_wait(ep.sk_flag + blockIdx.x + 1, ep.sk_epoch, ep.status,
                               abort_flag))
          add_partial_tmem<BN, EPI>(t_row, ep.sk_part + ((size_t)(blockIdx.x + 1) * BM + r) * BN,
                               part);
        epilogue_tile<BN, EPI>(t_row, row, row < M, nt * BN, M, N, part, ep, pre, lane);
        // every thread has read its rows: clear the flag for the next launch
        if (split && atomicAdd(&sk_count[1], 1) == kEpiWarps * 32 - 1)
          ep.sk_flag[blockIdx.x + 1] = 0;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG2)
          mbar_arrive_cluster(mapa_rank(&acc_empty[acc], 0));  // rank 0 issues
        else
          mbar_arrive(&acc_empty[acc]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG2) {
    // both CTAs are done with the pair's tensor memory (and with each
    // other's barriers) before the pair frees it
    cluster_sync();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
    return;
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
  // neither CTA of a pair leaves while the other may still write to it
  if constexpr (MC) cluster_sync();
}

template <int BN, int STAGES, int EPI, bool AMN = false, bool BMN = false, bool MC = false,
          bool CG2 = false>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N,
                   int K, const TcEpiArgs& ep, int grid, cudaStream_t s) {
  using L = Layout<BN, STAGES, CG2>;
  auto kern = gemm_tc_kernel<BN, STAGES, EPI, AMN, BMN, MC, CG2>;
  static std::atomic<uint64_t> attr_done{0};
  if (cudaError_t e = ensure_smem_attr(kern, (int)L::TOTAL, attr_done); e != cudaSuccess)
    return e;
  if (grid <= 0) return cudaSuccess;
  TcEpiArgs e = ep;
  const uintptr_t al = reinterpret_cast<uintptr_t>(e.out) |
                       reinterpret_cast<uintptr_t>(e.residual) |
                       reinterpret_cast<uintptr_t>(e.aux_in) |
                       reinterpret_cast<uintptr_t>(e.aux_out);
  e.vec32 = (al & 31) == 0 && e.ldo % 16 == 0;
  if (!e.status) {
    cudaError_t err = cudaGetSymbolAddress((void**)&e.status, g_tc_status);
    if (err != cudaSuccess) return err;
  }
  if constexpr (MC) {
    // pairs: grid = 2 x (pairs that can be resident at once, at most the
    // pair tiles)
    static int max_pairs[64] = {};
    int dev = 0;
    if (cudaError_t err = cudaGetDevice(&dev); err != cudaSuccess) return err;
    int pairs = dev < 64 ? max_pairs[dev] : 0;
    if (pairs <= 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(kGemmThreads);
      cfg.dynamicSmemBytes = L::TOTAL;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaError_t err = cudaOccupancyMaxActiveClusters(&pairs, kern, &cfg);
          err != cudaSuccess)
        return err;
      if (pairs <= 0) return cudaErrorInvalidConfiguration;
      if (dev < 64) max_pairs[dev] = pairs;
    }
    const int pair_tiles = grid;  // tc_gemm passes the pair tiles
    const int n = pair_tiles < pairs ? pair_tiles : pairs;
    return launch_cluster2(kern, dim3(2 * n), dim3(kGemmThreads), L::TOTAL, s, e.pdl != 0,
                           ta, tb, M, N, K, e);
  }
  // the split phase's CTAs wait on flags other CTAs set: make them co-resident
  if (e.sk_tiles > 0)
    return launch_coop(kern, dim3(grid), dim3(kGemmThreads), L::TOTAL, s, e.pdl != 0, ta,
                       tb, M, N, K, e);
  if (e.pdl) return launch_pdl(kern, dim3(grid), dim3(kGemmThreads), L::TOTAL, s, ta, tb, M, N, K, e);
  kern<<<grid, kGemmThreads, L::TOTAL, s>>>(ta, tb, M, N, K, e);
  return cudaGetLastError();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

cudaError_t tc_take_status(int* word) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_tc_status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
  return e;
}

bool tc_encode_bf16(CUtensorMap* map, const void* ptr, uint64_t rows,
                    uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

TcStreamK tc_streamk_plan(int M, int N, int K, int bn, int grid_limit) {
  TcStreamK p;
  p.tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  p.kb_total = (K + BK - 1) / BK;
  long long W = (long long)p.tiles * p.kb_total;
  p.grid = (int)(W < grid_limit ? W : grid_limit);
  p.slots = 0;
  for (int t = 0; t < p.tiles; ++t) {
    int n = tc_streamk_segments(p, t);
    if (n > p.slots) p.slots = n;
  }
  return p;
}

int tc_group_m(int M, int N, int K) {
  // M-tiles per band: the band's A rows (group_m x 128 rows x K) are read
  // from DRAM once and should stay in L2 while the band's B columns stream
  // past them; up to 48 MB of A (of the 126 MB L2) per band, in powers of
  // two between 16 and 64.  Measured on one B300 (gate_up, 100 steps each):
  // 1B (K = 2048) 64 M-tiles 4.7 % faster than 16; 8B and the varlen pack
  // (K = 4096) 32 M-tiles 2-2.5 % faster than 16, 64 slower; down_proj
  // (K = 14336) 16 and 32 alike, 8 about 1 % slower.
  (void)N;
  const double a_tile = 128.0 * K * 2;
  int g = 16;
  while (g < 64 && 2 * g * a_tile <= 48.0 * (1 << 20)) g *= 2;
  const int m_tiles = (M + BM - 1) / BM;
  return g < m_tiles ? g : (m_tiles > 0 ? m_tiles : 1);
}

int tc_split_tiles(int tiles, int grid, int kb_total) {
  // a split costs a 128 KB store and reload per cut tile and one more
  // epilogue pass: worth it only behind a long main loop
  if (kb_total < 64) return 0;
  if (grid <= 0 || tiles <= grid || tiles % grid == 0) return 0;
  const int rounds = (tiles + grid - 1) / grid;
  const double idle = rounds - (double)tiles / grid;  // in rounds
  if (idle <= 0.03 * rounds) return 0;
  return grid + tiles % grid;
}

cudaError_t tc_gemm(int epi, int bn, const CUtensorMap& ta,
                    const CUtensorMap& tb, int M, int N, int K,
                    const TcEpiArgs& ep, int grid_limit, cudaStream_t s) {
  int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  int grid = tiles < grid_limit ? tiles : grid_limit;
  TcEpiArgs e = ep;
  e.sk_tiles = 0;
  e.group_m = tc_group_m(M, N, K);
  if (ep.pair && epi != TC_PARTIAL) {
    // CTA pairs over pair tiles (two M-tiles of one N-tile), bands of
    // group_m M-tiles = group_m / 2 pair rows
    e.group_m = e.group_m / 2 > 0 ? e.group_m / 2 : 1;
    const int pair_tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + bn - 1) / bn);
    if (ep.pair == 2) {  // one M = 256 MMA over the pair (K-major operands)
      switch (epi) {
        case TC_QKV:
          return launch<256, 6, TC_QKV, false, false, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
        case TC_RESID_SS:
          return launch<256, 6, TC_RESID_SS, false, false, true, true>(ta, tb, M, N, K, e,
                                                                      pair_tiles, s);
        case TC_SWIGLU:
          return launch<256, 6, TC_SWIGLU, false, false, true, true>(ta, tb, M, N, K, e,
                                                                    pair_tiles, s);
        case TC_RESID:
          return launch<256, 6, TC_RESID, false, false, true, true>(ta, tb, M, N, K, e,
                                                                   pair_tiles, s);
        case TC_DW:
          return launch<256, 6, TC_DW, true, true, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
        case TC_SWIGLU_BWD:
          return launch<256, 6, TC_SWIGLU_BWD, false, true, true, true>(ta, tb, M, N, K, e,
                                                                       pair_tiles, s);
        case TC_F32_DOT:
          return launch<256, 6, TC_F32_DOT, false, true, true, true>(ta, tb, M, N, K, e,
                                                                    pair_tiles, s);
        case TC_DO:
          return launch<256, 6, TC_DO, false, true, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
        default: return cudaErrorInvalidValue;
      }
    }
    switch (epi) {
      case TC_QKV: return launch<256, 4, TC_QKV, false, false, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_RESID_SS:
        return launch<256, 4, TC_RESID_SS, false, false, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_SWIGLU:
        return launch<256, 4, TC_SWIGLU, false, false, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_RESID:
        return launch<256, 4, TC_RESID, false, false, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_DW: return launch<256, 4, TC_DW, true, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_SWIGLU_BWD:
        return launch<256, 4, TC_SWIGLU_BWD, false, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_F32_DOT:
        return launch<256, 4, TC_F32_DOT, false, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
      case TC_DO: return launch<256, 4, TC_DO, false, true, true>(ta, tb, M, N, K, e, pair_tiles, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (epi <= TC_RESID && ep.sk_part && ep.sk_flag && ep.sk_epoch != 0)
    e.sk_tiles = tc_split_tiles(tiles, grid, (K + BK - 1) / BK);
  switch (epi) {
    case TC_STORE: return launch<256, 4, TC_STORE>(ta, tb, M, N, K, e, grid, s);
    case TC_QKV: return launch<256, 4, TC_QKV>(ta, tb, M, N, K, e, grid, s);
    case TC_RESID_SS: return launch<256, 4, TC_RESID_SS>(ta, tb, M, N, K, e, grid, s);
    case TC_SWIGLU: return launch<256, 4, TC_SWIGLU>(ta, tb, M, N, K, e, grid, s);
    case TC_RESID: return launch<256, 4, TC_RESID>(ta, tb, M, N, K, e, grid, s);
    case TC_DW: return launch<256, 4, TC_DW, true, true>(ta, tb, M, N, K, e, grid, s);
    case TC_SWIGLU_BWD:
      return launch<256, 4, TC_SWIGLU_BWD, false, true>(ta, tb, M, N, K, e, grid, s);
    case TC_F32_DOT:
      return launch<256, 4, TC_F32_DOT, false, true>(ta, tb, M, N, K, e, grid, s);
    case TC_DO: return launch<256, 4, TC_DO, false, true>(ta, tb, M, N, K, e, grid, s);
    case TC_PARTIAL: {
      TcStreamK p = tc_streamk_plan(M, N, K, bn, grid_limit);
      if (p.slots != ep.part_slots) return cudaErrorInvalidValue;
      if (bn == 64) return launch<64, 8, TC_PARTIAL>(ta, tb, M, N, K, ep, p.grid, s);
      if (bn == 128) return launch<128, 6, TC_PARTIAL>(ta, tb, M, N, K, ep, p.grid, s);
      if (bn == 256) return launch<256, 4, TC_PARTIAL>(ta, tb, M, N, K, ep, p.grid, s);
      return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace llama
