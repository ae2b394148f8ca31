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
// Tiles are visited in bands of 16 M-tiles so that a wave of CTAs shares A
// and B slices in L2.  Every wait is bounded (see mbar_wait).
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "gemm_tc.cuh"

namespace llama {
namespace {

constexpr int BM = 128, BK = 64, GROUP_M = 16;
// warp 0 producer, warp 1 MMA, warps 2..9 epilogue (two per TMEM lane
// quadrant, each on half of the tile's columns)
constexpr int kEpiWarps = 8, kGemmThreads = 64 + 32 * kEpiWarps;

// Status word for GEMMs launched without a layer (llama_gemm_bf16).
__device__ int g_tc_status;

template <int BN, int STAGES>
struct Layout {
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t BAR_OFF = STAGES * STAGE;
  static constexpr uint32_t TOTAL = BAR_OFF + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles,
                                            int& m, int& n) {
  int group = GROUP_M * n_tiles;
  int g = t / group;
  int first_m = g * GROUP_M;
  int gm = min(m_tiles - first_m, GROUP_M);
  int w = t - g * group;
  m = first_m + w % gm;
  n = w / gm;
}

__device__ __forceinline__ void load_bf16x32(const void* p, float* v) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u = q[i];
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y),
           c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    v[8 * i + 0] = a.x; v[8 * i + 1] = a.y; v[8 * i + 2] = b.x;
    v[8 * i + 3] = b.y; v[8 * i + 4] = c.x; v[8 * i + 5] = c.y;
    v[8 * i + 6] = d.x; v[8 * i + 7] = d.y;
  }
}

__device__ __forceinline__ void store_bf16x32(void* p, const float* v) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    q[i] = u;
  }
}

__device__ __forceinline__ void store_f16x32(void* p, const float* v) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_f16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_f16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_f16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_f16x2(v[8 * i + 6], v[8 * i + 7]);
    q[i] = u;
  }
}

// bf16 or fp16 (16-bit elements) at element offset `off` of p.
__device__ __forceinline__ void store_16x32(void* p, size_t off, const float* v,
                                            bool f16) {
  if (f16)
    store_f16x32(static_cast<__half*>(p) + off, v);
  else
    store_bf16x32(static_cast<__nv_bfloat16*>(p) + off, v);
}

__device__ __forceinline__ void store_f32x32(float* p, const float* v) {
  float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

// Epilogue of one accumulator row (TMEM lane) over column half `part` (0 or
// 1) of the tile (two warps share each lane quadrant, one per half).
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(uint32_t t_row, int row, bool valid,
                                              int n0, int M, int N, int part,
                                              const TcEpiArgs& ep) {
  if constexpr (EPI == TC_STORE || EPI == TC_RESID || EPI == TC_RESID_SS) {
    float ss = 0.f;
#pragma unroll 1
    for (int c = part * (BN / 64); c < (part + 1) * (BN / 64); ++c) {
      float v[32];
      tmem_ld32(t_row + c * 32, v);
      int col = n0 + c * 32;
      if (valid && col < N) {
        size_t off = (size_t)row * ep.ldo + col;
        if constexpr (EPI == TC_RESID_SS) {
          float r[32];
          load_bf16x32(static_cast<const __nv_bfloat16*>(ep.residual) + off, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] += r[j];
            ss = fmaf(v[j], v[j], ss);
          }
          store_f32x32(static_cast<float*>(ep.out) + off, v);
          load_bf16x32(static_cast<const __nv_bfloat16*>(ep.colscale) + col, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] *= v[j] * ep.out_scale;
          store_16x32(ep.out2, off, r, ep.out_f16);
        } else {
          if constexpr (EPI == TC_RESID) {
            const float4* r4 =
                reinterpret_cast<const float4*>(static_cast<const float*>(ep.residual) + off);
            const float sc = ep.in_scale;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 rr = r4[q];
              v[4 * q] = fmaf(sc, v[4 * q], rr.x);
              v[4 * q + 1] = fmaf(sc, v[4 * q + 1], rr.y);
              v[4 * q + 2] = fmaf(sc, v[4 * q + 2], rr.z);
              v[4 * q + 3] = fmaf(sc, v[4 * q + 3], rr.w);
            }
          }
          store_bf16x32(static_cast<__nv_bfloat16*>(ep.out) + off, v);
        }
      }
    }
    if constexpr (EPI == TC_RESID_SS) {
      if (valid) atomicAdd(ep.ss_out + row, ss);
    }
  } else if constexpr (EPI == TC_QKV) {
    const int d = ep.head_dim, half = d / 2;
    float rs = 0.f;
    int p = 0;
    if (valid) {
      rs = ep.rowscale[row];
      p = ep.pos[row];
      if (p < 0 || p >= ep.max_pos) {
        set_status(ep.status, ST_BAD_POSITION);
        p = 0;
      }
    }
    const float* cs = ep.cos_t + (size_t)p * half;
    const float* sn = ep.sin_t + (size_t)p * half;
#pragma unroll 1
    for (int hb = part * (BN / 2); hb < (part + 1) * (BN / 2); hb += d) {
      const int hc = n0 + hb;
      const bool rope = hc < ep.rope_cols;
#pragma unroll 1
      for (int c = 0; c < half; c += 32) {
        float x1[32], x2[32];
        tmem_ld32(t_row + hb + c, x1);
        tmem_ld32(t_row + hb + half + c, x2);
        if (valid && hc < N) {
          if (rope) {
            const float4* c4 = reinterpret_cast<const float4*>(cs + c);
            const float4* s4 = reinterpret_cast<const float4*>(sn + c);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 cc = c4[q], ss = s4[q];
              float cv[4] = {cc.x, cc.y, cc.z, cc.w};
              float sv[4] = {ss.x, ss.y, ss.z, ss.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                int j = 4 * q + e;
                float a = rs * x1[j], b = rs * x2[j];
                x1[j] = a * cv[e] - b * sv[e];
                x2[j] = b * cv[e] + a * sv[e];
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              x1[j] *= rs;
              x2[j] *= rs;
            }
          }
          const size_t o = (size_t)row * ep.ldo + hc + c;
          store_16x32(ep.out, o, x1, ep.out_f16);
          store_16x32(ep.out, o + half, x2, ep.out_f16);
        }
      }
    }
  } else if constexpr (EPI == TC_SWIGLU) {
    static_assert(BN == 256, "gate/up interleave is 128 + 128");
    const float r2 =
        valid ? ep.in_scale * rsqrtf(ep.ss_in[row] * ep.inv_h + ep.eps) : 0.f;
#pragma unroll 1
    for (int c = part * 2; c < part * 2 + 2; ++c) {
      float g[32], u[32];
      tmem_ld32(t_row + c * 32, g);
      tmem_ld32(t_row + 128 + c * 32, u);
      int col = n0 / 2 + c * 32;
      if (valid && n0 < N) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          g[j] = silu(r2 * g[j]) * (r2 * u[j]) * ep.out_scale;
        store_16x32(ep.out, (size_t)row * ep.ldo + col, g, ep.out_f16);
      }
    }
  }
}

// Work of one CTA as a sequence of segments (tile, K-blocks [kb0, kb1), slot).
//   tile-stride mode: whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...,
//                     visited in bands of GROUP_M M-tiles.
//   stream-K mode:    the CTA owns the global K-block range
//                     [c W / G, (c + 1) W / G) of W = tiles * kb_total; each
//                     run inside one tile is a segment whose fp32 partial goes
//                     to slot (c - first CTA of that tile).
struct Sched {
  int m_tiles, n_tiles, kb_total, num_tiles, grid, cta;
  bool stream_k;
  long long W, g, g_end;
  int next_tile;

  __device__ Sched(int M, int N, int K, int bn, bool sk) {
    m_tiles = (M + BM - 1) / BM;
    n_tiles = (N + bn - 1) / bn;
    kb_total = (K + BK - 1) / BK;
    num_tiles = m_tiles * n_tiles;
    grid = gridDim.x;
    cta = blockIdx.x;
    stream_k = sk;
    W = (long long)num_tiles * kb_total;
    g = (long long)cta * W / grid;
    g_end = (long long)(cta + 1) * W / grid;
    next_tile = cta;
  }

  __device__ bool next(int& mt, int& nt, int& kb0, int& kb1, int& tile,
                       int& slot) {
    if (!stream_k) {
      if (next_tile >= num_tiles) return false;
      tile = next_tile;
      tile_coords(tile, m_tiles, n_tiles, mt, nt);
      kb0 = 0;
      kb1 = kb_total;
      slot = 0;
      next_tile += grid;
      return true;
    }
    if (g >= g_end) return false;
    tile = (int)(g / kb_total);
    kb0 = (int)(g - (long long)tile * kb_total);
    long long left = g_end - g;
    kb1 = (int)(kb0 + left < kb_total ? kb0 + left : kb_total);
    long long gs = (long long)tile * kb_total;
    int first = (int)(((gs + 1) * grid - 1) / W);
    slot = cta - first;
    mt = tile / n_tiles;
    nt = tile - mt * n_tiles;
    g += kb1 - kb0;
    return true;
  }
};

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
                   TcEpiArgs ep) {
  using L = Layout<BN, STAGES>;
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

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  Sched sched(M, N, K, BN, kStreamK);
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
      uint32_t pre = 0;
      {
        Sched s2 = sched;
        int pm, pn, pk0, pk1, pt, ps;
        if (s2.next(pm, pn, pk0, pk1, pt, ps)) {
          for (int kb = pk0; kb < pk1 && pre < (uint32_t)STAGES; ++kb, ++pre) {
            uint8_t* sa = smem + pre * L::STAGE;
            mbar_arrive_expect_tx(&full[pre], L::STAGE);
            if (kWeightsA)
              tma_load_2d(sa, &tmA, &full[pre], kb * BK, pm * BM);
            else
              tma_load_2d(sa + L::A_BYTES, &tmB, &full[pre], kb * BK, pn * BN);
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
          if (issued < pre) {  // weights already requested, tx already armed
            if (kWeightsA)
              tma_load_2d(sa + L::A_BYTES, &tmB, &full[stage], kb * BK, nt * BN);
            else
              tma_load_2d(sa, &tmA, &full[stage], kb * BK, mt * BM);
          } else {
            mbar_arrive_expect_tx(&full[stage], L::STAGE);
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, mt * BM);
            tma_load_2d(sa + L::A_BYTES, &tmB, &full[stage], kb * BK, nt * BN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {  // let the copies already issued land before leaving
        volatile int own = 0;
        if (issued < pre) issued = pre;  // prefetched stages are in flight too
        uint32_t n = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
        for (uint32_t j = 1; j <= n; ++j) {
          uint32_t idx = issued - j;
          mbar_wait(&full[idx % STAGES], (idx / STAGES) & 1, ep.status, &own);
        }
      }
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      const uint32_t idesc = ep.ab_f16 ? idesc_f16(BM, BN) : idesc_bf16(BM, BN);
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
          const uint64_t ad = sdesc_k128(sa), bd = sdesc_k128(sa + L::A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {  // a K step of 16 is 32 bytes
            tc_mma_bf16_nc(d_tmem, ad + 2 * k, bd + 2 * k, idesc,
                           (kb > kb0 || k > 0) ? 1u : 0u);
          }
          issued_any = true;
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(&acc_full[acc]);
      }
      if (!ok && issued_any) {  // wait for the MMAs in flight
        volatile int own = 0;
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
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&acc_full[acc], acc_phase, ep.status, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const int r = quad * 32 + lane;
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
      } else {
        const int row = mt * BM + r;
        epilogue_tile<BN, EPI>(t_row, row, row < M, nt * BN, M, N, part, ep);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

template <int BN, int STAGES, int EPI>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N,
                   int K, const TcEpiArgs& ep, int grid, cudaStream_t s) {
  using L = Layout<BN, STAGES>;
  auto kern = gemm_tc_kernel<BN, STAGES, EPI>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (grid <= 0) return cudaSuccess;
  TcEpiArgs e = ep;
  if (!e.status) {
    cudaError_t err = cudaGetSymbolAddress((void**)&e.status, g_tc_status);
    if (err != cudaSuccess) return err;
  }
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

cudaError_t tc_gemm(int epi, int bn, const CUtensorMap& ta,
                    const CUtensorMap& tb, int M, int N, int K,
                    const TcEpiArgs& ep, int grid_limit, cudaStream_t s) {
  int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  int grid = tiles < grid_limit ? tiles : grid_limit;
  switch (epi) {
    case TC_STORE: return launch<256, 4, TC_STORE>(ta, tb, M, N, K, ep, grid, s);
    case TC_QKV: return launch<256, 4, TC_QKV>(ta, tb, M, N, K, ep, grid, s);
    case TC_RESID_SS: return launch<256, 4, TC_RESID_SS>(ta, tb, M, N, K, ep, grid, s);
    case TC_SWIGLU: return launch<256, 4, TC_SWIGLU>(ta, tb, M, N, K, ep, grid, s);
    case TC_RESID: return launch<256, 4, TC_RESID>(ta, tb, M, N, K, ep, grid, s);
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
