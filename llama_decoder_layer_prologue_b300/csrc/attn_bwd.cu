// Backward pass of the causal grouped-query attention of the prefill
// ("模型层" 9.3 CausalSelfAttention; "parallel_attention.py" 2 and 3: the
// forward o = softmax(q k^T / sqrt(d) + causal mask) v per sequence, query
// head h reading kv head h / n_rep), differentiated by the chain rule:
//   P = softmax(z), z = q k^T / sqrt(d), dP = dO v^T,
//   dz = P * (dP - D) with D = rowsum(dO * O) (the softmax Jacobian),
//   dq = dz k / sqrt(d), dk = dz^T q / sqrt(d), dv = P^T dO,
// a kv head's dk and dv summed over its n_rep query heads (repeat_kv^T), and
// dq, dk rotated back by RoPE^T (y = a cos + rotate_half(a) sin has
// a-gradient dy cos + [ (dy sin)_2, -(dy sin)_1 ]).  P is recomputed from
// the forward's log2 softmax denominators, so nothing of size tokens^2 is
// stored.  q, k, v, dO, P and dz are fp16 on the tensor cores (fp32
// accumulation in tensor memory).
//
// Two tcgen05 kernels, each persistent (one CTA per SM), 10 warps:
//   warps 0..7  compute: thread r of warp w owns TMEM lane r (32 (w % 4) + lane)
//               and 32 of each half tile's 64 columns (warps 0..3 the first,
//               4..7 the second): softmax recomputation and dz, then half of
//               the accumulator's read-out with RoPE^T;
//   warp 8      TMA producer;
//   warp 9      allocates tensor memory; one elected lane issues tcgen05.mma.
// A 128 x 128 tile is handled as two halves of 64 columns: the compute warps
// work through half 0 and then half 1, and the tensor core runs the products
// of one half while they work on the other.
// attn_bwd_dq_kernel: a work item is one query tile (the forward's
//   GQA-packed 128 rows: hpc heads x 128 / hpc positions); per key tile j of
//   its causal range S = Q K_j^T and dP = dO V_j^T go to TMEM, the compute
//   warps turn them into dz (fp16, into TMEM), and dQ += dz K_j reads dz from
//   TMEM as the A operand and K_j as an MN-major B operand.
// attn_bwd_dkv_kernel: a work item is one key tile (128 keys of one kv
//   head); per query tile i of every query head of the group that sees it,
//   S^T = K Q_i^T and dP^T = V dO_i^T go to TMEM, the compute warps form P^T
//   and dz^T (fp16, over the S^T / dP^T columns they read), and
//   dV += P^T dO_i, dK += dz^T Q_i accumulate the whole group in TMEM (no
//   atomics, no repeat_kv).
// Both kernels take their items dynamically, longest range first (a global
// counter; the producer thread hands each to the MMA and compute warps
// through a shared-memory ring).  Every wait is bounded (2 s -> status bit,
// abort, drain, free TMEM).
#include <cuda_fp16.h>
#include <math.h>

#include "attn_bwd.cuh"
#include "common.cuh"
#include "gemm_tc.cuh"

namespace llama {
namespace {

constexpr int AM = 128;  // rows of a query tile (and keys of a key tile)
// warps 0..7 compute (warps w and w + 4 share TMEM lanes 32 (w % 4) ..);
// warp 8 TMA producer; warp 9 MMA issuer
constexpr int kThreads = 320;
constexpr int kCompute = 256;
constexpr int kProducerWarp = 8, kMmaWarp = 9;

// Bounded wait of this file's pipelines: the form that lets the hardware
// suspend a waiting warp (a spinning form measured the same here and takes
// issue slots from the compute warps).
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, int* status,
                                      volatile int* abort_flag) {
  return mbar_wait_sleep(bar, parity, status, abort_flag);
}

int heads_per_tile(int n_rep) {
  int h = 8;
  while (h > 1 && n_rep % h != 0) h >>= 1;
  return h;
}

// Start and length of sequence s (length 0 for a bad cu_seqlens entry, which
// the forward's positions kernel has already flagged).
__device__ __forceinline__ void seq_range(const AttnBwdArgs& a, int s, int& a0, int& L) {
  if (a.cu) {
    const int s0 = a.cu[s], s1 = a.cu[s + 1];
    if (s0 < 0 || s1 < s0 || s1 > a.tokens) {
      a0 = 0;
      L = 0;
    } else {
      a0 = s0;
      L = s1 - s0;
    }
  } else {
    a0 = s * a.seq_len;
    L = a.seq_len;
  }
}

// RoPE^T of 2 x 32 values (dimensions c .. c+31 and half + c .. half + c + 31
// of one head) at table row p, scaled by `sc`, stored as fp16 at dst[c] and
// dst[half + c].
__device__ __forceinline__ void rope_back_store(const AttnBwdArgs& a, int p, int c,
                                                int half, float sc, float* x1,
                                                float* x2, __half* dst) {
  const float* cs = a.cos_t + (size_t)p * half + c;
  const float* sn = a.sin_t + (size_t)p * half + c;
  uint32_t w1[16], w2[16];
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float y1[2], y2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float cj = __ldg(cs + j + e), sj = __ldg(sn + j + e);
      const float d1 = sc * x1[j + e], d2 = sc * x2[j + e];
      y1[e] = d1 * cj + d2 * sj;
      y2[e] = d2 * cj - d1 * sj;
    }
    w1[j / 2] = pack_f16x2(y1[0], y1[1]);
    w2[j / 2] = pack_f16x2(y2[0], y2[1]);
  }
  uint4* o1 = reinterpret_cast<uint4*>(dst + c);
  uint4* o2 = reinterpret_cast<uint4*>(dst + half + c);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    o1[q] = make_uint4(w1[4 * q], w1[4 * q + 1], w1[4 * q + 2], w1[4 * q + 3]);
    o2[q] = make_uint4(w2[4 * q], w2[4 * q + 1], w2[4 * q + 2], w2[4 * q + 3]);
  }
}

// 32 values as fp16 at dst.
__device__ __forceinline__ void store_f16x32(__half* dst, const float* v, float sc) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    o[q] = make_uint4(pack_f16x2(sc * v[8 * q], sc * v[8 * q + 1]),
                      pack_f16x2(sc * v[8 * q + 2], sc * v[8 * q + 3]),
                      pack_f16x2(sc * v[8 * q + 4], sc * v[8 * q + 5]),
                      pack_f16x2(sc * v[8 * q + 6], sc * v[8 * q + 7]));
}

__device__ __forceinline__ int table_row(const AttnBwdArgs& a, int t) {
  const int p = a.pos[t];
  return (p < 0 || p >= a.max_pos) ? 0 : p;  // flagged by the forward
}

// Loads the rows of one GQA-packed 128-row tile: `hpc` heads starting at
// column col0 (one head per BP rows), each 128-byte swizzle atom of 64
// columns 128 x 128 bytes apart.
template <int D>
__device__ __forceinline__ void load_packed_tile(uint8_t* dst, const CUtensorMap* m,
                                                 uint64_t* bar, int col0, int row0,
                                                 int hpc, int BP) {
  for (int hh = 0; hh < hpc; ++hh)
#pragma unroll
    for (int at = 0; at < D / 64; ++at)
      tma_load_2d(dst + at * (AM * 128) + hh * BP * 128, m, bar, col0 + hh * D + at * 64,
                  row0);
}

// One K / V (or other 128-row, one-head) tile.
template <int D>
__device__ __forceinline__ void load_head_tile(uint8_t* dst, const CUtensorMap* m,
                                               uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int at = 0; at < D / 64; ++at)
    tma_load_2d(dst + at * (AM * 128), m, bar, col0 + at * 64, row0);
}

// K-step offset (>> 4) of a K-major 128-row tile with D columns: 16 columns
// per step, 64-column swizzle atoms 128 x 128 bytes apart.
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
  return ((kk / 4) * (AM * 128) + (kk % 4) * 32) >> 4;
}

// =================================================================== dQ
// Tensor memory of the dQ kernel: S [0, 128), dP [128, 256), dQ [256,
// 256 + D), dz as fp16 pairs [256 + D, 320 + D).  A key tile is handled as
// two halves of 64 keys (S / dP columns 64 h ..; dz columns 32 h ..): every
// compute warp works through half 0 and then half 1, so that the tensor core
// runs one half's products (dQ += dz K and the next tile's S, dP) while the
// compute warps work on the other.
template <int D>
struct DqLayout {
  static constexpr uint32_t TILE = AM * D * 2;
  static constexpr int SLOTS = D == 64 ? 4 : 2;  // (K, V) pairs
  static constexpr uint32_t Q_OFF = 0, DO_OFF = TILE, KV_OFF = 2 * TILE;
  static constexpr uint32_t BAR_OFF = KV_OFF + SLOTS * 2 * TILE;
  static constexpr uint32_t TOTAL = BAR_OFF + 512 + 1024;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256, DZ_COL = 256 + D;
  static_assert(DZ_COL + 64 <= 512, "tensor memory budget");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

struct QItem {
  int a0, L, q0, h0, g, n_tiles;
};

// Work item i: query block from the top (longest causal range first), then
// head group, then sequence.
__device__ __forceinline__ QItem q_item(const AttnBwdArgs& a, int i, int n_hg, int n_seq,
                                        int n_qb, int BP) {
  QItem it;
  const int per_qb = n_hg * n_seq;
  const int qb = n_qb - 1 - i / per_qb;
  const int rem = i - (i / per_qb) * per_qb;
  const int hg = rem % n_hg, s = rem / n_hg;
  it.h0 = hg * a.hpc;
  it.g = it.h0 / (a.n_heads / a.n_kv_heads);
  it.q0 = qb * BP;
  seq_range(a, s, it.a0, it.L);
  const int hi = min(it.q0 + BP, it.L);
  it.n_tiles = it.q0 < it.L ? (hi + AM - 1) / AM : 0;
  return it;
}

// dz of 32 key columns of one query row: p = 2^(s scale - lse) where
// visible (MASK: key e visible when e <= lim), dz = p (dP - D) (ndd = -D),
// packed fp16 pairs into wz.  Two columns at a time: the exponent on the
// paired fp32 pipe, 2^x of the fp16 pair on the SFU (two results per
// instruction), p widened back to fp32 for dz.
template <bool MASK>
__device__ __forceinline__ void dq_chunk(const float* sv, const float* dp, float scale,
                                         float lse, float ndd, int lim, uint32_t* wz) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float2 x = ffma2(sv[e], sv[e + 1], scale, scale, -lse, -lse);
    uint32_t pw = ex2_f16x2(pack_f16x2(x.x, x.y));
    if (MASK) pw &= (e <= lim ? 0xffffu : 0u) | (e + 1 <= lim ? 0xffff0000u : 0u);
    const float2 p = unpack_f16x2(pw);
    const float2 t = ffma2(dp[e], dp[e + 1], 1.f, 1.f, ndd, ndd);  // dP - D
    const float2 z = ffma2(p.x, p.y, t.x, t.y, 0.f, 0.f);
    wz[e / 2] = pack_f16x2(z.x, z.y);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmKV,
                       const __grid_constant__ CUtensorMap tmdO, AttnBwdArgs a,
                       int n_items, int n_hg, int n_seq, int n_qb) {
  using L = DqLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bar;                   // [SLOTS]
  uint64_t* kv_empty = kv_full + L::SLOTS;   // [SLOTS]
  uint64_t* q_full = kv_empty + L::SLOTS;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_empty + 1;  // [2] commit: S, dP of a half computed
  uint64_t* p_full = s_full + 2;   // [2] 256 arrivals: the half's S, dP read, dz written
  uint64_t* dz_free = p_full + 2;  // [2] commit: the half's dQ += dz K done
  uint64_t* dq_full = dz_free + 2;
  uint64_t* dq_free = dq_full + 1; // 256 arrivals: dQ read out
  uint64_t* drain = dq_free + 1;
  ItemRing* ring = reinterpret_cast<ItemRing*>(drain + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int BP = AM / a.hpc;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::SLOTS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], kCompute);
      mbar_init(&dz_free[h], 1);
    }
    mbar_init(dq_full, 1);
    mbar_init(dq_free, kCompute);
    mbar_init(drain, 1);
    ring_init(ring, 9);  // taken by the MMA warp and the eight compute warps
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmKV);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // q|k|v, dO, lse and D come from earlier kernels

  if (warp == kProducerWarp) {
    if (lane == 0) {
      uint32_t n = 0, k = 0, hand = 0;
      bool ok = true;
      while (ok) {
        const int i = ring_fetch(a.sched);  // in order: the longest range first
        if (i >= n_items) break;
        const QItem it = q_item(a, i, n_hg, n_seq, n_qb, BP);
        if (it.n_tiles == 0) continue;
        if (!ring_put(ring, hand, i, a.status, abort_flag)) {
          ok = false;
          break;
        }
        if (k > 0 && !bwait(q_empty, (k - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * L::TILE);
        load_packed_tile<D>(smem + L::Q_OFF, &tmQ, q_full, it.h0 * D, it.a0 + it.q0,
                            a.hpc, BP);
        load_packed_tile<D>(smem + L::DO_OFF, &tmdO, q_full, it.h0 * D, it.a0 + it.q0,
                            a.hpc, BP);
        ++k;
        const int kcol = (a.n_heads + it.g) * D, vcol = (a.n_heads + a.n_kv_heads + it.g) * D;
        for (int j = 0; j < it.n_tiles; ++j, ++n) {
          const int sl = n % L::SLOTS;
          if (!bwait(&kv_empty[sl], ((n / L::SLOTS) & 1) ^ 1, a.status,
                               abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + L::KV_OFF + sl * 2 * L::TILE;
          mbar_arrive_expect_tx(&kv_full[sl], 2 * L::TILE);
          load_head_tile<D>(dst, &tmKV, &kv_full[sl], kcol, it.a0 + j * AM);
          load_head_tile<D>(dst + L::TILE, &tmKV, &kv_full[sl], vcol, it.a0 + j * AM);
        }
      }
      if (ok) ring_put(ring, hand, -1, a.status, abort_flag);  // end of the items
      if (!ok) {  // let the copies already issued land (bounded)
        volatile int own = 0;
        const uint32_t m = n < (uint32_t)L::SLOTS ? n : (uint32_t)L::SLOTS;
        for (uint32_t j = 1; j <= m; ++j) {
          const uint32_t idx = n - j;
          bwait(&kv_full[idx % L::SLOTS], (idx / L::SLOTS) & 1, a.status, &own);
        }
        if (k > 0) bwait(q_full, (k - 1) & 1, a.status, &own);
      }
    }
  } else if (warp == kMmaWarp) {
    constexpr uint32_t idesc_s = idesc_f16(AM, 64);                // one half's keys
    constexpr uint32_t idesc_dq = idesc_f16(AM, D) | (1u << 16);  // B MN-major
    const uint64_t q_desc = sdesc_k128(smem_u32(smem + L::Q_OFF));
    const uint64_t do_desc = sdesc_k128(smem_u32(smem + L::DO_OFF));
    const uint64_t kv_desc = sdesc_k128(smem_u32(smem + L::KV_OFF));
    const uint64_t kmn_desc = sdesc_mn128(smem_u32(smem + L::KV_OFF), AM * 128);
    constexpr uint32_t PAIR16 = (2 * L::TILE) >> 4, TILE16 = L::TILE >> 4;
    constexpr uint32_t HALF16 = (64 * 128) >> 4;  // rows 64 .. of a K-major tile
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, bwait(b, parity, a.status, abort_flag));
    };
    uint32_t g = 0, n = 0, k = 0, hand = 0;
    bool ok = true, issued_any = false;
    while (ok) {
      int i;
      if (!ring_get(ring, hand, i, a.status, abort_flag)) {
        ok = false;
        break;
      }
      if (i < 0) break;
      const QItem it = q_item(a, i, n_hg, n_seq, n_qb, BP);
      if (!wait_all(q_full, k & 1)) {
        ok = false;
        break;
      }
      ++k;
      const int nt = it.n_tiles;
      // S = Q K^T and dP = dO V^T of half h of key tile j (its S / dP
      // columns were read by the compute warps: p_full of the tile before,
      // waited for ahead of that tile's dQ product)
      auto issue_s = [&](int j, int h) -> bool {
        const uint32_t kn = n + j;
        if (h == 0 && !wait_all(&kv_full[kn % L::SLOTS], (kn / L::SLOTS) & 1)) return false;
        tc_fence_after();
        const uint64_t kd = kv_desc + (kn % L::SLOTS) * PAIR16 + h * HALF16;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = kmajor_step(kk);
            tc_mma_bf16_nc(tmem_base + L::S_COL + 64 * h, q_desc + o, kd + o, idesc_s,
                           kk > 0);
            tc_mma_bf16_nc(tmem_base + L::DP_COL + 64 * h, do_desc + o, kd + TILE16 + o,
                           idesc_s, kk > 0);
          }
          tc_commit(&s_full[h]);
          if (j == nt - 1 && h == 1) tc_commit(q_empty);
        }
        __syncwarp();
        issued_any = true;
        return true;
      };
      // dQ += dz K over the 64 keys of half h of tile j
      auto issue_dq = [&](int j, int h) -> bool {
        const uint32_t jn = n + j;
        if (!wait_all(&p_full[h], (g + j) & 1) ||
            (j == 0 && h == 0 && k > 1 && !wait_all(dq_free, (k - 2) & 1)))
          return false;
        tc_fence_after();
        const uint64_t bd = kmn_desc + (jn % L::SLOTS) * PAIR16;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // keys 64 h + 16 kk ..: warpgroup kk / 2 wrote them as 8 columns
            // at 8 (kk % 2) of its 16
            const uint32_t col = L::DZ_COL + 32 * h + (kk / 2) * 16 + (kk % 2) * 8;
            tc_mma_ts(tmem_base + L::DQ_COL, tmem_base + col,
                      bd + (4 * h + kk) * (2048 >> 4), idesc_dq,
                      (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&dz_free[h]);
          if (h == 1) tc_commit(&kv_empty[jn % L::SLOTS]);
          if (j == nt - 1 && h == 1) tc_commit(dq_full);
        }
        __syncwarp();
        issued_any = true;
        return true;
      };
      ok = issue_s(0, 0) && issue_s(0, 1);
      for (int j = 0; j < nt && ok; ++j)
        for (int h = 0; h < 2 && ok; ++h)
          ok = issue_dq(j, h) && (j + 1 >= nt || issue_s(j + 1, h));
      g += nt;
      n += nt;
    }
    if (!ok && issued_any) {
      volatile int own = 0;
      if (elect_one()) tc_commit(drain);
      __syncwarp();
      bwait(drain, 0, a.status, &own);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int wq = warp & 3, wg = warp >> 2;  // lane quadrant, 32-key slot of a half
    const int r = wq * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(wq * 32) << 16);
    const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
    auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      int w_ok = 1;
      if (lane == 0) w_ok = bwait(b, parity, a.status, abort_flag);
      return __shfl_sync(0xffffffffu, w_ok, 0) != 0;
    };
    uint32_t g = 0, k = 0, hand = 0;
    bool ok = true;
    while (ok) {
      int i;
      if (!ring_get(ring, hand, i, a.status, abort_flag)) {
        ok = false;
        break;
      }
      if (i < 0) break;
      const QItem it = q_item(a, i, n_hg, n_seq, n_qb, BP);
      ++k;
      const int pos = it.q0 + r % BP, head = it.h0 + r / BP;
      const bool valid = pos < it.L;
      const size_t row = (size_t)(it.a0 + (valid ? pos : 0));
      const float lse = valid ? a.lse[row * a.n_heads + head] : 0.f;
      const float dd = valid ? a.dsum[row * a.n_heads + head] : 0.f;
      for (int j = 0; j < it.n_tiles; ++j, ++g) {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          if (!warp_wait(&s_full[h], g & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int c0 = 64 * h + 32 * wg;  // first key column of this warp's chunk
          float sv[32], dp[32];
          tmem_ld32_nowait(lane_base + L::S_COL + c0, sv);
          tmem_ld32_nowait(lane_base + L::DP_COL + c0, dp);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            tmem_pin(sv[e]);
            tmem_pin(dp[e]);
          }
          // keys 0 .. lim of the chunk are visible (none for a row past the
          // sequence end); a warp whose rows all see the whole chunk skips
          // the mask
          const int lim = (valid ? pos - j * AM : -1) - c0;
          uint32_t wz[16];
          if (__all_sync(0xffffffffu, lim >= 31))
            dq_chunk<false>(sv, dp, scale, lse, -dd, lim, wz);
          else
            dq_chunk<true>(sv, dp, scale, lse, -dd, lim, wz);
          // the half's dz columns are free once its previous dQ += dz K is done
          if (!warp_wait(&dz_free[h], (g & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          tmem_st16_words(lane_base + L::DZ_COL + 32 * h + 16 * wg, wz);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&p_full[h]);
        }
        if (!ok) break;
      }
      if (!ok) break;
      // ---- dq = dQ / sqrt(d), rotated back, fp16 (32-column pairs shared
      // out between the warpgroups)
      if (!warp_wait(dq_full, (k - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int half = D / 2;
      const int tp = valid ? table_row(a, (int)row) : 0;
      __half* dst = a.dqkv + row * a.nqkv + head * D;
      const float sc = rsqrtf((float)D);
#pragma unroll 1
      for (int c = wg * 32; c < half; c += 64) {
        float x1[32], x2[32];
        tmem_ld32_nowait(lane_base + L::DQ_COL + c, x1);
        tmem_ld32_nowait(lane_base + L::DQ_COL + half + c, x2);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          tmem_pin(x1[e]);
          tmem_pin(x2[e]);
        }
        if (valid) rope_back_store(a, tp, c, half, sc, x1, x2, dst);
      }
      tc_fence_before();
      mbar_arrive(dq_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0) ring_leave(a.sched);
}

// =================================================================== dK, dV
// Tensor memory of the dK / dV kernel: S^T [0, 128), dP^T [128, 256), dK
// [256, 256 + D), dV [256 + D, 256 + 2 D).  A query tile is handled as two
// halves of 64 queries (columns 64 h .. 64 h + 63 of S^T and dP^T): every
// compute warp works through half 0 and then half 1, and P^T / dz^T of a
// half overwrite the first 16 of each 32 S^T / dP^T columns a warpgroup
// read, so that the tensor core runs one half's products (dV, dK and the
// next tile's S^T, dP^T) while the compute warps work on the other.
template <int D>
struct DkvLayout {
  static constexpr uint32_t TILE = AM * D * 2;
  static constexpr int SLOTS = D == 64 ? 3 : 2;  // (Q, dO) pairs
  static constexpr uint32_t K_OFF = 0, V_OFF = TILE, Q_OFF = 2 * TILE;
  static constexpr uint32_t LSE_OFF = Q_OFF + SLOTS * 2 * TILE;  // [2][128] -lse, [2][128] -D
  static constexpr uint32_t BAR_OFF = LSE_OFF + 4 * AM * 4;
  static constexpr uint32_t TOTAL = BAR_OFF + 512 + 1024;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DK_COL = 256, DV_COL = 256 + D;
  static_assert(DV_COL + D <= 512, "tensor memory budget");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

struct KItem {
  int a0, L, k0, g, qb0, nqb, nq;
};

// Work item i: key tile from the front (the longest list of query tiles
// first), then kv head, then sequence.  Its query tiles: for each of the
// group's n_rep / hpc head groups, the query blocks from the one holding
// position k0 to the end of the sequence.
__device__ __forceinline__ KItem k_item(const AttnBwdArgs& a, int i, int n_seq, int BP) {
  KItem it;
  const int per_kt = a.n_kv_heads * n_seq;
  const int kt = i / per_kt;
  const int rem = i - kt * per_kt;
  it.g = rem % a.n_kv_heads;
  const int s = rem / a.n_kv_heads;
  seq_range(a, s, it.a0, it.L);
  it.k0 = kt * AM;
  it.qb0 = it.k0 / BP;
  it.nqb = it.k0 < it.L ? (it.L + BP - 1) / BP - it.qb0 : 0;
  it.nq = it.nqb * ((a.n_heads / a.n_kv_heads) / a.hpc);
  return it;
}

// Query tile q of item `it`: first head and first position.
__device__ __forceinline__ void k_item_tile(const AttnBwdArgs& a, const KItem& it, int q,
                                            int BP, int& h0, int& q0) {
  const int hgl = q / it.nqb;
  q0 = (it.qb0 + (q - hgl * it.nqb)) * BP;
  h0 = it.g * (a.n_heads / a.n_kv_heads) + hgl * a.hpc;
}

// P^T and dz^T of 32 query columns of one key row: p = 2^(s scale - lse)
// where visible, dz = p (dP - D); packed fp16 pairs into wp / wz.  nls and
// nds hold -lse and -D of each column.  MASK: column c (of the tile) is
// visible when (c & bm) >= rel.  Two columns at a time as in dq_chunk; dz is
// formed from the same fp16 p that dV's product uses.
template <bool MASK>
__device__ __forceinline__ void dkv_chunk(const float* sv, const float* dp, const float* nls,
                                          const float* nds, float scale, int c0, int bm,
                                          int rel, uint32_t* wp, uint32_t* wz) {
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 l4 = reinterpret_cast<const float4*>(nls + c0)[e4];
    const float4 d4 = reinterpret_cast<const float4*>(nds + c0)[e4];
    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int j = e4 * 4 + e;
      const float2 x = ffma2(sv[j], sv[j + 1], scale, scale, lv[e], lv[e + 1]);
      uint32_t pw = ex2_f16x2(pack_f16x2(x.x, x.y));
      if (MASK)
        pw &= ((((c0 + j) & bm) >= rel) ? 0xffffu : 0u) |
              ((((c0 + j + 1) & bm) >= rel) ? 0xffff0000u : 0u);
      const float2 p = unpack_f16x2(pw);
      const float2 t = ffma2(dp[j], dp[j + 1], 1.f, 1.f, dv[e], dv[e + 1]);  // dP - D
      const float2 z = ffma2(p.x, p.y, t.x, t.y, 0.f, 0.f);
      wp[j / 2] = pw;
      wz[j / 2] = pack_f16x2(z.x, z.y);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmKV,
                        const __grid_constant__ CUtensorMap tmdO, AttnBwdArgs a,
                        int n_items, int n_seq) {
  using L = DkvLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* lse_s = reinterpret_cast<float*>(smem + L::LSE_OFF);  // [2][128] -lse
  float* dd_s = lse_s + 2 * AM;                                 // [2][128] -D
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bar;                   // [SLOTS]
  uint64_t* q_empty = q_full + L::SLOTS;    // [SLOTS]
  uint64_t* kv_full = q_empty + L::SLOTS;
  uint64_t* kv_empty = kv_full + 1;
  uint64_t* s_full = kv_empty + 1;   // [2] commit: S^T, dP^T of a half computed
  uint64_t* s_free = s_full + 2;     // [2] commit: the half's dV, dK products done
  uint64_t* p_full = s_free + 2;     // [2] 256 arrivals: the half's P^T, dz^T written
  uint64_t* acc_full = p_full + 2;
  uint64_t* acc_free = acc_full + 1;  // 256 arrivals: dK, dV read out
  uint64_t* lse_ready = acc_free + 1; // [2] 256 arrivals: lse / D of a tile in smem
  uint64_t* drain = lse_ready + 2;
  ItemRing* ring = reinterpret_cast<ItemRing*>(drain + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int BP = AM / a.hpc;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::SLOTS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&s_free[h], 1);
      mbar_init(&p_full[h], kCompute);
      mbar_init(&lse_ready[h], kCompute);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_free, kCompute);
    mbar_init(drain, 1);
    ring_init(ring, 9);  // taken by the MMA warp and the eight compute warps
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmKV);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();

  if (warp == kProducerWarp) {
    if (lane == 0) {
      uint32_t n = 0, k = 0, hand = 0;
      bool ok = true;
      while (ok) {
        const int i = ring_fetch(a.sched + 2);  // in order: the longest range first
        if (i >= n_items) break;
        const KItem it = k_item(a, i, n_seq, BP);
        if (it.nq == 0) continue;
        if (!ring_put(ring, hand, i, a.status, abort_flag)) {
          ok = false;
          break;
        }
        if (k > 0 && !bwait(kv_empty, (k - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(kv_full, 2 * L::TILE);
        load_head_tile<D>(smem + L::K_OFF, &tmKV, kv_full, (a.n_heads + it.g) * D,
                          it.a0 + it.k0);
        load_head_tile<D>(smem + L::V_OFF, &tmKV, kv_full,
                          (a.n_heads + a.n_kv_heads + it.g) * D, it.a0 + it.k0);
        ++k;
        for (int q = 0; q < it.nq; ++q, ++n) {
          int h0, q0;
          k_item_tile(a, it, q, BP, h0, q0);
          const int sl = n % L::SLOTS;
          if (!bwait(&q_empty[sl], ((n / L::SLOTS) & 1) ^ 1, a.status,
                               abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + L::Q_OFF + sl * 2 * L::TILE;
          mbar_arrive_expect_tx(&q_full[sl], 2 * L::TILE);
          load_packed_tile<D>(dst, &tmQ, &q_full[sl], h0 * D, it.a0 + q0, a.hpc, BP);
          load_packed_tile<D>(dst + L::TILE, &tmdO, &q_full[sl], h0 * D, it.a0 + q0, a.hpc,
                              BP);
        }
      }
      if (ok) ring_put(ring, hand, -1, a.status, abort_flag);  // end of the items
      if (!ok) {
        volatile int own = 0;
        const uint32_t m = n < (uint32_t)L::SLOTS ? n : (uint32_t)L::SLOTS;
        for (uint32_t j = 1; j <= m; ++j) {
          const uint32_t idx = n - j;
          bwait(&q_full[idx % L::SLOTS], (idx / L::SLOTS) & 1, a.status, &own);
        }
        if (k > 0) bwait(kv_full, (k - 1) & 1, a.status, &own);
      }
    }
  } else if (warp == kMmaWarp) {
    constexpr uint32_t idesc_s = idesc_f16(AM, 64);                 // one half's queries
    constexpr uint32_t idesc_acc = idesc_f16(AM, D) | (1u << 16);  // B MN-major
    const uint64_t k_desc = sdesc_k128(smem_u32(smem + L::K_OFF));
    const uint64_t v_desc = sdesc_k128(smem_u32(smem + L::V_OFF));
    const uint64_t q_desc = sdesc_k128(smem_u32(smem + L::Q_OFF));
    const uint64_t qmn_desc = sdesc_mn128(smem_u32(smem + L::Q_OFF), AM * 128);
    constexpr uint32_t PAIR16 = (2 * L::TILE) >> 4, TILE16 = L::TILE >> 4;
    constexpr uint32_t HALF16 = (64 * 128) >> 4;  // rows 64 .. of a K-major tile
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, bwait(b, parity, a.status, abort_flag));
    };
    uint32_t gi = 0, n = 0, k = 0, hand = 0;
    bool ok = true, issued_any = false;
    while (ok) {
      int i;
      if (!ring_get(ring, hand, i, a.status, abort_flag)) {
        ok = false;
        break;
      }
      if (i < 0) break;
      const KItem it = k_item(a, i, n_seq, BP);
      if (!wait_all(kv_full, k & 1)) {
        ok = false;
        break;
      }
      ++k;
      const int nq = it.nq;
      // S^T = K Q^T and dP^T = V dO^T of half h of query tile q (its S^T /
      // dP^T columns are free once the half's products of the tile before
      // are done)
      auto issue_s = [&](int q, int h) -> bool {
        const uint32_t qn = n + q;
        if ((h == 0 && !wait_all(&q_full[qn % L::SLOTS], (qn / L::SLOTS) & 1)) ||
            !wait_all(&s_free[h], ((gi + q) & 1) ^ 1))
          return false;
        tc_fence_after();
        const uint32_t so = (qn % L::SLOTS) * PAIR16 + h * HALF16;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = kmajor_step(kk);
            tc_mma_bf16_nc(tmem_base + L::S_COL + 64 * h, k_desc + o, q_desc + so + o,
                           idesc_s, kk > 0);
            tc_mma_bf16_nc(tmem_base + L::DP_COL + 64 * h, v_desc + o,
                           q_desc + so + TILE16 + o, idesc_s, kk > 0);
          }
          tc_commit(&s_full[h]);
          if (q == nq - 1 && h == 1) tc_commit(kv_empty);  // K and V no longer read
        }
        __syncwarp();
        issued_any = true;
        return true;
      };
      // dV += P^T dO, dK += dz^T Q over the 64 queries of half h of tile q
      auto issue_acc = [&](int q, int h) -> bool {
        const uint32_t qn = n + q;
        if (!wait_all(&p_full[h], (gi + q) & 1) ||
            (q == 0 && h == 0 && k > 1 && !wait_all(acc_free, (k - 2) & 1)))
          return false;
        tc_fence_after();
        const uint64_t qb = qmn_desc + (qn % L::SLOTS) * PAIR16;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (q > 0 || h > 0 || kk > 0) ? 1u : 0u;
            // queries 64 h + 16 kk ..: warpgroup kk / 2 wrote them as 8
            // columns at 8 (kk % 2) of its 32
            const uint32_t col = 64 * h + (kk / 2) * 32 + (kk % 2) * 8;
            const uint32_t kb = (4 * h + kk) * (2048 >> 4);
            tc_mma_ts(tmem_base + L::DV_COL, tmem_base + L::S_COL + col, qb + TILE16 + kb,
                      idesc_acc, acc);
            tc_mma_ts(tmem_base + L::DK_COL, tmem_base + L::DP_COL + col, qb + kb, idesc_acc,
                      acc);
          }
          tc_commit(&s_free[h]);
          if (h == 1) tc_commit(&q_empty[qn % L::SLOTS]);
          if (q == nq - 1 && h == 1) tc_commit(acc_full);
        }
        __syncwarp();
        issued_any = true;
        return true;
      };
      ok = issue_s(0, 0) && issue_s(0, 1);
      for (int q = 0; q < nq && ok; ++q)
        for (int h = 0; h < 2 && ok; ++h)
          ok = issue_acc(q, h) && (q + 1 >= nq || issue_s(q + 1, h));
      gi += nq;
      n += nq;
    }
    if (!ok && issued_any) {
      volatile int own = 0;
      if (elect_one()) tc_commit(drain);
      __syncwarp();
      bwait(drain, 0, a.status, &own);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int wq = warp & 3, wg = warp >> 2;  // lane quadrant, 32-column slot of a half
    const int r = wq * 32 + lane;             // key row of the tile == TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(wq * 32) << 16);
    const float scale = 1.4426950408889634f * rsqrtf((float)D);
    auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      int w_ok = 1;
      if (lane == 0) w_ok = bwait(b, parity, a.status, abort_flag);
      return __shfl_sync(0xffffffffu, w_ok, 0) != 0;
    };
    uint32_t gi = 0, k = 0, hand = 0;
    bool ok = true;
    while (ok) {
      int i;
      if (!ring_get(ring, hand, i, a.status, abort_flag)) {
        ok = false;
        break;
      }
      if (i < 0) break;
      const KItem it = k_item(a, i, n_seq, BP);
      ++k;
      const int kp = it.k0 + r;
      const bool kvalid = kp < it.L;
      // -lse (warpgroup 0) or -D (warpgroup 1) of query row r of tile q,
      // loaded one tile ahead so that the load overlaps the previous tile's
      // work (-inf, 0 past the sequence end)
      auto fetch = [&](int q) -> float {
        int h0, q0;
        k_item_tile(a, it, q, BP, h0, q0);
        const int qp = q0 + r % BP, qh = h0 + r / BP;
        const bool qv = qp < it.L;
        const size_t qrow = (size_t)(it.a0 + (qv ? qp : 0)) * a.n_heads + qh;
        const float v = ldg_now((wg == 0 ? a.lse : a.dsum) + qrow);
        if (wg == 0) return qv ? -v : -INFINITY;
        return qv ? -v : 0.f;
      };
      float next = fetch(0);
      for (int q = 0; q < it.nq; ++q, ++gi) {
        int h0, q0;
        k_item_tile(a, it, q, BP, h0, q0);
        // into shared memory (double buffered: a thread writes buffer b
        // again only after every thread has arrived for the tile in
        // between, i.e. is done reading it)
        {
          const int b = gi & 1;
          (wg == 0 ? lse_s : dd_s)[b * AM + r] = next;
          mbar_arrive(&lse_ready[b]);
          if (q + 1 < it.nq) next = fetch(q + 1);
        }
        if (!warp_wait(&lse_ready[gi & 1], (gi >> 1) & 1)) {
          ok = false;
          break;
        }
        const float* ls = lse_s + (gi & 1) * AM;
        const float* ds = dd_s + (gi & 1) * AM;
        // query column c sits at position q0 + (c & (BP - 1)) (BP a power of
        // two): key kp is visible to it when kp <= that position; lse = +inf
        // past the sequence end.  Below the diagonal (every key of this warp
        // at or before q0) nothing is masked.
        const bool full = q0 >= it.k0 + wq * 32 + 31;
        const int rel = kvalid ? kp - q0 : AM;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          if (!warp_wait(&s_full[h], gi & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int c0 = 64 * h + 32 * wg;  // first query column of this warp's chunk
          float sv[32], dp[32];
          tmem_ld32_nowait(lane_base + L::S_COL + c0, sv);
          tmem_ld32_nowait(lane_base + L::DP_COL + c0, dp);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            tmem_pin(sv[e]);
            tmem_pin(dp[e]);
          }
          uint32_t wp[16], wz[16];
          if (full)
            dkv_chunk<false>(sv, dp, ls, ds, scale, c0, BP - 1, rel, wp, wz);
          else
            dkv_chunk<true>(sv, dp, ls, ds, scale, c0, BP - 1, rel, wp, wz);
          tmem_st16_words(lane_base + L::S_COL + c0, wp);
          tmem_st16_words(lane_base + L::DP_COL + c0, wz);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&p_full[h]);
        }
        if (!ok) break;
      }
      if (!ok) break;
      // ---- dk (scaled, rotated back) and dv of the tile's keys, 32-column
      // pieces shared out between the warpgroups
      if (!warp_wait(acc_full, (k - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int half = D / 2;
      const size_t row = (size_t)(it.a0 + (kvalid ? kp : 0));
      const int tp = kvalid ? table_row(a, (int)row) : 0;
      __half* dk = a.dqkv + row * a.nqkv + (a.n_heads + it.g) * D;
      __half* dv = a.dqkv + row * a.nqkv + (a.n_heads + a.n_kv_heads + it.g) * D;
      const float sc = rsqrtf((float)D);
#pragma unroll 1
      for (int c = wg * 32; c < half; c += 64) {
        float x1[32], x2[32];
        tmem_ld32_nowait(lane_base + L::DK_COL + c, x1);
        tmem_ld32_nowait(lane_base + L::DK_COL + half + c, x2);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          tmem_pin(x1[e]);
          tmem_pin(x2[e]);
        }
        if (kvalid) rope_back_store(a, tp, c, half, sc, x1, x2, dk);
      }
#pragma unroll 1
      for (int c = wg * 32; c < D; c += 64) {
        float v[32];
        tmem_ld32(lane_base + L::DV_COL + c, v);
        if (kvalid) store_f16x32(dv + c, v, 1.f);
      }
      tc_fence_before();
      mbar_arrive(acc_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0) ring_leave(a.sched + 2);
}

template <int D>
cudaError_t launch(const AttnBwdArgs& a, int n_seq, int max_len, int sm_count,
                   cudaStream_t s) {
  const int BP = AM / a.hpc;
  CUtensorMap tq, tkv, tdo;
  if (!tc_encode_bf16(&tq, a.qkv, a.tokens, a.nqkv, BP) ||
      !tc_encode_bf16(&tkv, a.qkv, a.tokens, a.nqkv, AM) ||
      !tc_encode_bf16(&tdo, a.dout, a.tokens, (uint64_t)a.n_heads * D, BP))
    return cudaErrorInvalidValue;
  // dq: one item per query tile
  {
    const int n_qb = (max_len + BP - 1) / BP, n_hg = a.n_heads / a.hpc;
    const long long items = (long long)n_qb * n_hg * n_seq;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    if (items > 0) {
      auto kern = attn_bwd_dq_kernel<D>;
      static std::atomic<uint64_t> attr_done{0};
      if (cudaError_t e = ensure_smem_attr(kern, (int)DqLayout<D>::TOTAL, attr_done);
          e != cudaSuccess)
        return e;
      const int grid = (int)(items < sm_count ? items : sm_count);
      cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreads), DqLayout<D>::TOTAL, s, tq,
                                 tkv, tdo, a, (int)items, n_hg, n_seq, n_qb);
      if (e != cudaSuccess) return e;
    }
  }
  // dk, dv: one item per key tile and kv head
  {
    const int n_kt = (max_len + AM - 1) / AM;
    const long long items = (long long)n_kt * a.n_kv_heads * n_seq;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    if (items > 0) {
      auto kern = attn_bwd_dkv_kernel<D>;
      static std::atomic<uint64_t> attr_done{0};
      if (cudaError_t e = ensure_smem_attr(kern, (int)DkvLayout<D>::TOTAL, attr_done);
          e != cudaSuccess)
        return e;
      const int grid = (int)(items < sm_count ? items : sm_count);
      cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreads), DkvLayout<D>::TOTAL, s,
                                 tq, tkv, tdo, a, (int)items, n_seq);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t attn_backward(const AttnBwdArgs& args, int n_seq, int max_len, int sm_count,
                          cudaStream_t s) {
  AttnBwdArgs a = args;
  a.hpc = heads_per_tile(a.n_heads / a.n_kv_heads);
  if (n_seq <= 0 || max_len <= 0 || a.tokens <= 0) return cudaSuccess;
  if (!a.sched) return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch<128>(a, n_seq, max_len, sm_count, s);
  if (a.head_dim == 64) return launch<64>(a, n_seq, max_len, sm_count, s);
  return cudaErrorInvalidValue;
}

}  // namespace llama
