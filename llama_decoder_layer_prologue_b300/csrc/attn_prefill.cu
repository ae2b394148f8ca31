// Causal grouped-query attention for prefill, padded or packed varlen
// ("模型层" 9.3 CausalSelfAttention; "parallel_attention.py" 2 step 4 and 3
// flash_attn_varlen_func): o = softmax(q k^T / sqrt(d) + causal mask) v within
// each sequence, query head h reading kv head h / n_rep.  q and k arrive
// already rotated by the QKV GEMM epilogue; q, k, v, P and the output are
// fp16 (fp16 x fp16 -> fp32 on the tensor cores).
//
// tcgen05 / TMEM flash attention, persistent (one CTA per SM), 12 warps.  A
// work item is two query tiles A and B of 128 rows each: `hpc` query heads of
// one kv group times BP = 128 / hpc positions, B holding the BP positions
// after A's, so every K / V tile feeds 256 query rows (repeat_kv is never
// materialised).
//   warps 0..3  softmax of tile A, warps 4..7 softmax of tile B: thread r of
//               a warpgroup owns query row r (TMEM lane r).  Per K / V tile
//               it loads its S row, masks, keeps the running max m and sum l,
//               and writes P = 2^(s - m) as fp16 into the 128-byte swizzled
//               P tile (the A operand of P V); at the end it reads its O row,
//               divides by l and stores fp16.
//   warp 8      TMA producer: the two Q tiles once per item, then K(j), V(j)
//               into a ring of single-tile slots.
//   warps 9, 10 one thread of warp 9 + t issues the tcgen05.mma of query
//               tile t in the order S_t(0), then S_t(j+1), PV_t(j): S = Q K^T
//               into the tile's TMEM S buffer, O += P V into its TMEM O
//               buffer (V read as an MN-major operand straight from its TMA
//               tile, P from TMEM or shared memory: see AttnLayout).  The two
//               tiles' products reach the tensor core independently, so while
//               one warpgroup computes its softmax the tensor core works on
//               the other's products.
// Rescaling of O is lazy: a row's reference max only moves (and O is
// rescaled in TMEM) when the new max exceeds it by more than 8 in the log2
// domain, so P stays <= 2^8.  Items are listed longest causal range first
// and taken in that order from a global counter (the producer thread hands
// each to the MMA and softmax warps through a shared-memory ring), so the
// CTAs finish together.  Every wait is bounded (2 s -> status bit, abort,
// drain, free TMEM).
#include <cuda_bf16.h>
#include <math.h>

#include "attn_prefill.cuh"
#include "common.cuh"
#include "gemm_tc.cuh"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;
constexpr int AM = 128;  // query rows per tile (MMA M)
constexpr float kRescaleLog2 = 8.0f;
// 12 warps = 3 warpgroups: the register file is shared out per warpgroup,
// so the block launches at 168 registers a thread (384 x 168 = 64512) and
// then moves registers with setmaxnreg: the two softmax warpgroups go up to
// kSoftmaxRegs, the producer / MMA warpgroup (warps 8..11, 11 idle)
// down to kControlRegs; 2 x 128 x 216 + 128 x 72 = 64512 (the split with the
// fewest spills: the softmax row holds 128 scores).
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kSoftmaxRegs = 216, kControlRegs = 72;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168,
              "register split exceeds the launch allocation");

// Each query tile has its own P tile, so a warpgroup only waits for its own
// previous P V.  head_dim 64: P lives in tensor memory (P_TMEM, 64 columns of
// fp16 pairs after S and O) and the P V product reads it as its A operand;
// shared memory holds the two query tiles and 8 K / V slots.  head_dim 128:
// S and O fill the 512 columns, so the two P tiles are 128-byte swizzled
// shared-memory tiles, next to the query tiles and 3 K / V slots of 32 KB.
template <int D>
struct AttnLayout {
  static constexpr int AN = 128;                    // keys per K / V tile
  static constexpr bool P_TMEM = D == 64;
  static constexpr int ATOMS = D / 64;  // 128-byte swizzle atoms per row
  static constexpr uint32_t Q_BYTES = AM * D * 2;   // one query tile
  static constexpr uint32_t KV_BYTES = AN * D * 2;  // one K or V tile (a slot)
  static constexpr uint32_t P_BYTES = AM * AN * 2;  // one P tile
  static constexpr int SLOTS = D == 64 ? 8 : 3;
  static constexpr uint32_t Q_OFF = 0;              // Q_A, Q_B
  static constexpr uint32_t P_OFF = Q_OFF + 2 * Q_BYTES;
  static constexpr uint32_t KV_OFF = P_OFF + (P_TMEM ? 0 : 2 * P_BYTES);
  static constexpr uint32_t BAR_OFF = KV_OFF + SLOTS * KV_BYTES;
  static constexpr uint32_t TOTAL = BAR_OFF + 512 + 1024;
  // S_A [0, AN), S_B [AN, 2 AN), O_A [2 AN, 2 AN + D), O_B [2 AN + D, 2 AN + 2 D),
  // then (P_TMEM) P_A, P_B: AN / 2 columns each
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t P_COL = 2 * AN + 2 * D;
  static_assert(P_COL + (P_TMEM ? AN : 0) <= TMEM_COLS, "tensor memory budget");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

struct Item {
  int a0, L, q0, h0, g;  // sequence start and length, first position, heads
  int n_tiles;           // K / V tiles of the causal range (0: nothing to do)
  int sp;                // position of the sequence's first query (cache: start_pos)
  int kbase;             // row of the sequence's key 0 in the K / V tensor map
  int kv_end;            // keys the item's queries can see: rows [0, kv_end)
};

// Work item i: query block from the top (longest causal range first), then
// head group, then sequence.  A block is 2 BP positions.
template <bool CACHED>
__device__ __forceinline__ Item get_item(const AttnArgs& a, int i, int n_hg,
                                         int n_seq, int n_qb, int BP, int AN) {
  Item it;
  const int per_qb = n_hg * n_seq;
  const int qb = n_qb - 1 - i / per_qb;
  const int rem = i - (i / per_qb) * per_qb;
  const int hg = rem % n_hg, s = rem / n_hg;
  const int n_rep = a.n_heads / a.n_kv_heads;
  it.h0 = hg * a.hpc;
  it.g = it.h0 / n_rep;
  it.q0 = qb * 2 * BP;
  it.sp = 0;
  if constexpr (CACHED) {
    const int sp = a.start_pos[s];
    it.a0 = s * a.seq_len;
    it.kbase = s * a.max_seq;
    // flagged by the positions kernel when the chunk does not fit
    const bool ok = sp >= 0 && sp <= a.max_seq - a.seq_len && sp <= a.max_pos - a.seq_len;
    it.L = ok ? a.seq_len : 0;
    it.sp = ok ? sp : 0;
  } else if (a.cu) {
    const int s0 = a.cu[s], s1 = a.cu[s + 1];
    if (s0 < 0 || s1 < s0 || s1 > a.tokens) {  // flagged by the positions kernel
      it.a0 = 0; it.L = 0;
    } else {
      it.a0 = s0; it.L = s1 - s0;
    }
    it.kbase = it.a0;
  } else {
    it.a0 = s * a.seq_len;
    it.L = a.seq_len;
    it.kbase = it.a0;
  }
  const int hi = min(it.q0 + 2 * BP, it.L);
  it.kv_end = it.sp + hi;
  it.n_tiles = it.q0 < it.L ? (it.kv_end + AN - 1) / AN : 0;
  return it;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) * (b, b) + (c, c) on the paired fp32 pipe.
__device__ __forceinline__ void fma2(float& a0, float& a1, float b, float c) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(z) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(x), "l"(y), "l"(z));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(x));
}

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

// (s0, s1) += (a0, a1)
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  uint64_t x, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(a0), "f"(a1));
  asm("add.f32x2 %0, %1, %2;" : "=l"(x) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(x));
}

// 16-bit pair of the P operand: fp16 with the fp16 q | k | v of the prefill,
// bf16 with the bf16 cache of a cached chunk (an MMA's A and B share a type).
template <bool BF>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  return BF ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// CACHED: keys and values from the KV-cache maps tmK / tmV (rows
// sequence * max_seq + key, columns kv head * D), bf16 operands; otherwise
// both from the q|k|v map (tmK == tmV), fp16 operands.
template <int D, bool CACHED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, AttnArgs a,
                   int n_items, int n_hg, int n_seq, int n_qb) {
  using L = AttnLayout<D>;
  constexpr int AN = L::AN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bar;                    // [SLOTS]
  uint64_t* kv_empty = kv_full + L::SLOTS;    // [SLOTS]
  uint64_t* s_full = kv_empty + L::SLOTS;     // [2] per query tile
  uint64_t* s_free = s_full + 2;              // [2]
  uint64_t* p_full = s_free + 2;              // [2]
  uint64_t* pv_done = p_full + 2;             // [2]
  uint64_t* o_free = pv_done + 2;             // [2]
  uint64_t* q_full = o_free + 2;
  uint64_t* q_empty = q_full + 1;
  uint64_t* drain = q_empty + 1;             // [2] per MMA warp
  ItemRing* ring = reinterpret_cast<ItemRing*>(drain + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int BP = AM / a.hpc;  // positions per query tile
  if (threadIdx.x == 0) {
    ring_init(ring, 10);  // taken by the two MMA warps and the eight softmax warps
    for (int s = 0; s < L::SLOTS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 2);  // a commit from each MMA warp
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 128);
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
      mbar_init(&o_free[t], 128);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // q|k|v come from the previous kernel

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
    if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t n = 0, k = 0, hand = 0;  // K / V tiles loaded, items started, handed out
      bool ok = true;
      while (ok) {
        // items in index order (longest causal range first), the empty ones
        // skipped here, the rest handed to the MMA and softmax warps
        const int i = ring_fetch(a.sched);
        if (i >= n_items) break;
        const Item it = get_item<CACHED>(a, i, n_hg, n_seq, n_qb, BP, L::AN);
        if (it.n_tiles == 0) continue;
        if (!ring_put(ring, hand, i, a.status, abort_flag)) {
          ok = false;
          break;
        }
        if (k > 0 && !mbar_wait_sleep(q_empty, (k - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * L::Q_BYTES);
        for (int t = 0; t < 2; ++t)
          for (int hh = 0; hh < a.hpc; ++hh)
            for (int at = 0; at < L::ATOMS; ++at)
              tma_load_2d(smem + L::Q_OFF + t * L::Q_BYTES + at * (AM * 128) +
                              hh * BP * 128,
                          &tmQ, q_full, (it.h0 + hh) * D + at * 64,
                          it.a0 + it.q0 + t * BP);
        ++k;
        const int col[2] = {CACHED ? it.g * D : (a.n_heads + it.g) * D,
                            CACHED ? it.g * D : (a.n_heads + a.n_kv_heads + it.g) * D};
        for (int j = 0; ok && j < it.n_tiles; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++n) {  // K(j), then V(j)
            const int sl = n % L::SLOTS;
            if (!mbar_wait_sleep(&kv_empty[sl], ((n / L::SLOTS) & 1) ^ 1, a.status,
                           abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem + L::KV_OFF + sl * L::KV_BYTES;
            mbar_arrive_expect_tx(&kv_full[sl], L::KV_BYTES);
            for (int at = 0; at < L::ATOMS; ++at)
              tma_load_2d(dst + at * (AN * 128), kv ? &tmV : &tmK, &kv_full[sl],
                          col[kv] + at * 64, it.kbase + j * AN);
          }
        }
      }
      if (ok) ring_put(ring, hand, -1, a.status, abort_flag);  // end of the items
      if (!ok) {  // let the copies already issued land (bounded)
        volatile int own = 0;
        const uint32_t m = n < (uint32_t)L::SLOTS ? n : (uint32_t)L::SLOTS;
        for (uint32_t j = 1; j <= m; ++j) {
          const uint32_t idx = n - j;
          mbar_wait_sleep(&kv_full[idx % L::SLOTS], (idx / L::SLOTS) & 1, a.status, &own);
        }
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ MMA issuers
    // Warp kMmaWarp + t issues the products of query tile t in order,
    // S_t(0), then S_t(j+1), PV_t(j) for each j; the two warps share the
    // tensor core, so neither tile's products wait for the other tile's
    // softmax.  K / V slots and the Q tiles are released by a commit from
    // each warp (barrier count 2).  One elected lane issues.
    const int t = warp - kMmaWarp;
    constexpr uint32_t idesc_s = CACHED ? idesc_bf16(AM, AN) : idesc_f16(AM, AN);
    constexpr uint32_t idesc_pv =
        (CACHED ? idesc_bf16(AM, D) : idesc_f16(AM, D)) | (1u << 16);  // B MN-major
    // descriptor bases; a K step adds its byte offset >> 4 to the address
    const uint64_t q_desc = sdesc_k128(smem_u32(smem + L::Q_OFF));
    const uint64_t p_desc = sdesc_k128(smem_u32(smem + L::P_OFF));
    const uint64_t k_desc = sdesc_k128(smem_u32(smem + L::KV_OFF));
    const uint64_t v_desc = sdesc_mn128(smem_u32(smem + L::KV_OFF), AN * 128);
    constexpr uint32_t SLOT16 = L::KV_BYTES >> 4, Q16 = L::Q_BYTES >> 4;
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_sleep(b, parity, a.status, abort_flag));
    };
    const uint64_t qd = q_desc + t * Q16;
    const uint32_t s_tmem = tmem_base + t * AN;
    const uint32_t o_tmem = tmem_base + 2 * AN + t * D;
    uint32_t g = 0, n = 0, k = 0, hand = 0;  // tiles, K / V loads consumed, items
    bool ok = true, issued_any = false;
    while (ok) {
      int i;
      if (!ring_get(ring, hand, i, a.status, abort_flag)) {
        ok = false;
        break;
      }
      if (i < 0) break;
      const Item it = get_item<CACHED>(a, i, n_hg, n_seq, n_qb, BP, L::AN);
      if (!wait_all(q_full, k & 1)) {
        ok = false;
        break;
      }
      ++k;
      const int nt = it.n_tiles;
      // K(j) is K / V load number n + 2 j, V(j) number n + 2 j + 1.
      for (int step = -1; step < nt && ok; ++step) {
        const int js = step + 1;  // tile of the S product
        if (js < nt) {
          const uint32_t kn = n + 2 * js, gs = g + js;
          if (!wait_all(&kv_full[kn % L::SLOTS], (kn / L::SLOTS) & 1) ||
              !wait_all(&s_free[t], (gs & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = k_desc + (kn % L::SLOTS) * SLOT16;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t qo = ((kk / 4) * (AM * 128) + (kk % 4) * 32) >> 4;
              const uint32_t ko = ((kk / 4) * (AN * 128) + (kk % 4) * 32) >> 4;
              tc_mma_bf16_nc(s_tmem, qd + qo, kd + ko, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[t]);
            tc_commit(&kv_empty[kn % L::SLOTS]);  // this tile is done with K(js)
            if (js == nt - 1) tc_commit(q_empty);  // ... and with its Q tile
          }
          __syncwarp();
          issued_any = true;
        }
        if (step < 0) continue;
        // PV_t(j)
        const int j = step;
        const uint32_t vn = n + 2 * j + 1, gp = g + j;
        const bool first = j == 0;
        if (!wait_all(&kv_full[vn % L::SLOTS], (vn / L::SLOTS) & 1) ||
            !wait_all(&p_full[t], gp & 1) ||
            (first && k > 1 && !wait_all(&o_free[t], (k - 2) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (CACHED) {
          // cache rows past what any query of the item sees hold whatever the
          // caller left there (NaN included): P is 0 for them, and 0 * NaN
          // would still poison the sum, so their V rows become zeros
          const int r0 = it.kv_end - j * AN;
          if (r0 < AN) {
            uint8_t* vs = smem + L::KV_OFF + (vn % L::SLOTS) * L::KV_BYTES;
            const int n16 = (AN - r0) * 8;  // 16-byte pieces per atom
            for (int e = lane; e < n16 * L::ATOMS; e += 32) {
              const int at = e / n16, w = e - at * n16;
              *reinterpret_cast<uint4*>(vs + at * (AN * 128) + (r0 + w / 8) * 128 +
                                        (w % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        const uint64_t vd = v_desc + (vn % L::SLOTS) * SLOT16;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < AN / 16; ++kk) {
            if constexpr (L::P_TMEM) {  // A = P_t in tensor memory, 8 columns per K step
              tc_mma_ts(o_tmem, tmem_base + L::P_COL + t * (AN / 2) + kk * 8,
                        vd + kk * (2048 >> 4), idesc_pv, (!first || kk > 0) ? 1u : 0u);
            } else {
              const uint32_t po = ((kk / 4) * (AM * 128) + (kk % 4) * 32) >> 4;
              tc_mma_bf16_nc(o_tmem, p_desc + t * (L::P_BYTES >> 4) + po,
                             vd + kk * (2048 >> 4), idesc_pv,
                             (!first || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(&pv_done[t]);
          tc_commit(&kv_empty[vn % L::SLOTS]);  // this tile is done with V(j)
        }
        __syncwarp();
        issued_any = true;
      }
      g += nt;
      n += 2 * nt;
    }
    if (!ok && issued_any) {  // wait for this warp's MMAs in flight
      volatile int own = 0;
      if (elect_one()) tc_commit(&drain[t]);
      __syncwarp();
      mbar_wait_sleep(&drain[t], 0, a.status, &own);
    }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;               // query tile: 0 = A, 1 = B
    const int r = (warp & 3) * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = t * AN, o_col = 2 * AN + t * D;
    uint8_t* prow = smem + L::P_OFF + t * L::P_BYTES + r * 128;  // head_dim 128
    const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
    uint32_t g = 0, hand = 0;
    bool ok = true;
    auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait_sleep(b, parity, a.status, abort_flag);
      return __shfl_sync(0xffffffffu, w_ok, 0) != 0;
    };
    while (ok) {
      int i;
      if (!ring_get(ring, hand, i, a.status, abort_flag)) {
        ok = false;
        break;
      }
      if (i < 0) break;
      const Item it = get_item<CACHED>(a, i, n_hg, n_seq, n_qb, BP, L::AN);
      const int q0 = it.q0 + t * BP;  // first position of this tile
      const int pos = q0 + (r % BP);
      const int head = it.h0 + r / BP;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n_tiles; ++j, ++g) {
        if (!warp_wait(&s_full[t], g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[AN];
#pragma unroll
        for (int c = 0; c < AN / 32; ++c)
          tmem_ld32_nowait(lane_base + s_col + c * 32, s + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < AN; ++c) tmem_pin(s[c]);
        tc_fence_before();
        mbar_arrive(&s_free[t]);
        // causal mask (keys after the row's position), tile max of the raw
        // scores (8 independent chains)
        const int kb = j * AN;
        if (kb + AN - 1 > it.sp + q0) {
          const int lim = it.sp + pos - kb;
#pragma unroll
          for (int c = 0; c < AN; ++c) s[c] = c > lim ? -INFINITY : s[c];
        }
        float pm[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pm[e] = fmaxf(s[e], s[e + 8]);
#pragma unroll
        for (int c = 16; c < AN; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) pm[e] = max3(pm[e], s[c + e], s[c + 8 + e]);
        const float tmax =
            max3(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], pm[5]),
                 fmaxf(pm[6], pm[7])) * scale;
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m = tmax;
        } else if (tmax > m + kRescaleLog2) {
          alpha = ex2(m - tmax);
          rescale = true;
          m = tmax;
          l *= alpha;
        }
        const float mref = m == -INFINITY ? 0.f : m;
        // p = 2^(s * scale - m): the exponent in fp32 (paired FMA); fp16 P
        // (the fp16 q|k|v path) takes it as an fp16 pair through the packed
        // SFU exp2, two results per instruction, and sums the fp16 values
        // the P V product uses (eight fp16 pair partial sums of 8 pairs,
        // then fp32); bf16 P (a cached chunk) stays in fp32 throughout
        uint32_t pw[AN / 2];
        if constexpr (!CACHED) {
          uint32_t hs[8];
#pragma unroll
          for (int c = 0; c < AN; c += 2) {
            fma2(s[c], s[c + 1], scale, -mref);
            pw[c / 2] = ex2_f16x2(pack_f16x2(s[c], s[c + 1]));
            const int a8 = (c / 2) & 7;
            hs[a8] = c < 16 ? pw[c / 2] : hadd2_u32(hs[a8], pw[c / 2]);
          }
          float lt = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 f = unpack_f16x2(hs[e]);
            lt += f.x + f.y;
          }
          l += lt;
        } else {
          float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < AN; c += 2) {
            fma2(s[c], s[c + 1], scale, -mref);
            s[c] = ex2(s[c]);
            s[c + 1] = ex2(s[c + 1]);
            add2(ps[c & 7], ps[(c & 7) + 1], s[c], s[c + 1]);
            pw[c / 2] = pack_p<CACHED>(s[c], s[c + 1]);
          }
          l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        }
        // This tile's P buffer and O are free once its previous P V is done
        // (for the first tile of an item the epilogue already waited).
        if (j > 0) {
          if (!warp_wait(&pv_done[t], (g - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            const uint32_t ta = lane_base + o_col + c * 32;
            tmem_ld32(ta, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(ta, o);
          }
        }
        if constexpr (L::P_TMEM) {
          // P as fp16 pairs into this row's TMEM lane (the P V A operand)
          const uint32_t p_tmem = lane_base + L::P_COL + t * (AN / 2);
#pragma unroll
          for (int h = 0; h < AN / 32; ++h) tmem_st16_words(p_tmem + h * 16, pw + h * 16);
          tmem_wait_st();
        } else {
          // P as fp16 into the 128-byte swizzled A tile
#pragma unroll
          for (int c16 = 0; c16 < AN / 8; ++c16) {
            uint4 u;
            u.x = pw[c16 * 4 + 0];
            u.y = pw[c16 * 4 + 1];
            u.z = pw[c16 * 4 + 2];
            u.w = pw[c16 * 4 + 3];
            const int atom = c16 / 8, cc = c16 % 8;
            *reinterpret_cast<uint4*>(prow + atom * (AM * 128) + ((cc ^ (r & 7)) << 4)) = u;
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      if (!ok) break;
      // ---- epilogue: O / l -> fp16, rows inside the sequence only
      if (!warp_wait(&pv_done[t], (g - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool valid = pos < it.L;
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      if (a.lse && valid)  // the row's softmax is 2^(s * scale - lse)
        a.lse[(size_t)(it.a0 + pos) * a.n_heads + head] = m + __log2f(l);
      __half* out = a.out + (size_t)(it.a0 + (valid ? pos : 0)) * a.n_heads * D + head * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(lane_base + o_col + c * 32, o);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_f16x2(o[8 * q + 0] * inv, o[8 * q + 1] * inv);
            u.y = pack_f16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            u.z = pack_f16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            u.w = pack_f16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            dst[q] = u;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&o_free[t]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
  if (threadIdx.x == 0) ring_leave(a.sched);
}

int heads_per_cta(int n_rep) {
  int h = 8;
  while (h > 1 && n_rep % h != 0) h >>= 1;
  return h;
}

template <int D, bool CACHED>
cudaError_t launch(const AttnArgs& a, int n_seq, int max_len, int sm_count,
                   cudaStream_t s) {
  using L = AttnLayout<D>;
  constexpr int AN = L::AN;
  const int BP = AM / a.hpc;
  CUtensorMap tq, tk, tv;
  if (!tc_encode_bf16(&tq, a.qkv, a.tokens, a.nqkv, BP)) return cudaErrorInvalidValue;
  if constexpr (CACHED) {
    const uint64_t rows = (uint64_t)n_seq * a.max_seq, cols = (uint64_t)a.n_kv_heads * D;
    if (!tc_encode_bf16(&tk, a.cache_k, rows, cols, AN) ||
        !tc_encode_bf16(&tv, a.cache_v, rows, cols, AN))
      return cudaErrorInvalidValue;
  } else {
    if (!tc_encode_bf16(&tk, a.qkv, a.tokens, a.nqkv, AN)) return cudaErrorInvalidValue;
    tv = tk;
  }
  const int n_qb = (max_len + 2 * BP - 1) / (2 * BP);
  const int n_hg = a.n_heads / a.hpc;
  const long long items = (long long)n_qb * n_hg * n_seq;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffff || !a.sched) return cudaErrorInvalidValue;
  auto kern = attn_tc_kernel<D, CACHED>;
  static std::atomic<uint64_t> attr_done{0};
  if (cudaError_t e = ensure_smem_attr(kern, (int)L::TOTAL, attr_done); e != cudaSuccess)
    return e;
  const int grid = (int)(items < sm_count ? items : sm_count);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), L::TOTAL, s, tq, tk, tv, a,
                    (int)items, n_hg, n_seq, n_qb);
}

}  // namespace

cudaError_t attn_prefill(const AttnArgs& args, int n_seq, int max_len,
                         int sm_count, cudaStream_t s) {
  AttnArgs a = args;
  const int n_rep = a.n_heads / a.n_kv_heads;
  a.hpc = heads_per_cta(n_rep);
  if (n_seq <= 0 || max_len <= 0 || a.tokens <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch<128, false>(a, n_seq, max_len, sm_count, s);
  if (a.head_dim == 64) return launch<64, false>(a, n_seq, max_len, sm_count, s);
  return cudaErrorInvalidValue;
}

cudaError_t attn_prefill_cached(const AttnArgs& args, int n_seq, int sm_count,
                                cudaStream_t s) {
  AttnArgs a = args;
  const int n_rep = a.n_heads / a.n_kv_heads;
  a.hpc = heads_per_cta(n_rep);
  a.cu = nullptr;
  if (n_seq <= 0 || a.seq_len <= 0 || a.tokens <= 0) return cudaSuccess;
  if (!a.cache_k || !a.cache_v || !a.start_pos) return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch<128, true>(a, n_seq, a.seq_len, sm_count, s);
  if (a.head_dim == 64) return launch<64, true>(a, n_seq, a.seq_len, sm_count, s);
  return cudaErrorInvalidValue;
}

}  // namespace llama
