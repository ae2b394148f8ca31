// Causal grouped-query attention for prefill, padded or packed varlen
// ("模型层" 9.3 CausalSelfAttention; "parallel_attention.py" 2 step 4 and 3
// flash_attn_varlen_func): o = softmax(q k^T / sqrt(d) + causal mask) v within
// each sequence, query head h reading kv head h / n_rep.  q and k arrive
// already rotated by the QKV GEMM epilogue.
//
// tcgen05 / TMEM flash attention, persistent (one CTA per SM), 10 warps:
//   warps 0..7  softmax + epilogue: query row r of the tile (TMEM lane r) is
//               shared by warp r / 32 (keys 0..63 of each S tile, the first
//               half of O) and warp 4 + r / 32 (keys 64..127, second half of
//               O); the two threads swap their partial row maxima through
//               shared memory.  Each thread masks its scores, keeps the
//               running max m and its partial sum l, writes its half of
//               P = 2^(s - m) as bf16 into a 128-byte swizzled smem tile (the
//               A operand of P V), and at the end reads its half of O,
//               divides by the row's l and stores bf16.
//   warp 8      TMA producer: the Q tile once per work item, K / V tiles of
//               128 keys into a ring of stages.
//   warp 9      one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//               S buffers, O += P V into the TMEM O buffer (V is read as an
//               MN-major operand straight from its TMA tile).
// A tile of 128 query rows holds `hpc` query heads of one kv group times
// 128 / hpc positions, so each K / V tile feeds every head of the group
// (repeat_kv is never materialised).  Rescaling of O is lazy: a row's
// reference max only moves (and O is rescaled in TMEM) when the new max
// exceeds it by more than 8 in the log2 domain, so P stays <= 2^8.
// Work items (query block, head group, sequence) run longest causal range
// first.  Every wait is bounded (2 s -> status bit, abort, drain, free TMEM).
#include <cuda_bf16.h>
#include <math.h>

#include "attn_prefill.cuh"
#include "common.cuh"
#include "gemm_tc.cuh"

namespace llama {
namespace {

using bf16 = __nv_bfloat16;
constexpr int AM = 128;  // query rows per tile (MMA M)
constexpr int AN = 128;  // keys per K / V tile
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct AttnLayout {
  static constexpr int ATOMS = D / 64;  // 128-byte swizzle atoms per row
  static constexpr uint32_t Q_BYTES = AM * D * 2;
  static constexpr uint32_t KV_BYTES = AN * D * 2;  // K or V tile
  static constexpr uint32_t P_BYTES = AM * AN * 2;
  static constexpr int STAGES = D == 64 ? 4 : 2;
  static constexpr uint32_t STAGE = 2 * KV_BYTES;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t P_OFF = Q_OFF + Q_BYTES;
  static constexpr uint32_t KV_OFF = P_OFF + P_BYTES;
  static constexpr uint32_t BAR_OFF = KV_OFF + STAGES * STAGE;
  static constexpr uint32_t RED_OFF = BAR_OFF + 256;  // [2][2][128] maxima, [2][128] sums
  static constexpr uint32_t TOTAL = RED_OFF + 6 * 128 * 4 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // S0 [0,128) S1 [128,256) O [256,256+D)
  static constexpr uint32_t O_COL = 256;
  static_assert(TOTAL <= 232448, "shared memory budget");
};

struct Item {
  int a0, L, q0, h0, g;  // sequence start and length, first position, heads
  int n_tiles;           // K / V tiles of the causal range (0: nothing to do)
};

// Work item i: query block from the top (longest causal range first), then
// head group, then sequence.
__device__ __forceinline__ Item get_item(const AttnArgs& a, int i, int n_hg,
                                         int n_seq, int n_qb, int BP) {
  Item it;
  const int per_qb = n_hg * n_seq;
  const int qb = n_qb - 1 - i / per_qb;
  const int rem = i - (i / per_qb) * per_qb;
  const int hg = rem % n_hg, s = rem / n_hg;
  const int n_rep = a.n_heads / a.n_kv_heads;
  it.h0 = hg * a.hpc;
  it.g = it.h0 / n_rep;
  it.q0 = qb * BP;
  if (a.cu) {
    const int s0 = a.cu[s], s1 = a.cu[s + 1];
    if (s0 < 0 || s1 < s0 || s1 > a.tokens) {  // flagged by the positions kernel
      it.a0 = 0; it.L = 0;
    } else {
      it.a0 = s0; it.L = s1 - s0;
    }
  } else {
    it.a0 = s * a.seq_len;
    it.L = a.seq_len;
  }
  const int hi = min(it.q0 + BP, it.L);
  it.n_tiles = it.q0 < it.L ? (hi + AN - 1) / AN : 0;
  return it;
}

constexpr int kSoftmaxThreads = 256;
constexpr int kThreads = kSoftmaxThreads + 64;
constexpr int kProducerWarp = 8, kMmaWarp = 9;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmKV, AttnArgs a,
                   int n_items, int n_hg, int n_seq, int n_qb) {
  using L = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bar;                     // [STAGES]
  uint64_t* kv_empty = kv_full + L::STAGES;    // [STAGES]
  uint64_t* s_full = kv_empty + L::STAGES;     // [2]
  uint64_t* s_free = s_full + 2;               // [2]
  uint64_t* q_full = s_free + 2;
  uint64_t* q_empty = q_full + 1;
  uint64_t* p_full = q_empty + 1;
  uint64_t* pv_done = p_full + 1;
  uint64_t* o_free = pv_done + 1;
  uint64_t* drain = o_free + 1;
  uint64_t* mx_bar = drain + 1;                // [2] row-max exchange
  uint64_t* l_bar = mx_bar + 2;                // row-sum exchange
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(l_bar + 1);
  float* red_max = reinterpret_cast<float*>(smem + L::RED_OFF);  // [2][2][128]
  float* red_l = red_max + 4 * 128;                               // [2][128]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int BP = AM / a.hpc;  // positions per tile
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kSoftmaxThreads);
      mbar_init(&mx_bar[b], kSoftmaxThreads);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(p_full, kSoftmaxThreads);
    mbar_init(pv_done, 1);
    mbar_init(o_free, kSoftmaxThreads);
    mbar_init(drain, 1);
    mbar_init(l_bar, kSoftmaxThreads);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmKV);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kvc = 0, k = 0, issued = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const Item it = get_item(a, i, n_hg, n_seq, n_qb, BP);
        if (it.n_tiles == 0) continue;
        if (k > 0 && !mbar_wait(q_empty, (k - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, L::Q_BYTES);
        for (int hh = 0; hh < a.hpc; ++hh)
          for (int at = 0; at < L::ATOMS; ++at)
            tma_load_2d(smem + L::Q_OFF + at * (AM * 128) + hh * BP * 128, &tmQ,
                        q_full, (it.h0 + hh) * D + at * 64, it.a0 + it.q0);
        ++issued;
        ++k;
        const int kcol = (a.n_heads + it.g) * D;
        const int vcol = (a.n_heads + a.n_kv_heads + it.g) * D;
        for (int j = 0; j < it.n_tiles; ++j, ++kvc) {
          const int st = kvc % L::STAGES;
          if (!mbar_wait(&kv_empty[st], ((kvc / L::STAGES) & 1) ^ 1, a.status,
                         abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* base = smem + L::KV_OFF + st * L::STAGE;
          mbar_arrive_expect_tx(&kv_full[st], L::STAGE);
          for (int at = 0; at < L::ATOMS; ++at) {
            tma_load_2d(base + at * (AN * 128), &tmKV, &kv_full[st], kcol + at * 64,
                        it.a0 + j * AN);
            tma_load_2d(base + L::KV_BYTES + at * (AN * 128), &tmKV, &kv_full[st],
                        vcol + at * 64, it.a0 + j * AN);
          }
          ++issued;
        }
      }
      (void)issued;
      if (!ok) {  // let the copies already issued land (bounded)
        volatile int own = 0;
        const uint32_t n = kvc < (uint32_t)L::STAGES ? kvc : (uint32_t)L::STAGES;
        for (uint32_t j = 1; j <= n; ++j) {
          const uint32_t idx = kvc - j;
          mbar_wait(&kv_full[idx % L::STAGES], (idx / L::STAGES) & 1, a.status, &own);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(AM, AN);
      constexpr uint32_t idesc_pv = idesc_bf16(AM, D) | (1u << 16);  // B MN-major
      const uint32_t q_addr = smem_u32(smem + L::Q_OFF);
      const uint32_t p_addr = smem_u32(smem + L::P_OFF);
      const uint32_t o_tmem = tmem_base + L::O_COL;
      uint32_t g = 0, kvc = 0, k = 0;
      bool ok = true, issued_any = false;
      auto pv = [&](uint32_t gi, uint32_t kvi, bool first) -> bool {
        if (!mbar_wait(p_full, gi & 1, a.status, abort_flag)) return false;
        if (first && k > 1 && !mbar_wait(o_free, (k - 2) & 1, a.status, abort_flag))
          return false;
        tc_fence_after();
        const int st = kvi % L::STAGES;
        const uint32_t v_addr =
            smem_u32(smem + L::KV_OFF + st * L::STAGE + L::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < AN / 16; ++kk) {
          const uint64_t ad = sdesc_k128(p_addr + (kk / 4) * (AM * 128) + (kk % 4) * 32);
          const uint64_t bd = sdesc_mn128(v_addr + kk * 2048, AN * 128);
          tc_mma_bf16(o_tmem, ad, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
        }
        tc_commit(pv_done);
        tc_commit(&kv_empty[st]);
        return true;
      };
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const Item it = get_item(a, i, n_hg, n_seq, n_qb, BP);
        if (it.n_tiles == 0) continue;
        if (!mbar_wait(q_full, k & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        ++k;
        for (int j = 0; j < it.n_tiles; ++j) {
          const int st = (kvc + j) % L::STAGES;
          const uint32_t sb = (g + j) & 1;
          if (!mbar_wait(&kv_full[st], ((kvc + j) / L::STAGES) & 1, a.status,
                         abort_flag) ||
              !mbar_wait(&s_free[sb], (((g + j) >> 1) & 1) ^ 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + L::KV_OFF + st * L::STAGE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (AM * 128) + (kk % 4) * 32;
            const uint32_t koff = (kk / 4) * (AN * 128) + (kk % 4) * 32;
            tc_mma_bf16(tmem_base + sb * AN, sdesc_k128(q_addr + off),
                        sdesc_k128(k_addr + koff), idesc_s, kk > 0 ? 1u : 0u);
          }
          issued_any = true;
          tc_commit(&s_full[sb]);
          if (j == it.n_tiles - 1) tc_commit(q_empty);
          if (j >= 1 && !pv(g + j - 1, kvc + j - 1, j == 1)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (!pv(g + it.n_tiles - 1, kvc + it.n_tiles - 1, it.n_tiles == 1)) {
          ok = false;
          break;
        }
        g += it.n_tiles;
        kvc += it.n_tiles;
      }
      if (!ok && issued_any) {  // wait for the MMAs in flight
        volatile int own = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, a.status, &own);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    constexpr int HN = AN / 2, HD = D / 2;  // this thread's keys / O columns
    uint8_t* prow = smem + L::P_OFF + half * (AM * 128) + r * 128;
    const float scale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e)/sqrt(d)
    uint32_t g = 0, k = 0;
    bool ok = true;
    auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(b, parity, a.status, abort_flag);
      return __shfl_sync(0xffffffffu, w_ok, 0) != 0;
    };
    // every lane acquires: the exchanged values were written by other warps
    auto all_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, a.status, abort_flag));
    };
    for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
      const Item it = get_item(a, i, n_hg, n_seq, n_qb, BP);
      if (it.n_tiles == 0) continue;
      ++k;
      const int pos = it.q0 + (r % BP);
      const int head = it.h0 + r / BP;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n_tiles; ++j, ++g) {
        const uint32_t sb = g & 1;
        if (!warp_wait(&s_full[sb], (g >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[HN];
#pragma unroll
        for (int c = 0; c < HN / 32; ++c)
          tmem_ld32(lane_base + sb * AN + half * HN + c * 32, s + c * 32);
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
        // causal mask (keys after the row's position), partial max of the
        // raw scores (8 independent chains)
        const int kb = j * AN + half * HN;
        if (kb + HN - 1 > it.q0) {
          const int lim = pos - kb;
#pragma unroll
          for (int c = 0; c < HN; ++c) s[c] = c > lim ? -INFINITY : s[c];
        }
        float pm[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pm[e] = s[e];
#pragma unroll
        for (int c = 8; c < HN; ++c) pm[c & 7] = fmaxf(pm[c & 7], s[c]);
        float hmax = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                           fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
        // swap partial maxima with the thread holding the row's other half
        float* rm = red_max + sb * 256;
        rm[half * 128 + r] = hmax;
        mbar_arrive(&mx_bar[sb]);
        if (!all_wait(&mx_bar[sb], (g >> 1) & 1)) {
          ok = false;
          break;
        }
        const float tmax = fmaxf(hmax, rm[(half ^ 1) * 128 + r]) * scale;
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
        // p = 2^(s * scale - m), 8 independent partial sums
        float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < HN; ++c) {
          s[c] = ex2(fmaf(s[c], scale, -mref));
          ps[c & 7] += s[c];
        }
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        // the P buffer and O are free once P V of the previous tile is done
        if (j > 0) {
          if (!warp_wait(pv_done, (g - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
              float o[32];
              const uint32_t t = lane_base + L::O_COL + half * HD + c * 32;
              tmem_ld32(t, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(t, o);
            }
          }
        }
        // this thread's 64 keys of P as bf16: one 128-byte swizzle atom row
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 u;
          u.x = pack_bf16x2(s[cc * 8 + 0], s[cc * 8 + 1]);
          u.y = pack_bf16x2(s[cc * 8 + 2], s[cc * 8 + 3]);
          u.z = pack_bf16x2(s[cc * 8 + 4], s[cc * 8 + 5]);
          u.w = pack_bf16x2(s[cc * 8 + 6], s[cc * 8 + 7]);
          *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) = u;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, rows inside the sequence only
      red_l[half * 128 + r] = l;
      mbar_arrive(l_bar);
      if (!all_wait(l_bar, (k - 1) & 1) || !warp_wait(pv_done, (g - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float lsum = l + red_l[(half ^ 1) * 128 + r];
      const bool valid = pos < it.L;
      const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
      bf16* out = a.out + (size_t)(it.a0 + (valid ? pos : 0)) * a.n_heads * D +
                  head * D + half * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(lane_base + L::O_COL + half * HD + c * 32, o);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_bf16x2(o[8 * q + 0] * inv, o[8 * q + 1] * inv);
            u.y = pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            u.z = pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            u.w = pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            dst[q] = u;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(o_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

int heads_per_cta(int n_rep) {
  int h = 8;
  while (h > 1 && n_rep % h != 0) h >>= 1;
  return h;
}

template <int D>
cudaError_t launch(const AttnArgs& a, int n_seq, int max_len, int sm_count,
                   cudaStream_t s) {
  using L = AttnLayout<D>;
  const int BP = AM / a.hpc;
  CUtensorMap tq, tkv;
  if (!tc_encode_bf16(&tq, a.qkv, a.tokens, a.nqkv, BP) ||
      !tc_encode_bf16(&tkv, a.qkv, a.tokens, a.nqkv, AN))
    return cudaErrorInvalidValue;
  const int n_qb = (max_len + BP - 1) / BP;
  const int n_hg = a.n_heads / a.hpc;
  const long long items = (long long)n_qb * n_hg * n_seq;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  auto kern = attn_tc_kernel<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = (int)(items < sm_count ? items : sm_count);
  kern<<<grid, kThreads, L::TOTAL, s>>>(tq, tkv, a, (int)items, n_hg, n_seq, n_qb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_prefill(const AttnArgs& args, int n_seq, int max_len,
                         int sm_count, cudaStream_t s) {
  AttnArgs a = args;
  const int n_rep = a.n_heads / a.n_kv_heads;
  a.hpc = heads_per_cta(n_rep);
  if (n_seq <= 0 || max_len <= 0 || a.tokens <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch<128>(a, n_seq, max_len, sm_count, s);
  if (a.head_dim == 64) return launch<64>(a, n_seq, max_len, sm_count, s);
  return cudaErrorInvalidValue;
}

}  // namespace llama
