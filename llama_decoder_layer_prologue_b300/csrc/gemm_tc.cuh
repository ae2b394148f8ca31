// tcgen05 / TMEM GEMM fed by TMA: D = A[M, K] . B[N, K]^T, bf16 operands,
// fp32 accumulation in tensor memory, fused epilogues.  Host interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llama {

enum TcEpi : int {
  TC_STORE = 0,     // out = acc (bf16)
  TC_QKV = 1,       // out = r1[m] * acc (r1 = 1 without rowscale), RoPE on q / k
  TC_RESID_SS = 2,  // h = res (bf16) + acc: out = 16-bit(h * out_scale),
                    // ss_out[m * ss_np + s] = sum of h^2 over the row's
                    // columns of slot s (below)
  TC_SWIGLU = 3,    // gate|up interleaved by 128: out = silu(r2 g) * (r2 u)
  TC_RESID = 4,     // out = res_scale * res (fp16) + in_scale * acc (bf16)
  TC_PARTIAL = 5,   // stream-K fp32 partials: part[tile][slot][bn][128]
  // Backward-pass epilogues.  Their operands are not both K-major: TC_DW
  // multiplies two activations that share the token dimension (A and B
  // MN-major: A^T B over tokens), the others multiply an activation by a
  // weight read along its output dimension (B MN-major: D = A W).
  TC_DW = 6,        // fp32 out[src row][col] = in_scale * acc * colscale[col];
                    // dg[(m / 32) * N + col] = sum over the 32 rows m of a
                    // warp of w_orig[src row][col] * that value before
                    // colscale (src row: the gate/up interleave undone when
                    // inter > 0); the caller adds the row groups up
  TC_SWIGLU_BWD = 7,// acc = d act [T, I]; with gate / up from aux_in (fp16,
                    // packed gate|up order) and r2 = 1 / RMS(h) from ss_in
                    // (slots added as TC_SWIGLU does):
                    // out (fp16, packed order) = r2 * (d gate | d up) * out_scale
  TC_F32_DOT = 8,   // fp32 out = in_scale * acc; ss_out[m * ss_np + s] = sum
                    // over the row's columns of slot s of out * res_scale *
                    // residual (fp16, or bf16 if res_bf16)
  TC_DO = 9,        // fp16 out = in_scale * acc; aux_out[m * n_heads + head] =
                    // sum over the head's columns of fp16(out) * residual (fp16)
};

struct TcEpiArgs {
  void* out = nullptr;  // bf16 [M, ldo] (TC_SWIGLU: [M, N/2]); fp32 partials
  int ldo = 0;
  const void* residual = nullptr;  // TC_RESID_SS: bf16; TC_RESID: fp16 [M, ldo]
  const float* rowscale = nullptr; // r1 [M]
  // Row sums as fixed-order partials (so that a call's result does not
  // depend on the order in which tiles finish): slot 2 n + half holds the
  // sum over column half `half` of 256-column tile n; ss_np slots per row.
  const float* ss_in = nullptr;    // TC_SWIGLU / TC_SWIGLU_BWD: sums of h^2
  float* ss_out = nullptr;         // TC_RESID_SS, TC_F32_DOT
  int ss_np = 0;                   // slots per row: 2 * ceil(N / 256) of the
                                   // GEMM that wrote them
  float inv_h = 0.f, eps = 0.f;
  const int32_t* pos = nullptr;    // TC_QKV: position of every row
  const float* cos_t = nullptr;    // [max_pos, d/2]
  const float* sin_t = nullptr;
  int head_dim = 0, rope_cols = 0, max_pos = 0;  // rope on columns < rope_cols
  int part_slots = 0;              // TC_PARTIAL: slots per tile (plan.slots)
  int* status = nullptr;
  // operand / output types and power-of-two scales of the fp16 path
  int ab_f16 = 0;        // A and B are fp16 (else bf16)
  int out_f16 = 0;       // TC_QKV / TC_SWIGLU / TC_RESID_SS output is fp16
  float in_scale = 1.f;  // TC_SWIGLU: gate / up = in_scale * r2 * acc;
                         // TC_RESID: out = res_scale * res + in_scale * acc
  float res_scale = 1.f; // TC_RESID
  float out_scale = 1.f; // TC_SWIGLU: act stored * out_scale; TC_RESID_SS: h * out_scale
  int pdl = 0;           // launch with programmatic dependent launch
  int b_const = 1;       // B never depends on an earlier kernel (weights): its
                         // first K-slices may be loaded before the PDL wait
  // backward-pass epilogues
  const void* colscale = nullptr;  // TC_DW: bf16 [N] (null: 1)
  const void* w_orig = nullptr;    // TC_DW: bf16 [rows, ldo] for dg (null: no dg)
  float* dg = nullptr;             // TC_DW: fp32 [4 x (M-tiles run), N] row-group
                                   // sums (CTA pairs: M-tiles rounded up to even)
  int inter = 0;                   // TC_DW: undo the gate/up interleave of rows
  const void* aux_in = nullptr;    // TC_SWIGLU_BWD: fp16 gate|up [M, 2 N] (packed)
  void* aux_out = nullptr;         // TC_SWIGLU: fp16 gate|up [M, N] (packed), or
                                   // null; TC_DO: fp32 [M, n_heads]
  int res_bf16 = 0;                // TC_F32_DOT: the residual is bf16
  // Split tiles (whole-tile epilogues): when sk_part is set and the tiles do
  // not fill whole rounds of the grid, tc_gemm spreads the first
  // grid + (tiles % grid) tiles evenly over the CTAs by K-block.  A tile cut
  // between CTAs c and c + 1 is finished by c: c + 1 computes its K-blocks
  // first, stores the fp32 sums in sk_part[c + 1][128][bn] and sets
  // sk_flag[c + 1] = sk_epoch; c adds them in its epilogue and clears the
  // flag.  sk_part holds grid slots; sk_flag grid + 1 words, zero when no
  // launch is in flight; sk_epoch must be nonzero and differ from the
  // previous launch that used the same flags.  A GEMM with a split phase is
  // launched cooperatively, so every CTA that waits has its partner resident.
  float* sk_part = nullptr;
  uint32_t* sk_flag = nullptr;
  uint32_t sk_epoch = 0;
  int sk_tiles = 0;      // set by tc_gemm: tiles of the split phase
  int vec32 = 0;         // set by tc_gemm: out / residual rows are 32-byte aligned
  int group_m = 16;      // set by tc_gemm: M-tiles per band of the tile order
  // Run as CTA pairs (clusters of 2) on pairs of M-tiles sharing one N-tile,
  // B crossing from L2 once per pair.  1: each CTA loads half of every B
  // K-slice and multicasts it to both, and each runs its own M = 128 MMAs.
  // 2: each CTA loads only its half of B and the pair runs one M = 256 MMA
  // per K step (tcgen05 cta_group::2).  A K-major B map needs a box of
  // bn / 2 rows.  No split-tile phase.  Not for TC_PARTIAL or TC_STORE.
  int pair = 0;
};

// Encodes a 2-D bf16 tensor map over a row-major [rows, cols] matrix with a
// box of box_rows x 64 elements and the 128-byte swizzle.  false on failure.
bool tc_encode_bf16(CUtensorMap* map, const void* ptr, uint64_t rows,
                    uint64_t cols, uint32_t box_rows);

// Stream-K plan of a TC_PARTIAL GEMM: `grid` CTAs share the
// tiles * kb_total K-blocks evenly; tile t's partial sums land in
// tc_streamk_segments(plan, t) consecutive slots of part[t][slot][bn][128]
// (fp32, token-major: element [c][r] is output row 128 t + r, column c),
// slots <= plan.slots.
struct TcStreamK {
  int grid, tiles, kb_total, slots;
};
TcStreamK tc_streamk_plan(int M, int N, int K, int bn, int grid_limit);

__host__ __device__ inline int tc_streamk_segments(const TcStreamK& p, int t) {
  long long W = (long long)p.tiles * p.kb_total;
  long long g0 = (long long)t * p.kb_total, g1 = g0 + p.kb_total - 1;
  long long c0 = ((g0 + 1) * p.grid - 1) / W, c1 = ((g1 + 1) * p.grid - 1) / W;
  return (int)(c1 - c0 + 1);
}

// Launches the persistent GEMM.  TC_PARTIAL: bn in {64, 128, 256} (N <= bn
// tokens), stream-K over min(grid_limit, K-blocks) CTAs, ep.part_slots must
// equal tc_streamk_plan(...).slots.  Other epilogues: bn = 256, whole tiles
// over min(grid_limit, tiles) CTAs, with the split-tile phase when
// tc_split_tiles() is nonzero and ep.sk_part is set (K-major epilogues only).
// Operand maps: a K-major operand of R rows is tc_encode_bf16(map, ptr, R,
// K, box) over its [R, K] storage (box 128 for A, bn for B); an MN-major
// operand (TC_DW's A and B, the B of TC_SWIGLU_BWD / TC_F32_DOT / TC_DO) is
// stored [K, R] and takes tc_encode_bf16(map, ptr, K, R, 64).
cudaError_t tc_gemm(int epi, int bn, const CUtensorMap& ta,
                    const CUtensorMap& tb, int M, int N, int K,
                    const TcEpiArgs& ep, int grid_limit, cudaStream_t s);

// Reads and clears the status word that GEMMs launched without a status
// pointer of their own write (bounded waits that ran out), on the current
// device.  Synchronous with respect to the device (a plain memcpy).
cudaError_t tc_take_status(int* word);

// M-tiles per band of a whole-tile GEMM's tile order (tiles are visited band
// by band, all N-tiles of a band in turn).
int tc_group_m(int M, int N, int K);

// Tiles of the split phase for a whole-tile GEMM of `tiles` tiles of
// kb_total K-blocks on `grid` CTAs: grid + tiles % grid when the last round
// of plain tile rounds would leave more than 3 % of the rounds' time idle
// and a tile has at least 64 K-blocks, else 0.
int tc_split_tiles(int tiles, int grid, int kb_total);

}  // namespace llama
