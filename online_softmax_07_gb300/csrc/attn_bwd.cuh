// attn_bwd.cuh -- backward of the tcgen05 attention forward (sm_103a).
//
// "Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention" §7.2: the
// backward keeps only per-row statistics of the forward (here LSE) and recomputes the
// scores tile by tile instead of reading a stored probability matrix.  With
// P = exp(scale * Q K^T - LSE) recomputed per tile, the gradients of the exact
// attention function are
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D) with D_i = sum_c dO_ic O_ic,
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// GB300 mapping at d = 128, three launches (d = 64: see AttnBwd1Cfg below):
//  * bwd_prep: D_i and LSE_i * log2(e) for every query row into the caller's workspace
//    (rows past N get D = 0 and +inf, so that padded queries drop out of every sum);
//  * bwd_dkdv: one CTA per 128-key tile j keeps K_j, V_j in shared memory and dV_j, dK_j
//    in tensor memory while Q_i, dO_i stream through by TMA; per query tile it computes
//    S^T = K_j Q_i^T and dP^T = V_j dO_i^T (tcgen05, keys on TMEM lanes), the element-
//    wise warps turn them into P^T and dS^T (16-bit, stored back over S^T and dP^T in
//    TMEM), and dV += P^T dO_i, dK += dS^T Q_i take P^T and dS^T straight from TMEM;
//  * bwd_dq: one CTA per 128-query tile i keeps Q_i, dO_i and accumulates
//    dQ += dS K_j the same way while K_j, V_j stream.
// Splitting dQ into its own pass recomputes S and dP once more (7 tile products per
// tile pair instead of 5) but needs no atomic accumulation: every output element is
// written once, by one CTA, so the result is deterministic.  At d = 128 the key-outer
// pass fills all 512 TMEM columns (S^T, dP^T, dV, dK), leaving none for a dQ partial;
// at d = 64 there is room, and one pass does all (AttnBwd1Cfg).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "attn_tc.cuh"

namespace osfa {

// Warps 0-7: element-wise work, warp w on TMEM lanes 32 (w % 4) .. +31 and on the
// column half w / 4 of each tile; 8: MMA issue; 9: TMA loads; 10: in the one-pass kernel
// a second MMA-issuing warp (dK and dQ), else idle; 11 idle.
constexpr int kBwdThreads = 384;
constexpr int kBwdWarpMma = 8;
constexpr int kBwdWarpLoad = 9;
constexpr int kBwdWarpMma2 = 10;

// Two-pass backward (d = 128).
template <int D>
struct AttnBwdCfg {
  static_assert(D == 128, "the two-pass backward is for d = 128");
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // 128 rows x D, 16-bit
  static constexpr int kStages = 2;                       // streamed tile pairs in flight
  // A key-outer stage holds Q_i, dO_i and the query tile's statistics terms (128 rows x
  // 16 bf16, 32-byte swizzle), as in the one-pass kernel (AttnBwd1Cfg).
  static constexpr int kAugBytes = 128 * 32;
  static constexpr int kStageBytes = 2 * kTileBytes + kAugBytes;
  static constexpr int kSmemFixed0 = 0;           // resident tile 0 (K_j or Q_i)
  static constexpr int kSmemFixed1 = kTileBytes;  // resident tile 1 (V_j or dO_i)
  static constexpr int kSmemStages = 2 * kTileBytes;
  static constexpr int kSmemOnes = kSmemStages + kStages * kStageBytes;  // 2 x 4 KB
  static constexpr int kSmemBars = kSmemOnes + 2 * kAugBytes;
  static constexpr int kSmemBytes = kSmemBars + 512 + 1024;  // + barriers + alignment slack
  // TMEM columns: S (or S^T), dP (or dP^T), then one or two fp32 accumulators: all 512.
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  // Query-outer pass: K and V stream through separate rings, since K_j is held until
  // dQ += dS K_j (its last use) and V_j only until dP = dO V_j^T; K gets the deeper
  // ring, three slots, and V two, beside the resident Q_i, dO_i.
  static constexpr int kDqSlotsK = 3;
  static constexpr int kDqSlotsV = 2;
  static constexpr int kDqSmemK = kSmemStages;
  static constexpr int kDqSmemV = kDqSmemK + kDqSlotsK * kTileBytes;
  static constexpr int kDqSmemBars = kDqSmemV + kDqSlotsV * kTileBytes;
  static constexpr int kDqSmemBytes = kDqSmemBars + 512 + 1024;
};

// One-pass backward at d = 64 (the key-outer pass also forms dQ): each key-tile CTA
// computes, per query tile i, the partial dQ_i += dS_ij K_j with a fifth tile product
// (dS staged in shared memory, where dK += dS^T Q_i reads it too) into TMEM, and the
// element-wise warps
// add it into an fp32 dQ accumulator in the workspace by TMA reduce-adds (element-wise
// fp32 adds at L2), each warp its 32 x 32 share, during the next query tile (by then the
// partial is complete).  A finalize launch
// scales and rounds the accumulator into dQ.  This replaces the query-outer pass, which
// recomputes S, P, dP and dS once more; at d = 64 the element-wise work, not the tensor
// pipe, bounds both passes.  The accumulation order across CTAs varies, so dQ's fp32
// sums (and at times its last bit after rounding) vary from run to run; dK and dV stay
// deterministic.  Warp roles as in the two-pass kernels (a block of more than 384
// threads would be compiled with 128 registers a thread, too few for the element-wise
// warps), with warp 10 issuing dK and dQ beside the MMA warp.
//
// The row statistics enter through the tensor core instead of the element-wise warps:
// every query row carries bf16 terms of -LSE/scale and of -D (a high and a low part each,
// together exact to about 2^-18 of the value), and one more K = 16 step of S^T and of dP^T
// multiplies them by a constant tile of ones, so that TMEM receives S^T - LSE/scale and
// dP^T - D.  P = exp2(scale log2(e) (S - LSE/scale)) and dS = P (dP - D) then need no
// per-query value in the element-wise warps (each would be the same 64 values loaded by
// all 32 lanes of a warp).  The extra step is a bf16 product whatever the input type.

struct AttnBwd1Cfg {
  static constexpr int kBoxes = 1;
  static constexpr int kTileBytes = kBoxBytes;  // 128 rows x 64, 16-bit
  static constexpr int kStages = 3;
  // Statistics terms of a query tile: 128 rows x 16 bf16 (32 B, 32-byte swizzle):
  // [-LSE/scale high, low, -D high, low, 0 ...].
  static constexpr int kAugBytes = 128 * 32;
  static constexpr int kStageBytes = 2 * kTileBytes + kAugBytes;  // Q_i, dO_i, terms
  static constexpr int kSmemFixed0 = 0;           // K_j
  static constexpr int kSmemFixed1 = kTileBytes;  // V_j
  static constexpr int kSmemStages = 2 * kTileBytes;
  // The constant A operands of the statistics step, 128 rows x 16 bf16 each (32-byte
  // swizzle): rows [1, 1, 0, 0, 0, 0, 0, 0] (picks -LSE/scale) and [0, 0, 1, 1, 0, ...]
  // (picks -D), the same 8-element pattern in both 16-byte halves of a row, so that the
  // swizzle cannot move a one onto a term of the other statistic.
  static constexpr int kSmemOnes = kSmemStages + kStages * kStageBytes;
  // dS of the current tile pair, [key][query]: two 64-query boxes of 128 keys x 128 B,
  // 128-byte swizzle: the K-major A operand dS^T of dK += dS^T Q_i and the MN-major A
  // operand of dQ_i = dS K_j.
  static constexpr int kSmemDS = kSmemOnes + 2 * kAugBytes;
  // dQ staging: per element-wise warp one box of 32 rows x 32 fp32 (4 KB).
  static constexpr int kRedBoxBytes = 32 * 128;
  static constexpr int kSmemRed = kSmemDS + 2 * kTileBytes;
  static constexpr int kSmemBars = kSmemRed + 8 * kRedBoxBytes;
  static constexpr int kSmemBytes = kSmemBars + 512 + 1024;
  // TMEM: S^T, dP^T, dV, dK, P^T (16-bit, two queries a column: its own columns, so that
  // the next S^T may overwrite S^T as soon as the element-wise warps hold it in
  // registers; the next dP^T likewise, since dS goes to shared memory only) and the dQ
  // partial.
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 320;
  static constexpr uint32_t kColP = 384, kColDQ = 448;
  static constexpr uint32_t kTmemCols = 512;
};

struct AttnBwdParams {
  const float* lse2;   // query-outer pass: [BH, n_pad]: LSE * log2(e), +inf for rows >= N
  const float* dd;     // query-outer pass: [BH, n_pad]: D = rowsum(dO * O), 0 for rows >= N
  uint16_t* aug;       // key-outer passes: [BH, n_pad, 16] bf16 statistics terms, 0 for rows >= N
  float* dq_acc;       // one pass: [BH, n_pad, 64] fp32 dQ / scale accumulator
  void* dq;            // [BH, N, d] outputs, 16-bit
  void* dk;
  void* dv;
  unsigned* status;    // device status word
  int N;
  int BH;
  int nblk;            // ceil(N / 128)
  int n_pad;           // nblk * 128
  int head_group;      // heads scheduled together (1 <= head_group <= BH)
  int causal;
  float scale;
  float scale_log2;    // scale * log2(e)
};

// A second stream for the query-outer pass: it forks from the caller's stream after the
// prep launch and joins it again after the dQ pass, so that dQ blocks take the SMs the
// key-outer pass's causal tail leaves idle (both passes only read the prep's output and
// write disjoint gradients).  nullptr: all three launches on the caller's stream.
struct BwdFork {
  cudaStream_t side;
  cudaEvent_t fork, join;
};

// Workspace of the tensor-core backward, per padded query row: at d = 128 fp32
// LSE * log2(e) and D (8 bytes, for the query-outer pass) and then the 16 bf16 statistics
// terms (32 bytes, for the key-outer pass); at d = 64 the terms (32 bytes) and then the
// fp32 dQ accumulator row (256 bytes).  Each part covers all rows before the next.
inline long long bwd_tc_ws_bytes(long long BH, long long n_pad, int d) {
  return BH * n_pad * (d == 64 ? 32 + 64 * 4 : 2 * 4 + 32);
}

// tdq_acc: at d = 64 a TMA map of the dQ accumulator ([BH, n_pad, 64] fp32, boxes of
// 32 x 32, 128-byte swizzle; unused at d = 128); taug: a TMA map of the statistics terms
// ([BH, n_pad, 16] bf16, boxes of 128 rows, 32-byte swizzle).
template <int D, bool F16>
cudaError_t launch_attn_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq_acc,
                            const CUtensorMap& taug, const void* o,
                            const void* dout, const float* lse, float* ws, const AttnBwdParams& p,
                            cudaStream_t stream, const BwdFork* fork);

}  // namespace osfa
