// attn_tc.cuh -- bf16 / fp16 attention forward on the 5th-generation tensor cores (sm_103a).
//
// Computes, for every (batch, head) and query row i,
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j  and  LSE_i = ln sum_j exp(scale q_i.k_j)
// with the online-softmax tile loop of "Softmax 数值稳定性与 IO-Aware Attention：从在线
// 归一化到 FlashAttention", §七: per Q tile, m = -inf, l = 0, O = 0; for each K/V tile
// S = Q K^T, m_new = max(m, rowmax S), P = exp(S - m_new), alpha = exp(m - m_new),
// l = alpha l + rowsum P, O = alpha O + P V; finally O = O / l.  Alpha rescales both l
// and O.  The §八 work split is kept: Q is the outer loop (each O row is written once),
// and K/V tiles entirely above the causal diagonal are skipped, never loaded.
//
// GB300 mapping (not the pages' A100-era tiling):
//  * one CTA per SM holds TWO 128-row Q tiles that share one stream of K/V tiles;
//    the tensor pipe alternates between them, so the softmax of one tile overlaps
//    the two MMAs of the other ("ping-pong");
//  * S = Q K^T and O += P V are tcgen05.mma kind::f16 (bf16 or fp16 in, fp32
//    accumulate), issued by one elected thread of the MMA warp; S, P and O live in tensor memory (TMEM), never in HBM;
//  * Q, K, V tiles arrive by TMA into 128-byte-swizzled shared memory through a ring of
//    slots guarded by mbarriers; O leaves through shared memory and a TMA store;
//  * each softmax thread owns one query row of its tile (TMEM lane = row), so row max
//    and row sum need no shuffles;
//  * the rescale reference m is moved only when a row's maximum grows by more than
//    a factor 2^64 for bf16 (2^8 for fp16; kRescaleLog2); between moves alpha = 1 and
//    the O rescale is skipped.  The identity behind the merge rule holds for any common
//    reference, so O and LSE are the same in exact arithmetic; P then lies in
//    [0, 2^64] instead of [0, 1], which bf16 and fp32 represent with the same relative
//    precision.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace osfa {

constexpr int kBlockM = 128;        // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;        // keys per K/V tile
constexpr int kBoxCols = 64;        // bf16 per 128-byte swizzled row
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 128 bytes
// Warps 0-3: softmax of tile 0; 4-7: softmax of tile 1; 8: MMA issue; 9: TMA loads;
// 10-11 idle (they complete the third warpgroup so that it can hand its registers to
// the softmax warpgroups).
constexpr int kAttnThreads = 384;
constexpr int kRegsSoftmax = 208;  // per thread, softmax warpgroups
constexpr int kRegsIssue = 88;     // per thread, MMA / TMA warpgroup (384 x 168 = 256 x 208 + 128 x 88)
constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;
// Lazy rescale threshold in log2 units: P = 2^(s' - m) stays below 2^kRescaleLog2.  bf16
// holds any such P to the same relative precision (its range reaches 2^127), so the
// reference moves only for growth beyond 2^64 (sums of up to 2^17 such terms times |v|
// stay far inside fp32); fp16 P must stay below 65504, so 2^8 there.
template <bool F16>
constexpr float kRescaleLog2 = F16 ? 8.0f : 64.0f;

template <int D>
struct AttnTcCfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // 128 rows x D bf16
  static constexpr int kSlots = (D == 128) ? 5 : 8;       // K/V ring depth
  static constexpr bool kPairWait = (D == 64);  // one landing barrier per K/V pair
  static constexpr int kSmemQ0 = 0;
  static constexpr int kSmemQ1 = kTileBytes;
  static constexpr int kSmemSlots = 2 * kTileBytes;
  static constexpr int kSmemBars = kSmemSlots + kSlots * kTileBytes;
  static constexpr int kSmemBytes = kSmemBars + 512 + 1024;  // + barriers + alignment slack
  // TMEM columns.  d = 128: S/P of tile 0 and 1, then O of tile 0 and 1.  d = 64: the O
  // accumulators take only 128 columns, which leaves room for a third S/P buffer; the
  // two tiles then use three S/P buffers in rotation (kTripleS), so that the next S of a
  // tile can be computed while its current P is still being formed.
  static constexpr bool kTripleS = (D == 64);
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColS2 = 256;
  static constexpr uint32_t kColO0 = kTripleS ? 384 : 256, kColO1 = kColO0 + D;
  static constexpr uint32_t kTmemCols = 512;
};

struct AttnTcParams {
  float* lse;          // [BH, N] or nullptr
  unsigned* status;    // device status word
  int N;
  int BH;
  int nqb;             // number of 256-row query blocks per head
  int head_group;      // heads scheduled together (1 <= head_group <= BH)
  int causal;
  float scale_log2;    // scale * log2(e)
  // Split-KV: with splits > 1 block (q block, split) takes the split-th chunk of the
  // K/V tiles its query block needs and writes fp32 partials (O normalised by its own
  // l, and LSE) to ws_o [splits, BH, n_pad, d] and ws_lse [splits, BH, n_pad] instead
  // of O; splits == 1 is the plain forward.
  int splits;
  int n_pad;           // nqb * 256
  float* ws_o;
  float* ws_lse;
};

// F16 = false: bf16 Q, K, V, O (and P); F16 = true: fp16.
template <int D, bool F16>
cudaError_t launch_attn_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const AttnTcParams& p, cudaStream_t stream);

}  // namespace osfa
