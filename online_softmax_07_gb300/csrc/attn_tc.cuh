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
//    2^8 (kRescaleLog2); between moves alpha = 1 and the O rescale is skipped.  The
//    identity behind the merge rule holds for any common reference, so O and LSE are
//    the same in exact arithmetic; P then lies in [0, 2^8] instead of [0, 1], which
//    bf16 and fp32 represent with the same relative precision.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace osfa {

constexpr int kBlockM = 128;        // query rows per tile = TMEM lanes
constexpr int kDefaultBlockN = 128; // keys per K/V tile unless a block size is chosen
constexpr int kBoxCols = 64;        // bf16 per 128-byte swizzled row
constexpr int kBoxBytes = 128 * 128;  // one TMA box of a Q or O tile: 128 rows x 128 bytes
// Warps 0-3: softmax of tile 0; 4-7: softmax of tile 1; 8: MMA issue; 9: TMA loads;
// 10-11 idle (they complete the third warpgroup so that it can hand its registers to
// the softmax warpgroups).
constexpr int kAttnThreads = 384;
constexpr int kRegsSoftmax = 208;  // per thread, softmax warpgroups
constexpr int kRegsIssue = 88;     // per thread, MMA / TMA warpgroup (384 x 168 = 256 x 208 + 128 x 88)
constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;
// Lazy rescale threshold in log2 units: P = 2^(s' - m) stays below 2^kRescaleLog2.  The
// range of bf16 would allow far more, but a stale reference also costs accuracy: with
// the reference at the row maximum the largest term of a row is P = 1 exactly, with a
// stale one it is rounded to 16 bits like the rest, and on rows dominated by one key
// that rounding goes straight into O.  A 2^64 threshold (rescales almost never) raised
// the largest O error on a Q-std-4 set from 1.6e-2 to 2.7e-2 (kernel-arithmetic
// emulation against the fp64 oracle); 2^8 keeps it near that of an eager reference
// (1.5e-2) and keeps fp16 P below its 65504 limit.
template <bool F16>
constexpr float kRescaleLog2 = 8.0f;

// D: head dimension; BN: keys per K/V tile (the "block size" of the tile loop).  BN = 128
// is the kernel the library runs; BN = 64 (both d) and 192, 256 (d = 64) are built for
// the block-size study.
template <int D, int BN>
struct AttnTcCfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(BN == 64 || BN == 128 || ((BN == 192 || BN == 256) && D == 64), "key block");
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kQTileBytes = kBoxes * kBoxBytes;  // 128 query rows x D
  static constexpr int kKvBoxBytes = BN * 128;            // BN keys x 64 columns
  static constexpr int kTileBytes = kBoxes * kKvBoxBytes; // one K or V tile: BN keys x D
  // K/V ring depth: the slots that fit next to the two Q tiles in about 224 KB.
  static constexpr int kSlots =
      (D == 128) ? (BN == 64 ? 10 : 5) : (BN == 64 ? 16 : BN == 128 ? 8 : BN == 192 ? 8 : 6);
  // One landing barrier per K/V pair (d = 64 with three S buffers or one), else one per
  // slot (the two-buffer issue order of d = 128, also used by 192-key tiles).
  static constexpr bool kPairWait = (D == 64 && BN != 192);
  static constexpr int kSmemQ0 = 0;
  static constexpr int kSmemQ1 = kQTileBytes;
  static constexpr int kSmemSlots = 2 * kQTileBytes;
  static constexpr int kSmemBars = kSmemSlots + kSlots * kTileBytes;
  static constexpr int kSmemBytes = kSmemBars + 512 + 1024;  // + barriers + alignment slack
  // TMEM columns: kSBufs S/P buffers of BN columns, then O of tile 0 and 1.  d = 128:
  // two buffers (one per tile).  d = 64: the O accumulators take only 128 columns, which
  // leaves room for a third buffer, so that the next S of a tile can be computed while
  // its current P is still being formed; at BN = 192 two buffers fit (as at d = 128), at
  // BN = 256 one 256-column buffer is all that fits, and the two tiles take turns.
  static constexpr int kSBufs = (D == 128 || BN == 192) ? 2 : (BN == 256 ? 1 : 3);
  static constexpr uint32_t kColO0 = kSBufs * BN, kColO1 = kColO0 + D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColO1 + D <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
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

// F16 = false: bf16 Q, K, V, O (and P); F16 = true: fp16.  tk and tv have BN-row boxes,
// tq and to 128-row boxes.
template <int D, int BN, bool F16>
cudaError_t launch_attn_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const AttnTcParams& p, cudaStream_t stream);

}  // namespace osfa
