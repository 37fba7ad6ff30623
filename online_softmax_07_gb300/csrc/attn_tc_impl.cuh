// attn_tc_impl.cuh -- kernel body of the tcgen05 attention forward (see attn_tc.cuh).
// Included by one translation unit per head dimension.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "attn_tc.cuh"

namespace osfa {

// K/V pairs tracked at once (kv_full / kv_empty barriers in pair mode); more than the
// ring holds.  Per-slot mode uses kv_full[slot] for up to kKvFullBars slots.
constexpr int kKvBars = 8;
constexpr int kKvFullBars = 16;

struct AttnTcBarriers {
  uint64_t q_full;       // TMA -> MMA: Q tile 0 is in shared memory
  uint64_t q1_full;      // ... Q tile 1 (loaded after the first K tile, which S_0(0) needs)
  // s_full and p_ready come in pairs per tile, used alternately: S_t(j) completes on
  // s_full[2 t + (j & 1)] and is waited with parity (j >> 1) & 1, P_t(j) likewise on
  // p_ready.  With three S buffers the MMA warp issues S_t(j+1) before it needs P_t(j),
  // so two S_t completions can be pending at once; on a single barrier the second would
  // hide the first from a parity wait if the softmax warps fell behind.  On alternating
  // barriers neither side can get two phases ahead of the other.
  uint64_t s_full[4];    // MMA -> softmax t: S_t of a K/V tile is in TMEM
  uint64_t p_ready[4];   // softmax t -> MMA: P_t stored in TMEM and O_t rescaled
  uint64_t o_final[2];   // MMA -> softmax t: last P_t V product done
  uint64_t pv_done[2];   // MMA -> softmax 1: P_1(n1 - 2) V done (three-buffer mode, once)
  uint64_t mma_drain;    // MMA thread: all of its MMAs finished (before TMEM is freed)
  // Landing of the K/V loads.  d = 64 (kPairWait): K_j and V_j both land on
  // kv_full[j % 8], so one wait covers the pair.  d = 128: each ring slot has its own
  // full barrier (kv_full[slot]): the MMA warp waits for K_{j+1} without waiting for
  // V_{j+1}, which an odd-sized ring may load a tile later.  Each ring slot is released on
  // its own (slot_empty) when the products reading it are done, except with kPairWait,
  // where the ring is deep enough to release both slots of pair j once, after the last
  // product reading the pair (kv_empty[j % 8]).
  uint64_t kv_full[kKvFullBars];
  uint64_t slot_empty[kKvFullBars];
  uint64_t kv_empty[8];  // kPairWait: both slots of pair j released at once
  uint32_t tmem_base;
  int abort;
};

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (tcgen05 "matrix
// descriptor"): start address, leading and stride byte offsets (all >> 4), the
// descriptor version 1 at bit 46 and the swizzle mode (2 = 128 B) at bits 61-63.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 (format 1) or
// both fp16 (format 0), A K-major, B K-major or MN-major, N >> 3 at bit 17, M >> 4 at
// bit 24.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool b_mn_major, bool f16) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Two fp32 to the kernel's 16-bit element type (round to nearest even), `lo` in bits 0..15.
template <bool F16>
__device__ __forceinline__ uint32_t pack_elem2(float lo, float hi) {
  if constexpr (F16) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  } else {
    return pack_bf16x2(lo, hi);
  }
}

template <int D, int BN, bool F16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const AttnTcParams p) {
  using Cfg = AttnTcCfg<D, BN>;
  constexpr int NS = Cfg::kSBufs;
  static_assert(Cfg::kSlots <= kKvFullBars, "a landing / release barrier per ring slot");
  static_assert(!Cfg::kPairWait || Cfg::kSlots / 2 <= kKvBars, "pairs in flight within kKvBars");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  AttnTcBarriers* bars = reinterpret_cast<AttnTcBarriers*>(smem + Cfg::kSmemBars);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item.  Heads are taken in groups of p.head_group (sized on the host so that
  // the group's K and V fit in L2); inside a group, the heavy (late) query blocks of
  // all its heads come first, so that causal tails overlap lighter work.
  int bh, qb;
  const int split = blockIdx.x % p.splits;
  {
    const int L = blockIdx.x / p.splits;
    const int per_group = p.head_group * p.nqb;
    const int full = p.BH / p.head_group;
    const int g = L / per_group;
    if (g < full) {
      const int r = L - g * per_group;
      qb = p.nqb - 1 - r / p.head_group;
      bh = g * p.head_group + r % p.head_group;
    } else {
      const int rem = p.BH - full * p.head_group;
      const int r = L - full * per_group;
      qb = p.nqb - 1 - r / rem;
      bh = full * p.head_group + r % rem;
    }
  }
  const int nblk = (p.N + BN - 1) / BN;
  // K/V tiles each Q tile needs: all of them, or up to its diagonal tile (causal).
  const int nb0 = p.causal ? min(nblk, (qb * 2 * kBlockM + kBlockM - 1) / BN + 1) : nblk;
  const int nb1 = p.causal ? min(nblk, (qb * 2 * kBlockM + 2 * kBlockM - 1) / BN + 1) : nblk;
  // This block's K/V tiles: all of them, or (split-KV) the split-th chunk of the tiles
  // tile 1 needs; tile 0 takes the part of the chunk below its own limit.  Tiles are
  // numbered from jlo; n0, n1 count them (n0 may be 0, and with splits > 1 so may n1).
  const int chunk = (nb1 + p.splits - 1) / p.splits;
  const int jlo = split * chunk;
  const int n1 = max(0, min(nb1, jlo + chunk) - jlo);
  const int n0 = max(0, min(nb0, jlo + chunk) - jlo);
  const bool split_mode = p.splits > 1;
  // Split mode: the combine kernel that follows may be scheduled once every block of this
  // grid has started (it waits for the grid's completion before reading the partials).
  if (split_mode) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  auto part_row = [&](int r) {  // index of query row r of this head in the partials
    return (static_cast<int64_t>(split) * p.BH + bh) * p.n_pad + r;
  };
  if (n1 == 0) {
    // Nothing to do for this split: the empty partial (LSE = -inf, O = 0) for its rows.
    for (int rr = threadIdx.x; rr < 2 * kBlockM; rr += blockDim.x) {
      const int64_t pr = part_row(qb * 2 * kBlockM + rr);
      p.ws_lse[pr] = -INFINITY;
      float4* orow = reinterpret_cast<float4*>(p.ws_o + pr * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q1_full), 1);
    for (int t = 0; t < 2; ++t) {
      for (int u = 0; u < 2; ++u) {
        mbar_init(smem_u32(&bars->s_full[2 * t + u]), 1);
        mbar_init(smem_u32(&bars->p_ready[2 * t + u]), 4);  // one arrival per softmax warp
      }
      mbar_init(smem_u32(&bars->o_final[t]), 1);
      mbar_init(smem_u32(&bars->pv_done[t]), 1);
    }
    mbar_init(smem_u32(&bars->mma_drain), 1);
    // Every landing barrier either mode may use: kv_full[j % kKvBars] for pairs,
    // kv_full[slot] per slot (up to kSlots of them).
    for (int u = 0; u < kKvFullBars; ++u) mbar_init(smem_u32(&bars->kv_full[u]), 1);
    for (int u = 0; u < kKvBars; ++u) mbar_init(smem_u32(&bars->kv_empty[u]), 1);
    for (int s = 0; s < Cfg::kSlots; ++s) mbar_init(smem_u32(&bars->slot_empty[s]), 1);
    bars->abort = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  volatile int* abort = &bars->abort;

  if (warp >= 8) {
    // One setmaxnreg for the whole issue warpgroup (warps 8-11).
    regs_decrease<kRegsIssue>();
  }
  if (warp >= 10) {
    // idle warps of the issue warpgroup
  } else if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      // Q_0, the first K (and V) tile, then Q_1: the first S product needs only Q_0 and
      // K_0.
      const uint32_t qbar = smem_u32(&bars->q_full);
      const uint32_t q1bar = smem_u32(&bars->q1_full);
      auto load_q = [&](int t, uint32_t bar) {
        mbar_arrive_expect_tx(bar, Cfg::kQTileBytes);
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_load_3d(sbase + (t ? Cfg::kSmemQ1 : Cfg::kSmemQ0) + b * kBoxBytes, &tm_q, bar,
                      b * kBoxCols, qb * 2 * kBlockM + t * kBlockM, bh);
      };
      load_q(0, qbar);
      bool q1_issued = false;
      int no_abort = 0;
      if constexpr (Cfg::kPairWait) {
        // Pair j: K_j into ring slot 2j % kSlots and V_j into the next slot, both landing
        // on kv_full[j % kKvBars], once pair j - kSlots / 2 (the previous occupant of both
        // slots) has been released.
        static_assert(Cfg::kSlots % 2 == 0, "pairs of slots");
        int issued = 0;
        for (int j = 0; j < n1; ++j) {
          const int jp = j - Cfg::kSlots / 2;
          if (jp >= 0 && !mbar_wait(smem_u32(&bars->kv_empty[jp % kKvBars]), (jp / kKvBars) & 1,
                                    abort, p.status))
            break;
          const uint32_t full = smem_u32(&bars->kv_full[j % kKvBars]);
          mbar_arrive_expect_tx(full, 2 * Cfg::kTileBytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t dst =
                sbase + Cfg::kSmemSlots + ((2 * j + h) % Cfg::kSlots) * Cfg::kTileBytes;
#pragma unroll
            for (int b = 0; b < Cfg::kBoxes; ++b)
              tma_load_3d(dst + b * Cfg::kKvBoxBytes, h ? &tm_v : &tm_k, full, b * kBoxCols,
                          (jlo + j) * BN, bh);
          }
          issued = j + 1;
          if (!q1_issued) {
            load_q(1, q1bar);
            q1_issued = true;
          }
        }
        // Every issued copy must land before the block's shared memory goes away: the
        // pairs not yet known to be released (the ring holds fewer than kKvBars pairs).
        if (!q1_issued) load_q(1, q1bar);  // (no pair issued: Q_1 still completes its barrier)
        mbar_wait(qbar, 0, &no_abort, p.status);
        mbar_wait(q1bar, 0, &no_abort, p.status);
        for (int j = max(0, issued - kKvBars); j < issued; ++j)
          mbar_wait(smem_u32(&bars->kv_full[j % kKvBars]), (j / kKvBars) & 1, &no_abort, p.status);
      } else {
        // Load it: K_j at it = 2j, V_j at 2j + 1, into ring slot it % kSlots once the
        // slot's previous load has been consumed; load it completes kv_full[slot].
        int issued = 0;
        const int nload = 2 * n1;  // K_j, V_j for j < n1 (tile 1 needs the most)
        for (int it = 0; it < nload; ++it) {
          const int slot = it % Cfg::kSlots;
          const int phase = (it / Cfg::kSlots) & 1;
          if (!mbar_wait(smem_u32(&bars->slot_empty[slot]), phase ^ 1, abort, p.status)) break;
          const uint32_t full = smem_u32(&bars->kv_full[slot]);
          mbar_arrive_expect_tx(full, Cfg::kTileBytes);
          const CUtensorMap* tm = (it & 1) ? &tm_v : &tm_k;
          const uint32_t dst = sbase + Cfg::kSmemSlots + slot * Cfg::kTileBytes;
#pragma unroll
          for (int b = 0; b < Cfg::kBoxes; ++b)
            tma_load_3d(dst + b * Cfg::kKvBoxBytes, tm, full, b * kBoxCols, (jlo + (it >> 1)) * BN,
                        bh);
          issued = it + 1;
          if (!q1_issued) {
            load_q(1, q1bar);
            q1_issued = true;
          }
        }
        // Every issued copy must land before the block's shared memory goes away: the
        // last load issued into each slot.
        if (!q1_issued) load_q(1, q1bar);  // (no load issued: Q_1 still completes its barrier)
        mbar_wait(qbar, 0, &no_abort, p.status);
        mbar_wait(q1bar, 0, &no_abort, p.status);
        for (int it = max(0, issued - Cfg::kSlots); it < issued; ++it)
          mbar_wait(smem_u32(&bars->kv_full[it % Cfg::kSlots]), (it / Cfg::kSlots) & 1, &no_abort,
                    p.status);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop with warp-uniform values; elect.sync inside the
    // MMA and commit wrappers lets one lane issue each instruction.
    constexpr uint32_t kIdescS = idesc_f16kind(kBlockM, BN, false, F16);
    constexpr uint32_t kIdescPV = idesc_f16kind(kBlockM, D, true, F16);
    // Descriptors of the tile bases; an operand at byte offset `off` inside a tile is
    // base + (off >> 4) (the start-address field never overflows: shared memory is
    // below 256 KB).
    const uint64_t dQ0 = desc_sw128(sbase + Cfg::kSmemQ0, 16, 1024);
    const uint64_t dQ1 = desc_sw128(sbase + Cfg::kSmemQ1, 16, 1024);
    const uint64_t dSlot0K = desc_sw128(sbase + Cfg::kSmemSlots, 16, 1024);
    const uint64_t dSlot0V = desc_sw128(sbase + Cfg::kSmemSlots, Cfg::kKvBoxBytes, 1024);
    const uint32_t tS0 = tbase, tS1 = tbase + BN;  // two-buffer mode
    const uint32_t tO0 = tbase + Cfg::kColO0, tO1 = tbase + Cfg::kColO1;
    auto slot_off16 = [](int it) {
      return static_cast<uint64_t>(((it % Cfg::kSlots) * Cfg::kTileBytes) >> 4);
    };
    // K_j and V_j have landed (kPairWait).
    auto wait_kv = [&](int j) {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->kv_full[j % kKvBars]),
                                               (j / kKvBars) & 1, abort, p.status));
    };
    // Load `it` of the ring has landed (per-slot barriers).
    auto wait_full = [&](int it) {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->kv_full[it % Cfg::kSlots]),
                                               (it / Cfg::kSlots) & 1, abort, p.status));
    };
    // S_t = Q_t K^T: K-major A and B, 16 columns (32 bytes) of d per instruction, all
    // issued under one elect; columns 64.. of d lie in the second box of each tile.
    auto issue_s = [&](uint32_t tS, uint64_t dQ, int itK) {
      const uint64_t dK = dSlot0K + slot_off16(itK);
      uint64_t a[D / 16], b[D / 16];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        a[kk] = dQ + (((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
        b[kk] = dK + (((kk >> 2) * Cfg::kKvBoxBytes + (kk & 3) * 32) >> 4);
      }
      if constexpr (D == 64) mma_ss4_elect(tS, a, b, kIdescS, 0u);
      else mma_ss8_elect(tS, a, b, kIdescS, 0u);
    };
    // O_t += P_t V: P from TMEM (bf16 packed two per column), V MN-major in shared
    // memory; 16 keys (2 KB of the V tile) per instruction, all under one elect.
    auto issue_pv = [&](uint32_t tO, uint32_t tP, int itV, bool acc) {
      const uint64_t dV = dSlot0V + slot_off16(itV);
      uint32_t a[BN / 16];
      uint64_t b[BN / 16];
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        a[kk] = tP + kk * 8;
        b[kk] = dV + ((kk * 2048) >> 4);
      }
      if constexpr (BN == 64) mma_ts4_elect(tO, a, b, kIdescPV, acc ? 1u : 0u);
      else if constexpr (BN == 128) mma_ts8_elect(tO, a, b, kIdescPV, acc ? 1u : 0u);
      else if constexpr (BN == 192) {
        mma_ts8_elect(tO, a, b, kIdescPV, acc ? 1u : 0u);
        mma_ts4_elect(tO, a + 8, b + 8, kIdescPV, 1u);
      }
      else mma_ts16_elect(tO, a, b, kIdescPV, acc ? 1u : 0u);
    };

    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_full), 0, abort, p.status));
    if constexpr (Cfg::kPairWait) ok = ok && wait_kv(0);
    else ok = ok && wait_full(0);
    // Q_1 lands after Q_0 and the first K/V tile: waited for once, before the first S_1.
    bool q1_ready = false;
    auto wait_q1 = [&]() {
      if (!q1_ready) {
        q1_ready = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q1_full), 0, abort, p.status));
        if (q1_ready) tc_fence_after();
      }
      return q1_ready;
    };
    if constexpr (NS == 1) {
      // One S/P buffer (BN = 256 at d = 64): the tiles take turns.  The S at position q
      // of the sequence S_0(0), S_1(0), S_0(1), ... (S_1(j) at min(j+1, n0) + j once tile 0
      // has run out) overwrites the P of position q - 1, so it is issued right after that
      // P V: S(0), P(0) V, S(1), P(1) V, ...
      const int npos = n0 + n1;
      auto pos_tile = [&](int q) { return q < 2 * n0 ? (q & 1) : 1; };
      auto pos_j = [&](int q) { return q < 2 * n0 ? (q >> 1) : q - n0; };
      if (ok) {
        tc_fence_after();
        const int t0 = pos_tile(0);
        if (t0 == 0 || (ok = wait_q1())) {
          issue_s(tbase, t0 ? dQ1 : dQ0, 0);
          mma_commit_elect(smem_u32(&bars->s_full[2 * t0]));
        }
      }
      for (int q = 0; ok && q < npos; ++q) {
        const int t = pos_tile(q), j = pos_j(q);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->p_ready[2 * t + (j & 1)]),
                                                     (j >> 1) & 1, abort, p.status))))
          break;
        tc_fence_after();
        issue_pv(tbase + (t ? Cfg::kColO1 : Cfg::kColO0), tbase, 2 * j + 1, j > 0);
        if (j + 1 == (t ? n1 : n0)) mma_commit_elect(smem_u32(&bars->o_final[t]));
        // P_1(j) V is the last product reading K_j or V_j.
        if (t == 1) mma_commit_elect(smem_u32(&bars->kv_empty[j % kKvBars]));
        if (q + 1 < npos) {
          const int tn = pos_tile(q + 1), jn = pos_j(q + 1);
          if (jn > j) {
            if (!(ok = wait_kv(jn))) break;
            tc_fence_after();
          }
          if (tn == 1 && !(ok = wait_q1())) break;
          issue_s(tbase, tn ? dQ1 : dQ0, 2 * jn);
          mma_commit_elect(smem_u32(&bars->s_full[2 * tn + (jn & 1)]));
        }
      }
    } else if constexpr (NS == 3) {
      // Three S/P buffers in rotation: the S issued at position pos of the sequence
      // S_0(0), S_1(0), S_0(1), S_1(1), ... (S_0(j) at 2j, S_1(j) at min(j+1, n0) + j once
      // tile 0 has run out) goes to buffer pos % 3.  Per K/V tile j the pipe receives
      // S_0(j+1), P_0(j) V, S_1(j+1), P_1(j) V: the next S of a tile is computed while its
      // softmax still works on the current one.  The buffer an S overwrites last held the
      // S three positions earlier, whose P V was issued before (in-order pipe).
      auto colS = [&](int pos) { return tbase + static_cast<uint32_t>((pos % 3) * BN); };
      auto wait_bar = [&](uint64_t* bar, int parity) {
        const bool r = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, abort, p.status));
        if (r) tc_fence_after();
        return r;
      };
      if (ok) {
        tc_fence_after();
        if (n0 > 0) {
          issue_s(colS(0), dQ0, 0);
          mma_commit_elect(smem_u32(&bars->s_full[0]));
        }
        if ((ok = wait_q1())) {
          issue_s(colS(n0 > 0 ? 1 : 0), dQ1, 0);
          mma_commit_elect(smem_u32(&bars->s_full[2]));
        }
      }
      for (int j = 0; ok && j < n1; ++j) {
        const int itV = 2 * j + 1, itK = 2 * j + 2;
        // K_{j+1} (and V_{j+1}); V_j landed with K_j.
        if (j + 1 < n1) {
          if (!(ok = wait_kv(j + 1))) break;
          tc_fence_after();
        }
        if (j < n0) {
          if (j + 1 < n0) {
            issue_s(colS(2 * j + 2), dQ0, itK);
            mma_commit_elect(smem_u32(&bars->s_full[(j + 1) & 1]));
          }
          if (!(ok = wait_bar(&bars->p_ready[j & 1], (j >> 1) & 1))) break;
          issue_pv(tO0, colS(2 * j), itV, j > 0);
          if (j + 1 == n0) mma_commit_elect(smem_u32(&bars->o_final[0]));
        }
        if (j + 1 < n1) {
          issue_s(colS(min(j + 2, n0) + j + 1), dQ1, itK);
          mma_commit_elect(smem_u32(&bars->s_full[2 + ((j + 1) & 1)]));
        }
        if (!(ok = wait_bar(&bars->p_ready[2 + (j & 1)], (j >> 1) & 1))) break;
        issue_pv(tO1, colS(min(j + 1, n0) + j), itV, j > 0);
        // The one P_1 V that no later product of this thread follows before tile 1's next
        // step (see the softmax's rescale wait).
        if (j + 2 == n1 && j + 1 >= n0) mma_commit_elect(smem_u32(&bars->pv_done[1]));
        // P_1(j) V is the last product reading K_j or V_j.
        mma_commit_elect(smem_u32(&bars->kv_empty[j % kKvBars]));
        if (j + 1 == n1) mma_commit_elect(smem_u32(&bars->o_final[1]));
      }
    } else {
      if (ok) {
        tc_fence_after();
        if (n0 > 0) {
          issue_s(tS0, dQ0, 0);
          mma_commit_elect(smem_u32(&bars->s_full[0]));
        }
        if ((ok = wait_q1())) {
          issue_s(tS1, dQ1, 0);
          mma_commit_elect(smem_u32(&bars->s_full[2]));
          mma_commit_elect(smem_u32(&bars->slot_empty[0]));
        }
      }
      for (int j = 0; ok && j < n1; ++j) {
        const int itV = 2 * j + 1, itK = 2 * j + 2;
        if (!(ok = wait_full(itV))) break;
        bool k_ready = false;
        if (j < n0) {
          if (!(ok = __all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&bars->p_ready[j & 1]), (j >> 1) & 1, abort,
                                          p.status))))
            break;
          tc_fence_after();
          issue_pv(tO0, tS0, itV, j > 0);
          if (j + 1 < n0) {
            if (!(ok = wait_full(itK))) break;
            k_ready = true;
            tc_fence_after();
            issue_s(tS0, dQ0, itK);
            mma_commit_elect(smem_u32(&bars->s_full[(j + 1) & 1]));
          } else {
            mma_commit_elect(smem_u32(&bars->o_final[0]));
          }
        }
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&bars->p_ready[2 + (j & 1)]), (j >> 1) & 1,
                                        abort, p.status))))
          break;
        tc_fence_after();
        issue_pv(tO1, tS1, itV, j > 0);
        mma_commit_elect(smem_u32(&bars->slot_empty[itV % Cfg::kSlots]));
        if (j + 1 < n1) {
          if (!k_ready) {
            if (!(ok = wait_full(itK))) break;
            tc_fence_after();
          }
          issue_s(tS1, dQ1, itK);
          mma_commit_elect(smem_u32(&bars->s_full[2 + ((j + 1) & 1)]));
          mma_commit_elect(smem_u32(&bars->slot_empty[itK % Cfg::kSlots]));
        } else {
          mma_commit_elect(smem_u32(&bars->o_final[1]));
        }
      }
    }
    // Drain: nothing may still read shared memory or TMEM when the block exits.
    mma_commit_elect(smem_u32(&bars->mma_drain));
    int no_abort = 0;
    mbar_wait(smem_u32(&bars->mma_drain), 0, &no_abort, p.status);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax tile t
    regs_increase<kRegsSoftmax>();
    const int t = warp >> 2;       // warps 0-3 -> tile 0, 4-7 -> tile 1
    const int wq = warp & 3;       // TMEM lane quarter this warp may access
    const int rr = wq * 32 + lane; // row within the tile
    const int r0 = qb * 2 * kBlockM + t * kBlockM;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tbase + lane_off + (t ? Cfg::kColO1 : Cfg::kColO0);
    const float sl2 = p.scale_log2;
    float m2 = -INFINITY;  // rescale reference, log2 units of the scaled score
    float l = 0.f;
    bool ok = true;

    const int nbt = t ? n1 : n0;
    for (int j = 0; j < nbt; ++j) {
      ok = mbar_wait(smem_u32(&bars->s_full[2 * t + (j & 1)]), (j >> 1) & 1, abort, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // Where S_t(j) is: two buffers, one per tile; three buffers in rotation, S_t(j) in
      // buffer (its position in the sequence S_0(0), S_1(0), S_0(1), ...) % 3; one buffer
      // shared by both tiles.
      const int pos = t ? min(j + 1, n0) + j : 2 * j;
      const int buf = NS == 2 ? t : (NS == 3 ? pos % 3 : 0);
      const uint32_t tS = tbase + lane_off + static_cast<uint32_t>(buf * BN);

      // Keys >= N (ragged last tile) and, on the diagonal tile, keys > row are masked.
      // (The condition is the same for the whole warp.)
      const int key0 = (jlo + j) * BN;
      const bool masked = (p.causal && (key0 + BN - 1 > r0)) || key0 + BN > p.N;
      int lim = p.N - 1 - key0;
      if (p.causal) lim = min(lim, r0 + rr - key0);
      // Loads columns c0 .. c0 + W - 1 of S_t(j) (W = 64 or 128) with their maximum from
      // the TMEM load's reduction; on a masked tile the masked keys become -inf and the
      // maximum is taken again over the kept ones (four chains of three-input max).
      auto load_chunk = [&](int c0, auto width, uint32_t* sr) -> float {
        constexpr int W = decltype(width)::value;
        float mxl;
        if constexpr (W == 128) tmem_ld128_max_wait(tS + c0, sr, mxl);
        else tmem_ld64_max_wait(tS + c0, sr, mxl);
        if (masked) {
          float* sv = reinterpret_cast<float*>(sr);
#pragma unroll
          for (int c = 0; c < W; ++c) sv[c] = (c0 + c <= lim) ? sv[c] : -INFINITY;
          float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
          for (int c = 4; c < W; c += 2) mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], sv[c], sv[c + 1]);
          mxl = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
        }
        return mxl;
      };
      constexpr int kChunk = BN < 128 ? BN : 128;   // columns held in registers at once
      using ChunkW = std::integral_constant<int, kChunk>;
      uint32_t sr[kChunk];
      float* s = reinterpret_cast<float*>(sr);
      float rowmax;
      if constexpr (BN == 256) {
        // Two 128-column halves: the upper half for its maximum only, then the lower
        // half, which stays in registers (the upper one is loaded again below).
        const float mx_hi = load_chunk(128, ChunkW{}, sr);
        rowmax = fmaxf(load_chunk(0, ChunkW{}, sr), mx_hi);
      } else if constexpr (BN == 192) {
        // The 64 upper columns for their maximum only, then the 128 lower ones, which
        // stay in registers (the upper ones are loaded again below).
        const float mx_hi = load_chunk(128, std::integral_constant<int, 64>{}, sr);
        rowmax = fmaxf(load_chunk(0, ChunkW{}, sr), mx_hi);
      } else {
        rowmax = load_chunk(0, ChunkW{}, sr);
      }
      const float m2_new = fmaxf(m2, rowmax * sl2);
      const float m2_use = (m2_new > m2 + kRescaleLog2<F16>) ? m2_new : m2;
      const float alpha = ex2_approx(m2 - m2_use);  // 1 if unchanged, 0 on the first tile

      // Rescale O_t by alpha.  With one or two S buffers, S_t(j) complete implies P_t(j-1)
      // V done (one issuing thread, S_t(j) issued after it, completion tracked in order),
      // so O_t is stable here.  (With three buffers that does not hold; the rescale then
      // comes after the exponentials.)
      const bool rescale = j > 0 && __any_sync(0xffffffffu, m2_use != m2);
      if (NS != 3 && rescale) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + 32 * c, o);
        }
      }
      m2 = m2_use;

      // P = exp2(s * scale * log2 e - m2) on pairs (packed fp32 FMA, two MUFU ex2),
      // row sum in packed fp32, P packed to 16-bit pairs and stored over the first BN / 2
      // columns of S_t, 16 columns (32 keys) at a time.
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t negm2 = f2_pack(-m2, -m2);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      // The W scores in s are keys c0 .. c0 + W - 1.
      // 64 keys (32 packed columns) per TMEM store; 32 keys with 256-key tiles, where the
      // larger packed block would not fit beside the 128 scores held (it spilled).
      constexpr int kStoreKeys = BN == 256 ? 32 : 64;
      auto exp_chunk = [&](int c0, auto width) {
        constexpr int W = decltype(width)::value;
#pragma unroll
        for (int h = 0; h < W / kStoreKeys; ++h) {
          uint32_t pk[kStoreKeys / 2];
#pragma unroll
          for (int i = 0; i < kStoreKeys / 2; ++i) {
            const int c = kStoreKeys * h + 2 * i;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, negm2), x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
            pk[i] = pack_elem2<F16>(p0, p1);
          }
          if constexpr (kStoreKeys == 64) tmem_st32(tS + c0 / 2 + 32 * h, pk);
          else tmem_st16(tS + c0 / 2 + 16 * h, pk);
        }
      };
      exp_chunk(0, ChunkW{});
      if constexpr (BN == 256) {
        // The upper half again (its columns are still S: the P of the lower half went to
        // columns 0 .. 63).
        load_chunk(128, ChunkW{}, sr);
        exp_chunk(128, ChunkW{});
      } else if constexpr (BN == 192) {
        // The upper 64 columns again (still S: the P of the lower 128 went to 0 .. 63).
        load_chunk(128, std::integral_constant<int, 64>{}, sr);
        exp_chunk(128, std::integral_constant<int, 64>{});
      }
      float a0, a1, a2, a3, a4, a5, a6, a7;
      f2_unpack(acc[0], a0, a1);
      f2_unpack(acc[1], a2, a3);
      f2_unpack(acc[2], a4, a5);
      f2_unpack(acc[3], a6, a7);
      l = l * alpha + (((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)));
      if constexpr (NS == 3) {
        if (rescale) {
          // S_t(j) may have finished before P_t(j-1) V.  The MMA thread's products
          // complete in issue order, so wait for the first product it issues after
          // P_t(j-1) V (none of which depends on this step): S_1(j) for tile 0; for tile 1
          // S_0(j+1), else P_0(j) V (tile 0's last, o_final), else S_1(j+1), else the
          // one-off pv_done[1] commit.  None of these barriers can have run two phases
          // ahead: their next phases need this tile's next step.  Then rescale O_t before
          // P_t(j) V is issued.
          uint32_t bar;
          int parity;
          if (t == 0) {
            bar = smem_u32(&bars->s_full[2 + (j & 1)]);
            parity = (j >> 1) & 1;
          } else if (j + 1 < n0) {
            bar = smem_u32(&bars->s_full[(j + 1) & 1]);
            parity = ((j + 1) >> 1) & 1;
          } else if (j < n0) {
            bar = smem_u32(&bars->o_final[0]);
            parity = 0;
          } else if (j + 1 < n1) {
            bar = smem_u32(&bars->s_full[2 + ((j + 1) & 1)]);
            parity = ((j + 1) >> 1) & 1;
          } else {
            bar = smem_u32(&bars->pv_done[1]);
            parity = 0;
          }
          ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, p.status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_wait(tO + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_ready[2 * t + (j & 1)]));
    }

    if (ok && nbt > 0) {
      ok = mbar_wait(smem_u32(&bars->o_final[t]), 0, abort, p.status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (split_mode) {
      // Split-KV partial of this row: O / l (fp32) and LSE; an empty range (tile 0
      // past its diagonal in this chunk) gives LSE = -inf and O = 0.
      const int64_t pr = part_row(r0 + rr);
      float4* orow = reinterpret_cast<float4*>(p.ws_o + pr * D);
      if (ok && nbt > 0) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + 32 * c, o);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            orow[8 * c + q] = make_float4(
                __uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
        }
        p.ws_lse[pr] = m2 * 0.69314718055994531f + logf(l);
      } else if (ok) {
#pragma unroll
        for (int c = 0; c < D / 4; ++c) orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        p.ws_lse[pr] = -INFINITY;
      }
    } else {
      // Epilogue: O / l -> bf16 -> swizzled staging in the (now unused) Q_t buffer ->
      // TMA store; LSE = m + ln l in natural-log units of the scaled score.
      uint8_t* stage = smem + (t ? Cfg::kSmemQ1 : Cfg::kSmemQ0);
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tO + 32 * c, o);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_elem2<F16>(__uint_as_float(o[2 * i]) * inv_l,
                                    __uint_as_float(o[2 * i + 1]) * inv_l);
          // columns 32c .. 32c+31 = box (32c / 64), 16-byte chunks (32c % 64) / 8 .. +3
          uint8_t* rowp = stage + (c >> 1) * kBoxBytes + rr * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = ((c & 1) * 4 + q) ^ (rr & 7);
            *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        if (p.lse != nullptr && r0 + rr < p.N)
          p.lse[static_cast<int64_t>(bh) * p.N + r0 + rr] = m2 * 0.69314718055994531f + logf(l);
      }
      fence_proxy_async_smem();
      named_barrier_sync(1 + t, 128);
      if (rr == 0 && ok && !*abort && r0 < p.N) {
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_store_3d(&tm_o, smem_u32(stage + b * kBoxBytes), b * kBoxCols, r0, bh);
        bulk_commit_group();
        bulk_wait_group_read_0();  // staging read: the block may exit
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, Cfg::kTmemCols);
  }
}

// The register hand-off of a 384-thread block (two warpgroups raised to kRegsSoftmax,
// one lowered to kRegsIssue) draws on the registers the block was launched with: it needs
// 168 a thread.  A kernel compiled with fewer would leave setmaxnreg.inc waiting for
// registers that never come, so such a kernel is not launched.  Checked once per kernel.
template <typename Kernel>
cudaError_t check_register_split(Kernel kernel) {
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, kernel);
  if (e != cudaSuccess) return e;
  constexpr int kNeeded = 2 * 128 * kRegsSoftmax + 128 * kRegsIssue;
  static_assert(kNeeded == kAttnThreads * 168, "the split hands over exactly 384 x 168");
  return a.numRegs * kAttnThreads >= kNeeded ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int D, int BN, bool F16>
cudaError_t launch_attn_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const AttnTcParams& p, cudaStream_t stream) {
  using Cfg = AttnTcCfg<D, BN>;
  static_assert(sizeof(AttnTcBarriers) <= 512, "barrier block");
  static const cudaError_t split_ok = check_register_split(attn_fwd_tc_kernel<D, BN, F16>);
  if (split_ok != cudaSuccess) return split_ok;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D, BN, F16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.nqb) * p.BH * p.splits;
  attn_fwd_tc_kernel<D, BN, F16><<<static_cast<unsigned>(grid), kAttnThreads, Cfg::kSmemBytes, stream>>>(
      tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace osfa
