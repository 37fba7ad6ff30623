// attn_bwd_impl.cuh -- kernel bodies of the tcgen05 attention backward (see attn_bwd.cuh).
// Included by one translation unit per head dimension.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "attn_bwd.cuh"
#include "attn_tc_impl.cuh"  // shared-memory / instruction descriptors, 16-bit packing

namespace osfa {

struct AttnBwdBarriers {
  uint64_t fixed_full;   // TMA -> all: the first resident tile (K_j, or Q_i) is in shared memory
  uint64_t fixed1_full;  // ... and the second (V_j, or dO_i), loaded after the first stage's
                         // first tile, which the first product needs with the first one
  uint64_t s_full;       // MMA -> element-wise: S (or S^T) of a tile pair in TMEM
  uint64_t dp_full;      // MMA -> element-wise: dP (or dP^T) in TMEM
  uint64_t p_done;       // element-wise -> MMA: P^T stored (key-outer) / S read (query-outer)
  uint64_t ds_ready;     // element-wise -> MMA: dS (or dS^T) stored in TMEM
  uint64_t acc_final;    // MMA -> element-wise: the last accumulation finished
  uint64_t mma_drain;    // MMA warp: all of its MMAs finished (before TMEM is freed)
  uint64_t mma_drain2;   // one pass: the same for the second MMA warp
  uint64_t stage_full[4];   // key-outer: Q_i and its statistics terms; query-outer: the K ring
  uint64_t stage_do_full[4];  // key-outer: dO_i of the stage (loaded after Q_i: S^T needs
                              // only Q_i and the terms, dP^T and dV need dO_i)
  uint64_t stage_empty[4];
  uint64_t v_full[4];       // query-outer: the V ring
  uint64_t v_empty[4];
  uint64_t s_free;          // one-pass (d = 64): the element-wise warps hold S^T in registers
  uint64_t dp_free;         // one-pass: ... and dP^T
  uint64_t dq_done;         // one-pass: dK and the dQ partial of a tile pair finished
  uint32_t tmem_base;
  int abort;
};

// Element-wise add of a shared-memory box into the global tensor of `tmap` (fp32 adds,
// done at L2); completion tracked like a TMA store, by bulk groups.
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int x, int y,
                                                  int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// mbar_wait with a non-blocking probe first: in these loops most waits find their phase
// complete, and mbarrier.test_wait reports that sooner than the potentially suspending
// try_wait (measured: 1.6 % on the d = 64 backward).
__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                         unsigned* status) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0 || mbar_wait(bar, parity, abort, status);
}

// Issues the load of 32 lanes x 32 TMEM columns (taddr) into d[], stores the 32 words
// of v[] as eight 16-byte chunks of a 128-byte-swizzled row (`base` = row address plus
// the row's swizzle offset, as for st_shared_swz4) while the load is in flight, then
// waits for the load.  The outputs are early-clobber: the load may land before the
// stores have read v[].
__device__ __forceinline__ void tmem_ld32_st_swz8_wait(uint32_t taddr, uint32_t* d, uint32_t base,
                                                       const uint32_t* v) {
  asm volatile(
      "{\n\t.reg .b32 a;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "xor.b32 a, %33, 0;\n\tst.shared.v4.b32 [a], {%34, %35, %36, %37};\n\t"
      "xor.b32 a, %33, 16;\n\tst.shared.v4.b32 [a], {%38, %39, %40, %41};\n\t"
      "xor.b32 a, %33, 32;\n\tst.shared.v4.b32 [a], {%42, %43, %44, %45};\n\t"
      "xor.b32 a, %33, 48;\n\tst.shared.v4.b32 [a], {%46, %47, %48, %49};\n\t"
      "xor.b32 a, %33, 64;\n\tst.shared.v4.b32 [a], {%50, %51, %52, %53};\n\t"
      "xor.b32 a, %33, 80;\n\tst.shared.v4.b32 [a], {%54, %55, %56, %57};\n\t"
      "xor.b32 a, %33, 96;\n\tst.shared.v4.b32 [a], {%58, %59, %60, %61};\n\t"
      "xor.b32 a, %33, 112;\n\tst.shared.v4.b32 [a], {%62, %63, %64, %65};\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t}"
      : "=&r"(d[0]), "=&r"(d[1]), "=&r"(d[2]), "=&r"(d[3]), "=&r"(d[4]), "=&r"(d[5]),
        "=&r"(d[6]), "=&r"(d[7]), "=&r"(d[8]), "=&r"(d[9]), "=&r"(d[10]), "=&r"(d[11]),
        "=&r"(d[12]), "=&r"(d[13]), "=&r"(d[14]), "=&r"(d[15]), "=&r"(d[16]), "=&r"(d[17]),
        "=&r"(d[18]), "=&r"(d[19]), "=&r"(d[20]), "=&r"(d[21]), "=&r"(d[22]), "=&r"(d[23]),
        "=&r"(d[24]), "=&r"(d[25]), "=&r"(d[26]), "=&r"(d[27]), "=&r"(d[28]), "=&r"(d[29]),
        "=&r"(d[30]), "=&r"(d[31])
      : "r"(taddr), "r"(base), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]),
        "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
        "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),
        "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Issues the load of 32 lanes x 32 TMEM columns (taddr) into d[] and, while it is in
// flight, forms P of the 32 scores in s[] (already loaded): x = s * scale log2(e) on pairs,
// p = exp2(x), pv[i] = the fp32 pair (p_2i, p_2i+1) and pk[i] the same pair in the
// kernel's 16-bit type; then waits for the load.  All outputs are early-clobber: the load
// may land, and pv / pk are written, while s[] is still being read.
template <bool F16>
__device__ __forceinline__ void tmem_ld32_exp_chunk(uint32_t taddr, uint32_t* d, const uint32_t* s,
                                                    uint64_t sl2x2, uint64_t* pv, uint32_t* pk) {
  if constexpr (F16) {
#define CVT "cvt.rn.f16x2.f32"
    asm volatile(
        "{\n\t.reg .b64 t;\n\t.reg .f32 x0, x1, q0, q1;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "mov.b64 t, {%66, %67};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %32, {q0, q1};\n\t" CVT " %48, q1, q0;\n\t"
        "mov.b64 t, {%68, %69};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %33, {q0, q1};\n\t" CVT " %49, q1, q0;\n\t"
        "mov.b64 t, {%70, %71};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %34, {q0, q1};\n\t" CVT " %50, q1, q0;\n\t"
        "mov.b64 t, {%72, %73};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %35, {q0, q1};\n\t" CVT " %51, q1, q0;\n\t"
        "mov.b64 t, {%74, %75};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %36, {q0, q1};\n\t" CVT " %52, q1, q0;\n\t"
        "mov.b64 t, {%76, %77};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %37, {q0, q1};\n\t" CVT " %53, q1, q0;\n\t"
        "mov.b64 t, {%78, %79};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %38, {q0, q1};\n\t" CVT " %54, q1, q0;\n\t"
        "mov.b64 t, {%80, %81};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %39, {q0, q1};\n\t" CVT " %55, q1, q0;\n\t"
        "mov.b64 t, {%82, %83};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %40, {q0, q1};\n\t" CVT " %56, q1, q0;\n\t"
        "mov.b64 t, {%84, %85};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %41, {q0, q1};\n\t" CVT " %57, q1, q0;\n\t"
        "mov.b64 t, {%86, %87};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %42, {q0, q1};\n\t" CVT " %58, q1, q0;\n\t"
        "mov.b64 t, {%88, %89};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %43, {q0, q1};\n\t" CVT " %59, q1, q0;\n\t"
        "mov.b64 t, {%90, %91};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %44, {q0, q1};\n\t" CVT " %60, q1, q0;\n\t"
        "mov.b64 t, {%92, %93};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %45, {q0, q1};\n\t" CVT " %61, q1, q0;\n\t"
        "mov.b64 t, {%94, %95};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %46, {q0, q1};\n\t" CVT " %62, q1, q0;\n\t"
        "mov.b64 t, {%96, %97};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %47, {q0, q1};\n\t" CVT " %63, q1, q0;\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : "=&r"(d[0]), "=&r"(d[1]), "=&r"(d[2]), "=&r"(d[3]), "=&r"(d[4]), "=&r"(d[5]), "=&r"(d[6]), "=&r"(d[7]), "=&r"(d[8]), "=&r"(d[9]), "=&r"(d[10]), "=&r"(d[11]), "=&r"(d[12]), "=&r"(d[13]), "=&r"(d[14]), "=&r"(d[15]), "=&r"(d[16]), "=&r"(d[17]), "=&r"(d[18]), "=&r"(d[19]), "=&r"(d[20]), "=&r"(d[21]), "=&r"(d[22]), "=&r"(d[23]), "=&r"(d[24]), "=&r"(d[25]), "=&r"(d[26]), "=&r"(d[27]), "=&r"(d[28]), "=&r"(d[29]), "=&r"(d[30]), "=&r"(d[31]), "=&l"(pv[0]), "=&l"(pv[1]), "=&l"(pv[2]), "=&l"(pv[3]), "=&l"(pv[4]), "=&l"(pv[5]), "=&l"(pv[6]), "=&l"(pv[7]), "=&l"(pv[8]), "=&l"(pv[9]), "=&l"(pv[10]), "=&l"(pv[11]), "=&l"(pv[12]), "=&l"(pv[13]), "=&l"(pv[14]), "=&l"(pv[15]), "=&r"(pk[0]), "=&r"(pk[1]), "=&r"(pk[2]), "=&r"(pk[3]), "=&r"(pk[4]), "=&r"(pk[5]), "=&r"(pk[6]), "=&r"(pk[7]), "=&r"(pk[8]), "=&r"(pk[9]), "=&r"(pk[10]), "=&r"(pk[11]), "=&r"(pk[12]), "=&r"(pk[13]), "=&r"(pk[14]), "=&r"(pk[15])
        : "r"(taddr), "l"(sl2x2), "r"(s[0]), "r"(s[1]), "r"(s[2]), "r"(s[3]), "r"(s[4]), "r"(s[5]), "r"(s[6]), "r"(s[7]), "r"(s[8]), "r"(s[9]), "r"(s[10]), "r"(s[11]), "r"(s[12]), "r"(s[13]), "r"(s[14]), "r"(s[15]), "r"(s[16]), "r"(s[17]), "r"(s[18]), "r"(s[19]), "r"(s[20]), "r"(s[21]), "r"(s[22]), "r"(s[23]), "r"(s[24]), "r"(s[25]), "r"(s[26]), "r"(s[27]), "r"(s[28]), "r"(s[29]), "r"(s[30]), "r"(s[31])
        : "memory");
#undef CVT
  } else {
#define CVT "cvt.rn.bf16x2.f32"
    asm volatile(
        "{\n\t.reg .b64 t;\n\t.reg .f32 x0, x1, q0, q1;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "mov.b64 t, {%66, %67};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %32, {q0, q1};\n\t" CVT " %48, q1, q0;\n\t"
        "mov.b64 t, {%68, %69};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %33, {q0, q1};\n\t" CVT " %49, q1, q0;\n\t"
        "mov.b64 t, {%70, %71};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %34, {q0, q1};\n\t" CVT " %50, q1, q0;\n\t"
        "mov.b64 t, {%72, %73};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %35, {q0, q1};\n\t" CVT " %51, q1, q0;\n\t"
        "mov.b64 t, {%74, %75};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %36, {q0, q1};\n\t" CVT " %52, q1, q0;\n\t"
        "mov.b64 t, {%76, %77};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %37, {q0, q1};\n\t" CVT " %53, q1, q0;\n\t"
        "mov.b64 t, {%78, %79};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %38, {q0, q1};\n\t" CVT " %54, q1, q0;\n\t"
        "mov.b64 t, {%80, %81};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %39, {q0, q1};\n\t" CVT " %55, q1, q0;\n\t"
        "mov.b64 t, {%82, %83};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %40, {q0, q1};\n\t" CVT " %56, q1, q0;\n\t"
        "mov.b64 t, {%84, %85};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %41, {q0, q1};\n\t" CVT " %57, q1, q0;\n\t"
        "mov.b64 t, {%86, %87};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %42, {q0, q1};\n\t" CVT " %58, q1, q0;\n\t"
        "mov.b64 t, {%88, %89};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %43, {q0, q1};\n\t" CVT " %59, q1, q0;\n\t"
        "mov.b64 t, {%90, %91};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %44, {q0, q1};\n\t" CVT " %60, q1, q0;\n\t"
        "mov.b64 t, {%92, %93};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %45, {q0, q1};\n\t" CVT " %61, q1, q0;\n\t"
        "mov.b64 t, {%94, %95};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %46, {q0, q1};\n\t" CVT " %62, q1, q0;\n\t"
        "mov.b64 t, {%96, %97};\n\tmul.rn.f32x2 t, t, %65;\n\tmov.b64 {x0, x1}, t;\n\t"
        "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\t"
        "mov.b64 %47, {q0, q1};\n\t" CVT " %63, q1, q0;\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : "=&r"(d[0]), "=&r"(d[1]), "=&r"(d[2]), "=&r"(d[3]), "=&r"(d[4]), "=&r"(d[5]), "=&r"(d[6]), "=&r"(d[7]), "=&r"(d[8]), "=&r"(d[9]), "=&r"(d[10]), "=&r"(d[11]), "=&r"(d[12]), "=&r"(d[13]), "=&r"(d[14]), "=&r"(d[15]), "=&r"(d[16]), "=&r"(d[17]), "=&r"(d[18]), "=&r"(d[19]), "=&r"(d[20]), "=&r"(d[21]), "=&r"(d[22]), "=&r"(d[23]), "=&r"(d[24]), "=&r"(d[25]), "=&r"(d[26]), "=&r"(d[27]), "=&r"(d[28]), "=&r"(d[29]), "=&r"(d[30]), "=&r"(d[31]), "=&l"(pv[0]), "=&l"(pv[1]), "=&l"(pv[2]), "=&l"(pv[3]), "=&l"(pv[4]), "=&l"(pv[5]), "=&l"(pv[6]), "=&l"(pv[7]), "=&l"(pv[8]), "=&l"(pv[9]), "=&l"(pv[10]), "=&l"(pv[11]), "=&l"(pv[12]), "=&l"(pv[13]), "=&l"(pv[14]), "=&l"(pv[15]), "=&r"(pk[0]), "=&r"(pk[1]), "=&r"(pk[2]), "=&r"(pk[3]), "=&r"(pk[4]), "=&r"(pk[5]), "=&r"(pk[6]), "=&r"(pk[7]), "=&r"(pk[8]), "=&r"(pk[9]), "=&r"(pk[10]), "=&r"(pk[11]), "=&r"(pk[12]), "=&r"(pk[13]), "=&r"(pk[14]), "=&r"(pk[15])
        : "r"(taddr), "l"(sl2x2), "r"(s[0]), "r"(s[1]), "r"(s[2]), "r"(s[3]), "r"(s[4]), "r"(s[5]), "r"(s[6]), "r"(s[7]), "r"(s[8]), "r"(s[9]), "r"(s[10]), "r"(s[11]), "r"(s[12]), "r"(s[13]), "r"(s[14]), "r"(s[15]), "r"(s[16]), "r"(s[17]), "r"(s[18]), "r"(s[19]), "r"(s[20]), "r"(s[21]), "r"(s[22]), "r"(s[23]), "r"(s[24]), "r"(s[25]), "r"(s[26]), "r"(s[27]), "r"(s[28]), "r"(s[29]), "r"(s[30]), "r"(s[31])
        : "memory");
#undef CVT
  }
}

// Issues the load of 32 lanes x 32 TMEM columns (taddr) into d[] and, while it is in
// flight, forms P of the 32 scores in s[] (already loaded) with the row's statistic:
// pv[i] = exp2(s * scale log2(e) - LSE log2(e)) of the pair, fp32; then waits for the
// load.  All outputs are early-clobber.
__device__ __forceinline__ void tmem_ld32_exp_lse_chunk(uint32_t taddr, uint32_t* d, const uint32_t* s,
                                                        uint64_t sl2x2, uint64_t negl2, uint64_t* pv) {
  asm volatile(
      "{\n\t.reg .b64 t;\n\t.reg .f32 x0, x1, q0, q1;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%48];\n\t"
      "mov.b64 t, {%51, %52};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %32, {q0, q1};\n\t"
      "mov.b64 t, {%53, %54};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %33, {q0, q1};\n\t"
      "mov.b64 t, {%55, %56};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %34, {q0, q1};\n\t"
      "mov.b64 t, {%57, %58};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %35, {q0, q1};\n\t"
      "mov.b64 t, {%59, %60};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %36, {q0, q1};\n\t"
      "mov.b64 t, {%61, %62};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %37, {q0, q1};\n\t"
      "mov.b64 t, {%63, %64};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %38, {q0, q1};\n\t"
      "mov.b64 t, {%65, %66};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %39, {q0, q1};\n\t"
      "mov.b64 t, {%67, %68};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %40, {q0, q1};\n\t"
      "mov.b64 t, {%69, %70};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %41, {q0, q1};\n\t"
      "mov.b64 t, {%71, %72};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %42, {q0, q1};\n\t"
      "mov.b64 t, {%73, %74};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %43, {q0, q1};\n\t"
      "mov.b64 t, {%75, %76};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %44, {q0, q1};\n\t"
      "mov.b64 t, {%77, %78};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %45, {q0, q1};\n\t"
      "mov.b64 t, {%79, %80};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %46, {q0, q1};\n\t"
      "mov.b64 t, {%81, %82};\n\tfma.rn.f32x2 t, t, %49, %50;\n\tmov.b64 {x0, x1}, t;\n\t"
      "ex2.approx.ftz.f32 q0, x0;\n\tex2.approx.ftz.f32 q1, x1;\n\tmov.b64 %47, {q0, q1};\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t}"
      : "=&r"(d[0]), "=&r"(d[1]), "=&r"(d[2]), "=&r"(d[3]), "=&r"(d[4]), "=&r"(d[5]), "=&r"(d[6]), "=&r"(d[7]), "=&r"(d[8]), "=&r"(d[9]), "=&r"(d[10]), "=&r"(d[11]), "=&r"(d[12]), "=&r"(d[13]), "=&r"(d[14]), "=&r"(d[15]), "=&r"(d[16]), "=&r"(d[17]), "=&r"(d[18]), "=&r"(d[19]), "=&r"(d[20]), "=&r"(d[21]), "=&r"(d[22]), "=&r"(d[23]), "=&r"(d[24]), "=&r"(d[25]), "=&r"(d[26]), "=&r"(d[27]), "=&r"(d[28]), "=&r"(d[29]), "=&r"(d[30]), "=&r"(d[31]), "=&l"(pv[0]), "=&l"(pv[1]), "=&l"(pv[2]), "=&l"(pv[3]), "=&l"(pv[4]), "=&l"(pv[5]), "=&l"(pv[6]), "=&l"(pv[7]), "=&l"(pv[8]), "=&l"(pv[9]), "=&l"(pv[10]), "=&l"(pv[11]), "=&l"(pv[12]), "=&l"(pv[13]), "=&l"(pv[14]), "=&l"(pv[15])
      : "r"(taddr), "l"(sl2x2), "l"(negl2), "r"(s[0]), "r"(s[1]), "r"(s[2]), "r"(s[3]), "r"(s[4]), "r"(s[5]), "r"(s[6]), "r"(s[7]), "r"(s[8]), "r"(s[9]), "r"(s[10]), "r"(s[11]), "r"(s[12]), "r"(s[13]), "r"(s[14]), "r"(s[15]), "r"(s[16]), "r"(s[17]), "r"(s[18]), "r"(s[19]), "r"(s[20]), "r"(s[21]), "r"(s[22]), "r"(s[23]), "r"(s[24]), "r"(s[25]), "r"(s[26]), "r"(s[27]), "r"(s[28]), "r"(s[29]), "r"(s[30]), "r"(s[31])
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand with 32-byte swizzle (rows of 16
// 16-bit elements; 8-row groups 256 bytes apart): swizzle mode 6 at bits 61-63.
__device__ __forceinline__ uint64_t desc_sw32(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(256 >> 4) << 32) | (1ull << 46) | (6ull << 61);
}

// x as the sum of two bf16 values (high in bits 0..15, low in 16..31): the high part is x
// rounded, the low part the rounded remainder, together within about 2^-18 |x|.
__device__ __forceinline__ uint32_t bf16_hi_lo(float x) {
  const uint32_t hi = pack_bf16x2(x, 0.f) & 0xFFFFu;
  return pack_bf16x2(x, x - __uint_as_float(hi << 16));
}

// Instruction-descriptor bit 15 (kind::f16): the A operand is MN-major in shared memory.
constexpr uint32_t kIdescAMnMajor = 1u << 15;

// Two 16-bit values of the kernel's element type (lower address in bits 0..15) to fp32.
template <bool F16>
__device__ __forceinline__ void unpack_elem2(uint32_t v, float& lo, float& hi) {
  if constexpr (F16) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(v));
  } else {
    lo = __uint_as_float(v << 16);
    hi = __uint_as_float(v & 0xFFFF0000u);
  }
}

// Four 16-byte shared-memory stores of v[0..15] to the chunks C0 .. C0+3 of a 128-byte-
// swizzled row: chunk c goes to (base ^ (16 c)), base being the row's address plus its
// swizzle term 16 (row % 8).  The XORs sit inside the asm, so that one base register
// stays live instead of an address per chunk.
template <int C0>
__device__ __forceinline__ void st_shared_swz4(uint32_t base, const uint32_t* v) {
  asm volatile(
      "{\n\t.reg .b32 a;\n\t"
      "xor.b32 a, %0, %17;\n\tst.shared.v4.b32 [a], {%1, %2, %3, %4};\n\t"
      "xor.b32 a, %0, %18;\n\tst.shared.v4.b32 [a], {%5, %6, %7, %8};\n\t"
      "xor.b32 a, %0, %19;\n\tst.shared.v4.b32 [a], {%9, %10, %11, %12};\n\t"
      "xor.b32 a, %0, %20;\n\tst.shared.v4.b32 [a], {%13, %14, %15, %16};\n\t}"
      ::"r"(base), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
      "r"(v[13]), "r"(v[14]), "r"(v[15]), "n"(C0 * 16), "n"((C0 + 1) * 16), "n"((C0 + 2) * 16),
      "n"((C0 + 3) * 16)
      : "memory");
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Tile order shared by both passes: heads in groups of p.head_group (their streamed
// tiles fit in L2 together); inside a group tile-major, heavy tiles first.  For the
// key-outer pass the heavy causal tiles are the low ones (they meet the most query
// tiles), for the query-outer pass the high ones.
__device__ __forceinline__ void bwd_work(const AttnBwdParams& p, bool low_first, int* bh,
                                         int* tile) {
  const int L = blockIdx.x;
  const int per_group = p.head_group * p.nblk;
  const int full = p.BH / p.head_group;
  const int g = L / per_group;
  int r, hg, base;
  if (g < full) {
    r = L - g * per_group;
    hg = p.head_group;
    base = g * p.head_group;
  } else {
    r = L - full * per_group;
    hg = p.BH - full * p.head_group;
    base = full * p.head_group;
  }
  const int t = r / hg;
  *tile = low_first ? t : p.nblk - 1 - t;
  *bh = base + r % hg;
}

// D_i = sum_c dO_ic O_ic and LSE_i * log2(e); rows N .. n_pad-1 of each head get D = 0 and
// +inf.  A warp takes kPrepRows<D> query rows and issues all their loads before reducing
// any, so that enough bytes are in flight to stream O and dO at HBM speed (eight rows at
// d = 64, whose rows are half as long; four at d = 128, where eight measured slower).
template <int D>
constexpr int kPrepRows = D == 64 ? 8 : 4;

template <int D, bool F16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                            const uint16_t* __restrict__ dout,
                                                            const float* __restrict__ lse,
                                                            float* __restrict__ lse2,
                                                            float* __restrict__ dd, int BH, int N,
                                                            int n_pad, float* __restrict__ dq_acc,
                                                            uint16_t* __restrict__ aug,
                                                            float inv_scale) {
  constexpr int kPer = D / 32;  // 16-bit elements per lane and row: 2 or 4
  const long long total = static_cast<long long>(BH) * n_pad;
  const long long row0 =
      (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kPrepRows<D>;
  const int lane = threadIdx.x & 31;
  if (dq_acc != nullptr) {
    // One-pass backward (d = 64): the fp32 dQ accumulator rows of these query rows start
    // at zero (64 floats = 16 float4 per row).
#pragma unroll
    for (int r = 0; r < kPrepRows<D>; ++r) {
      const long long row = row0 + r;
      if (row < total && lane < 16)
        reinterpret_cast<float4*>(dq_acc + row * 64)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  uint32_t av[kPrepRows<D>][kPer / 2], bv[kPrepRows<D>][kPer / 2];
  bool real[kPrepRows<D>];
#pragma unroll
  for (int r = 0; r < kPrepRows<D>; ++r) {
    const long long row = row0 + r;
    const long long bh = row / n_pad;
    const int q = static_cast<int>(row - bh * n_pad);
    real[r] = row < total && q < N;
#pragma unroll
    for (int i = 0; i < kPer / 2; ++i) av[r][i] = bv[r][i] = 0u;
    if (real[r]) {
      const long long off = (bh * N + q) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(o + off);
        const uint2 b = *reinterpret_cast<const uint2*>(dout + off);
        av[r][0] = a.x; av[r][1] = a.y;
        bv[r][0] = b.x; bv[r][1] = b.y;
      } else {
        av[r][0] = *reinterpret_cast<const uint32_t*>(o + off);
        bv[r][0] = *reinterpret_cast<const uint32_t*>(dout + off);
      }
    }
  }
  float acc[kPrepRows<D>];
#pragma unroll
  for (int r = 0; r < kPrepRows<D>; ++r) {
    acc[r] = 0.f;
#pragma unroll
    for (int i = 0; i < kPer / 2; ++i) {
      float a0, a1, b0, b1;
      unpack_elem2<F16>(av[r][i], a0, a1);
      unpack_elem2<F16>(bv[r][i], b0, b1);
      acc[r] = fmaf(a0, b0, acc[r]);
      acc[r] = fmaf(a1, b1, acc[r]);
    }
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
    for (int r = 0; r < kPrepRows<D>; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], sh);
  if (lane < kPrepRows<D>) {
    float mine = acc[0];
#pragma unroll
    for (int r = 1; r < kPrepRows<D>; ++r) mine = (lane == r) ? acc[r] : mine;
    const long long row = row0 + lane;
    if (row < total) {
      const long long bh = row / n_pad;
      const int q = static_cast<int>(row - bh * n_pad);
      // The key-outer kernels' statistics terms [-LSE/scale high, low, -D high, low, 0 ...]
      // (all 0 for rows >= N: those queries have zero dO and dP rows, so whatever P they
      // get adds nothing), and for the query-outer pass LSE * log2(e) and D.
      const float c = q < N ? -lse[bh * N + q] * inv_scale : 0.f;
      const float nd = q < N ? -mine : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(aug + row * 16);
      dst[0] = make_uint4(bf16_hi_lo(c), bf16_hi_lo(nd), 0u, 0u);
      dst[1] = make_uint4(0u, 0u, 0u, 0u);
      if (lse2 != nullptr) {
        dd[row] = q < N ? mine : 0.f;
        lse2[row] = q < N ? lse[bh * N + q] * 1.4426950408889634f : INFINITY;
      }
    }
  }
}

// Writes 32 fp32 accumulator columns (times `mul`) of one row as 16-bit values.
template <bool F16>
__device__ __forceinline__ void store_row32(uint8_t* dst, const uint32_t* a, float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack_elem2<F16>(__uint_as_float(a[2 * i]) * mul, __uint_as_float(a[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// ------------------------------------------------------------------------------------
// Key-outer pass: dK_j, dV_j; with Fused (d = 64 only) also the dQ partials dS K_j.
// ------------------------------------------------------------------------------------
template <int D, bool F16, bool Fused>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dqacc,
                         const __grid_constant__ CUtensorMap tm_aug, const AttnBwdParams p) {
  static_assert(!Fused || D == 64, "the one-pass backward is for d = 64");
  using Cfg = std::conditional_t<Fused, AttnBwd1Cfg, AttnBwdCfg<D>>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  AttnBwdBarriers* bars = reinterpret_cast<AttnBwdBarriers*>(smem + Cfg::kSmemBars);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int bh, j;
  bwd_work(p, true, &bh, &j);
  const int i0 = p.causal ? j : 0;  // query tiles i < j see none of these keys
  const int nq = p.nblk - i0;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->fixed_full), 1);
    mbar_init(smem_u32(&bars->fixed1_full), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->p_done), 8);    // one arrival per element-wise warp
    mbar_init(smem_u32(&bars->ds_ready), 8);
    // One pass: the two MMA warps each commit once to acc_final and to stage_empty.
    mbar_init(smem_u32(&bars->acc_final), Fused ? 2 : 1);
    mbar_init(smem_u32(&bars->mma_drain), 1);
    mbar_init(smem_u32(&bars->mma_drain2), 1);
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(smem_u32(&bars->stage_full[s]), 1);
      mbar_init(smem_u32(&bars->stage_do_full[s]), 1);
      mbar_init(smem_u32(&bars->stage_empty[s]), Fused ? 2 : 1);
    }
    mbar_init(smem_u32(&bars->s_free), 8);
    mbar_init(smem_u32(&bars->dp_free), 8);
    mbar_init(smem_u32(&bars->dq_done), 1);
    bars->abort = 0;
    mbar_init_fence();
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(smem_u32(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish();
  }
  {
    // The two constant A tiles of the statistics step (2 x 256 16-byte chunks): in every
    // row [1, 1, 0, ...] (bf16) then [0, 0, 1, 1, 0, ...], repeated in both halves.
    constexpr uint32_t kOne2 = 0x3F803F80u;  // two bf16 ones
    uint4* ones = reinterpret_cast<uint4*>(smem + Cfg::kSmemOnes);
    for (int c = threadIdx.x; c < 2 * Cfg::kAugBytes / 16; c += kBwdThreads)
      ones[c] = c < Cfg::kAugBytes / 16 ? make_uint4(kOne2, 0u, 0u, 0u) : make_uint4(0u, kOne2, 0u, 0u);
    fence_proxy_async_smem();  // read by the tensor pipe
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  volatile int* abort = &bars->abort;
  auto stage_addr = [&](int s) { return sbase + Cfg::kSmemStages + s * Cfg::kStageBytes; };

  if (warp == 11 || (!Fused && warp == kBwdWarpMma2)) {
    // idle
  } else if (warp == kBwdWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      // K_j, then Q_i0 and its terms (all the first S^T needs), then V_j, then dO_i0, ...
      const uint32_t fbar = smem_u32(&bars->fixed_full);
      const uint32_t fbar1 = smem_u32(&bars->fixed1_full);
      mbar_arrive_expect_tx(fbar, Cfg::kTileBytes);
#pragma unroll
      for (int b = 0; b < Cfg::kBoxes; ++b)
        tma_load_3d(sbase + Cfg::kSmemFixed0 + b * kBoxBytes, &tm_k, fbar, b * kBoxCols, j * kBlockM, bh);
      auto load_v = [&]() {
        mbar_arrive_expect_tx(fbar1, Cfg::kTileBytes);
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_load_3d(sbase + Cfg::kSmemFixed1 + b * kBoxBytes, &tm_v, fbar1, b * kBoxCols,
                      j * kBlockM, bh);
      };
      bool v_issued = false;
      int issued = 0;
      for (int it = 0; it < nq; ++it) {
        const int s = it % Cfg::kStages;
        if (!bwd_wait(smem_u32(&bars->stage_empty[s]), ((it / Cfg::kStages) & 1) ^ 1, abort,
                       p.status))
          break;
        const uint32_t full = smem_u32(&bars->stage_full[s]);
        const uint32_t do_full = smem_u32(&bars->stage_do_full[s]);
        const int i = i0 + it;
        const uint32_t dst = stage_addr(s);
        // Q_i and the terms first (the next S^T waits for them alone), then dO_i.
        mbar_arrive_expect_tx(full, Cfg::kTileBytes + Cfg::kAugBytes);
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_load_3d(dst + b * kBoxBytes, &tm_q, full, b * kBoxCols, i * kBlockM, bh);
        tma_load_3d(dst + 2 * Cfg::kTileBytes, &tm_aug, full, 0, i * kBlockM, bh);
        if (!v_issued) {
          load_v();
          v_issued = true;
        }
        mbar_arrive_expect_tx(do_full, Cfg::kTileBytes);
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_load_3d(dst + Cfg::kTileBytes + b * kBoxBytes, &tm_do, do_full, b * kBoxCols,
                      i * kBlockM, bh);
        issued = it + 1;
      }
      // Every issued copy must land before the block's shared memory goes away.
      int no_abort = 0;
      bwd_wait(fbar, 0, &no_abort, p.status);
      if (v_issued) bwd_wait(fbar1, 0, &no_abort, p.status);
      for (int it = max(0, issued - Cfg::kStages); it < issued; ++it) {
        bwd_wait(smem_u32(&bars->stage_full[it % Cfg::kStages]), (it / Cfg::kStages) & 1,
                  &no_abort, p.status);
        bwd_wait(smem_u32(&bars->stage_do_full[it % Cfg::kStages]), (it / Cfg::kStages) & 1,
                 &no_abort, p.status);
      }
    }
  } else if (warp == kBwdWarpMma || (Fused && warp == kBwdWarpMma2)) {
    // ------------------------------------------------------------ MMA issuers
    // One pass: two warps issue the products, each on its own SM sub-partition (both
    // share theirs with two element-wise warps, and every instruction on an issuing
    // warp's path costs).  The products of one issuing thread complete in issue order; a
    // stage is released by one commit of each warp, and acc_final takes one of each.
    const bool second = warp == kBwdWarpMma2;
    constexpr uint32_t kIdescS = idesc_f16kind(kBlockM, kBlockM, false, F16);
    constexpr uint32_t kIdescAcc = idesc_f16kind(kBlockM, D, true, F16);
    const uint64_t dK = desc_sw128(sbase + Cfg::kSmemFixed0, 16, 1024);   // A of S^T
    const uint64_t dV = desc_sw128(sbase + Cfg::kSmemFixed1, 16, 1024);   // A of dP^T
    const uint32_t tS = tbase + Cfg::kColS, tDP = tbase + Cfg::kColDP;
    const uint32_t tDV = tbase + Cfg::kColAcc0, tDK = tbase + Cfg::kColAcc1;
    auto wait_bar = [&](uint64_t* bar, int parity) {
      const bool r = __all_sync(0xffffffffu, bwd_wait(smem_u32(bar), parity, abort, p.status));
      if (r) tc_fence_after();
      return r;
    };
    auto desc_k = [&](int it, int tile) {  // K-major view of a streamed tile
      return desc_sw128(stage_addr(it % Cfg::kStages) + tile * Cfg::kTileBytes, 16, 1024);
    };
    auto desc_mn = [&](int it, int tile) {  // MN-major view of a streamed tile
      return desc_sw128(stage_addr(it % Cfg::kStages) + tile * Cfg::kTileBytes, kBoxBytes, 1024);
    };
    // The statistics step: the constant ones tile `dOnes` (A) times the query tile's terms
    // (B, in stage st) adds -LSE/scale (dOnesS) or -D (dOnesD) to every column; a bf16
    // product, whatever the element type of the others.
    constexpr uint32_t kIdescAug = idesc_f16kind(kBlockM, kBlockM, false, false);
    const uint64_t dOnesS = desc_sw32(sbase + Cfg::kSmemOnes);
    const uint64_t dOnesD = desc_sw32(sbase + Cfg::kSmemOnes + Cfg::kAugBytes);
    auto issue_aug = [&](uint32_t tD, uint64_t dOnes, int st) {
      mma_bf16_ss_elect(tD, dOnes, desc_sw32(stage_addr(st % Cfg::kStages) + 2 * Cfg::kTileBytes),
                        kIdescAug, 1u);
    };
    // S^T - LSE/scale = K_j Q_i^T + (stats) into tS, or dP^T - D = V_j dO_i^T + (stats) into
    // tDP: keys on lanes, queries on columns; the streamed tile is the K-major B operand.
    auto issue_t = [&](uint32_t tD, uint64_t dA, uint64_t dB, uint64_t dOnes, int st) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off16 = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss_elect(tD, dA + off16, dB + off16, kIdescS, kk > 0 ? 1u : 0u);
      }
      issue_aug(tD, dOnes, st);
    };
    // tAcc += A^T-part from TMEM (16 queries = 8 packed columns per step; column half h
    // of the tile was packed into columns 64h .. 64h+31) times a streamed MN-major tile.
    auto issue_acc = [&](uint32_t tAcc, uint32_t tA, uint64_t dB, bool acc) {
#pragma unroll
      for (int kk = 0; kk < kBlockM / 16; ++kk) {
        const uint32_t acol = (kk >> 2) * 64 + (kk & 3) * 8;
        mma_bf16_ts_elect(tAcc, tA + acol, dB + ((kk * 2048) >> 4), kIdescAcc,
                          (acc || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = wait_bar(&bars->fixed_full, 0) && wait_bar(&bars->stage_full[0], 0);
    auto wait_do = [&](int it) {  // dO_it has landed
      return wait_bar(&bars->stage_do_full[it % Cfg::kStages], (it / Cfg::kStages) & 1);
    };
    auto wait_v_do0 = [&]() {  // V_j and dO of the first query tile have landed
      return wait_bar(&bars->fixed1_full, 0) && wait_do(0);
    };
    if constexpr (Fused) {
      // One pass (d = 64).  The first warp issues, per query tile it,
      //   S^T(it+1) (once the element-wise warps hold S^T(it) in registers)  |
      //   dV(it) = P^T(it) dO_it (P^T in its own columns)  |
      //   dP^T(it+1) (once they hold dP^T(it) as well),
      // and the second dK(it) = dS^T(it) Q_it and dQ(it) = dS(it) K_j once dS(it) is
      // staged.  dS of the tile pair is staged in shared memory once,
      // [key][query] in two 64-query boxes (128-byte swizzle), and read by both of its
      // products: K-major as the A operand dS^T of dK, MN-major (the boxes 16 KB apart) as
      // the A operand dS of dQ.  dS^T is not stored in TMEM, so dP^T(it+1) need not wait
      // for dK(it) and runs while the element-wise warps form dS(it).  The products of one
      // issuing thread complete in issue order: the commit of dP^T(it) also reports
      // dV(it-1) done (P^T may be overwritten), and the second warp's commit after dQ(it)
      // (dq_done) reports dK(it) done too (the staging may be rewritten, the partial
      // drained); dQ(it+1) is issued only after ds_ready(it+1), which the element-wise
      // warps signal after that drain.
      // S^T (or dP^T), K = 64 under one elect, then the statistics step.
      auto group_t = [&](uint32_t tD, uint64_t dA, uint64_t dB, uint64_t dOnes, int st) {
        uint64_t a[4], b[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          a[kk] = dA + 2 * kk;
          b[kk] = dB + 2 * kk;
        }
        mma_ss4_elect(tD, a, b, kIdescS, 0u);
        issue_aug(tD, dOnes, st);
      };
      const uint32_t tP = tbase + Cfg::kColP;
      if (second) {
        // dK += dS^T(it) Q_it: A = the staging read K-major, 16 queries (32 bytes of a
        // 128-byte row) per step, the second 64-query box 16 KB on; dQ(it) = dS(it) K_j:
        // A = the staging read MN-major, B = K_j MN-major, 16 keys per step.
        constexpr uint32_t kIdescDQ = kIdescAcc | kIdescAMnMajor;
        const uint64_t dDS = desc_sw128(sbase + Cfg::kSmemDS, kBoxBytes, 1024);
        const uint64_t dDSt = desc_sw128(sbase + Cfg::kSmemDS, 16, 1024);
        const uint64_t dKmn = desc_sw128(sbase + Cfg::kSmemFixed0, kBoxBytes, 1024);
        const uint32_t tDQ = tbase + Cfg::kColDQ;
        for (int it = 0; ok && it < nq; ++it) {
          const int st = it % Cfg::kStages;
          if (!(ok = wait_bar(&bars->stage_full[st], (it / Cfg::kStages) & 1) &&
                     wait_bar(&bars->ds_ready, it & 1)))
            break;
          {
            uint64_t a[8], b[8];
            const uint64_t dB = desc_mn(it, 0);  // Q_it
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              a[kk] = dDSt + ((((kk >> 2) * kBoxBytes) + (kk & 3) * 32) >> 4);
              b[kk] = dB + kk * 128;
            }
            mma_ss8_elect(tDK, a, b, kIdescAcc, it > 0 ? 1u : 0u);
          }
          mma_commit_elect(smem_u32(&bars->stage_empty[st]));
          {
            uint64_t a[8], b[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              a[kk] = dDS + kk * 128;
              b[kk] = dKmn + kk * 128;
            }
            mma_ss8_elect(tDQ, a, b, kIdescDQ, 0u);
          }
          mma_commit_elect(smem_u32(&bars->dq_done));
        }
      } else {
        if (ok) {
          group_t(tS, dK, desc_k(0, 0), dOnesS, 0);
          mma_commit_elect(smem_u32(&bars->s_full));
          if ((ok = wait_v_do0())) {
            group_t(tDP, dV, desc_k(0, 1), dOnesD, 0);
            mma_commit_elect(smem_u32(&bars->dp_full));
          }
        }
        for (int it = 0; ok && it < nq; ++it) {
          const bool more = it + 1 < nq;
          if (more) {
            if (!(ok = wait_bar(&bars->stage_full[(it + 1) % Cfg::kStages],
                                ((it + 1) / Cfg::kStages) & 1) &&
                       wait_bar(&bars->s_free, it & 1)))
              break;
            group_t(tS, dK, desc_k(it + 1, 0), dOnesS, it + 1);
            mma_commit_elect(smem_u32(&bars->s_full));
          }
          if (!(ok = wait_bar(&bars->p_done, it & 1))) break;
          {
            // dV += P^T(it) dO_it: A = 16 queries (8 packed columns) per step, the 64-query
            // halves 32 columns apart.
            uint32_t a[8];
            uint64_t b[8];
            const uint64_t dB = desc_mn(it, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              a[kk] = tP + (kk >> 2) * 32 + (kk & 3) * 8;
              b[kk] = dB + kk * 128;
            }
            mma_ts8_elect(tDV, a, b, kIdescAcc, it > 0 ? 1u : 0u);
          }
          // This warp's last product reading stage it.
          mma_commit_elect(smem_u32(&bars->stage_empty[it % Cfg::kStages]));
          if (more) {
            if (!(ok = wait_bar(&bars->dp_free, it & 1) && wait_do(it + 1))) break;
            group_t(tDP, dV, desc_k(it + 1, 1), dOnesD, it + 1);
            mma_commit_elect(smem_u32(&bars->dp_full));
          }
        }
      }
    } else {
      // Two passes (d = 128), one issuing warp; software pipeline on the tensor pipe, per
      // query tile it:
      //   dV += P^T(it) dO_it  |  S^T(it+1)  |  dK += dS^T(it) Q_it  |  dP^T(it+1)
      // dV needs only P^T, so it and the next S^T run while the element-wise warps form
      // dS^T; the next element-wise step starts on S^T(it+1) while dK and dP^T(it+1) run.
      // P^T is stored over S^T and dS^T over dP^T: each region is overwritten only after
      // the product that reads it (issue order).  (Issuing dK and dP^T from a second warp,
      // as the one-pass kernel does, lets dK overtake the next S^T and was slower here.)
      if (ok) {
        issue_t(tS, dK, desc_k(0, 0), dOnesS, 0);
        mma_commit_elect(smem_u32(&bars->s_full));
        if ((ok = wait_v_do0())) {
          issue_t(tDP, dV, desc_k(0, 1), dOnesD, 0);
          mma_commit_elect(smem_u32(&bars->dp_full));
        }
      }
      for (int it = 0; ok && it < nq; ++it) {
        const bool more = it + 1 < nq;
        if (!(ok = wait_bar(&bars->p_done, it & 1))) break;
        issue_acc(tDV, tS, desc_mn(it, 1), it > 0);
        if (more) {
          if (!(ok = wait_bar(&bars->stage_full[(it + 1) % Cfg::kStages],
                              ((it + 1) / Cfg::kStages) & 1)))
            break;
          issue_t(tS, dK, desc_k(it + 1, 0), dOnesS, it + 1);
          mma_commit_elect(smem_u32(&bars->s_full));
        }
        if (!(ok = wait_bar(&bars->ds_ready, it & 1))) break;
        issue_acc(tDK, tDP, desc_mn(it, 0), it > 0);
        mma_commit_elect(smem_u32(&bars->stage_empty[it % Cfg::kStages]));
        if (more) {
          if (!(ok = wait_do(it + 1))) break;
          issue_t(tDP, dV, desc_k(it + 1, 1), dOnesD, it + 1);
          mma_commit_elect(smem_u32(&bars->dp_full));
        }
      }
    }
    if (ok) mma_commit_elect(smem_u32(&bars->acc_final));
    uint64_t* drain = second ? &bars->mma_drain2 : &bars->mma_drain;
    mma_commit_elect(smem_u32(drain));
    int no_abort = 0;
    bwd_wait(smem_u32(drain), 0, &no_abort, p.status);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int h = warp >> 2;         // column half of the tile
    const int wq = warp & 3;         // TMEM lane quarter
    const int r = wq * 32 + lane;    // key within the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + Cfg::kColS, tDP = tbase + lane_off + Cfg::kColDP;
    const float sl2 = p.scale_log2;
    bool ok = true;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    // P^T of 32 queries (columns c0 .. c0+31 of this key's row) from S^T - LSE/scale:
    // exp2(scale log2 e (S^T - LSE/scale)), kept in fp32 pairs (pv, for dS^T) and packed
    // to 16 bits (pk, the A operand of dV); causal diagonal tile: query q sees key r iff
    // r <= q.
    auto p_chunk = [&](const uint32_t* sr, int c0, bool diag, uint64_t* pv, uint32_t* pk) {
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float x0, x1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2),
                  x0, x1);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (diag) {
          if (c0 + c < r) p0 = 0.f;
          if (c0 + c + 1 < r) p1 = 0.f;
        }
        pv[c >> 1] = f2_pack(p0, p1);
        pk[c >> 1] = pack_elem2<F16>(p0, p1);
      }
    };
    // dS^T = P^T * (dP^T - D) of 32 queries from dP^T - D, packed to 16 bits.
    auto ds_chunk = [&](const uint32_t* dr, const uint64_t* pv, uint32_t* pd) {
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float d0, d1;
        f2_unpack(f2_mul(pv[c >> 1], f2_pack(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1]))),
                  d0, d1);
        pd[c >> 1] = pack_elem2<F16>(d0, d1);
      }
    };
    // One-pass: the dQ partial of query tile t (TMEM lanes 32 wq .. +31 = its queries,
    // columns 32 h .. +31) goes through this warp's 32 x 32 fp32 staging box (128-byte
    // swizzle) into the accumulator by a TMA reduce-add.  Called once the partial is
    // known complete (dP^T of tile t + 1 seen, or the final commit).
    // One pass: the dQ partial of a query tile (TMEM lanes 32 wq .. +31 = its queries,
    // columns 32 h .. +31) goes through this warp's 32 x 32 fp32 staging box (128-byte
    // swizzle) into the accumulator by a TMA reduce-add, in two steps around the caller's
    // fence.proxy.async: the partial into the box (once the partial is known complete and
    // the box's previous reduce-add has read it), then the reduce-add of query tile t.
    auto dq_to_box = [&]() {
      if constexpr (Fused) {
        uint32_t a[32];
        tmem_ld32_wait(tbase + lane_off + Cfg::kColDQ + 32 * h, a);
        tc_fence_before();
        if (lane == 0) bulk_wait_group_read_0();  // the last reduce-add has read the box
        __syncwarp();
        const uint32_t row =
            sbase + Cfg::kSmemRed + warp * Cfg::kRedBoxBytes + lane * 128 + ((lane & 7) << 4);
        st_shared_swz4<0>(row, a);
        st_shared_swz4<4>(row, a + 16);
      }
    };
    auto box_to_acc = [&](int t) {
      if constexpr (Fused) {
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dqacc, sbase + Cfg::kSmemRed + warp * Cfg::kRedBoxBytes, 32 * h,
                            (i0 + t) * kBlockM + wq * 32, bh);
          bulk_commit_group();
        }
      }
    };
    if constexpr (Fused) {
      // One pass (d = 64), per query tile it: S^T - LSE/scale into registers, "S^T free"
      // (the next S^T may overwrite it), P; then, once dP^T(it) - D is in (which also
      // reports dV of tile it - 1 complete), P^T into its own columns, p_done; dP^T into
      // registers, "dP^T free"; once dK and dQ of tile it - 1 are complete (dq_done), its
      // dQ partial into the staging box, dS into the shared-memory staging, one proxy
      // fence for both, the partial's reduce-add, ds_ready.  The statistics came in
      // through the tensor core, so these warps read nothing from the stages.
      const uint32_t tP = tbase + lane_off + Cfg::kColP;
      for (int it = 0; ok && it < nq; ++it) {
        ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->s_full), it & 1, abort, p.status));
        if (!ok) break;
        tc_fence_after();
        const bool diag = p.causal && i0 + it == j;
        uint64_t pv[32];
        uint32_t pk[32];
        if (!diag) {
          // The second half of this warp's S^T loads while P of the first half is formed.
          uint32_t sr0[32], sr1[32];
          tmem_ld32_wait(tS + 64 * h, sr0);
          tmem_ld32_exp_chunk<F16>(tS + 64 * h + 32, sr1, sr0, sl2x2, pv, pk);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->s_free));
          p_chunk(sr1, 64 * h + 32, false, pv + 16, pk + 16);
        } else {
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t sr[32];
            tmem_ld32_wait(tS + 64 * h + 32 * ch, sr);
            if (ch == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&bars->s_free));
            }
            p_chunk(sr, 64 * h + 32 * ch, true, pv + 16 * ch, pk + 16 * ch);
          }
        }
        ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->dp_full), it & 1, abort, p.status));
        if (!ok) break;
        tc_fence_after();
        // P^T: query q of this warp's half in column q / 2 of the P^T columns.
        tmem_st16(tP + 32 * h, pk);
        tmem_st16(tP + 32 * h + 16, pk + 16);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_done));
        // dS^T = P^T * (dP^T - D) of this warp's 64 queries, 16-bit.
        uint32_t pd[32];
        {
          uint32_t dr[32];
          tmem_ld32_wait(tDP + 64 * h, dr);
          ds_chunk(dr, pv, pd);
          tmem_ld32_wait(tDP + 64 * h + 32, dr);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->dp_free));
          ds_chunk(dr, pv + 16, pd + 16);
        }
        // Row r (this key) of box h: queries 64h .. 64h+63 are its 16-byte chunks 0 .. 7,
        // each at its 128-byte-swizzle position (chunk ^ (r % 8)).
        const uint32_t row = sbase + Cfg::kSmemDS + h * kBoxBytes + r * 128 + ((r & 7) << 4);
        if (it > 0) {
          ok = __all_sync(0xffffffffu,
                          bwd_wait(smem_u32(&bars->dq_done), (it - 1) & 1, abort, p.status));
          if (!ok) break;
          tc_fence_after();
          // The dQ partial of tile it - 1 is loaded while dS goes to the staging, then
          // goes to this warp's box.
          uint32_t a[32];
          tmem_ld32_st_swz8_wait(tbase + lane_off + Cfg::kColDQ + 32 * h, a, row, pd);
          tc_fence_before();
          if (lane == 0) bulk_wait_group_read_0();  // the last reduce-add has read the box
          __syncwarp();
          const uint32_t rrow =
              sbase + Cfg::kSmemRed + warp * Cfg::kRedBoxBytes + lane * 128 + ((lane & 7) << 4);
          st_shared_swz4<0>(rrow, a);
          st_shared_swz4<4>(rrow, a + 16);
        } else {
          st_shared_swz4<0>(row, pd);
          st_shared_swz4<4>(row, pd + 16);
        }
        fence_proxy_async_smem();  // dS and the dQ box are read by the async proxy
        tc_fence_before();
        __syncwarp();
        if (it > 0) box_to_acc(it - 1);
        if (lane == 0) mbar_arrive(smem_u32(&bars->ds_ready));
      }
    } else {
    // The statistics came in through the tensor core (S^T - LSE/scale, dP^T - D), so these
    // warps read nothing from the stages.
    for (int it = 0; ok && it < nq; ++it) {
      ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->s_full), it & 1, abort, p.status));
      if (!ok) break;
      tc_fence_after();
      const int i = i0 + it;
      const bool diag = p.causal && i == j;  // query q sees key r iff r <= q
      // P^T: kept in registers for dS^T and stored (16-bit) over the first half of this
      // warp's S^T columns for dV.
      uint64_t pv[32];
      if (!diag) {
        // The second half of this warp's S^T loads while P of the first half is formed.
        uint32_t sr0[32], sr1[32], pk[16];
        tmem_ld32_wait(tS + 64 * h, sr0);
        tmem_ld32_exp_chunk<F16>(tS + 64 * h + 32, sr1, sr0, sl2x2, pv, pk);
        tmem_st16(tS + 64 * h, pk);
        p_chunk(sr1, 64 * h + 32, false, pv + 16, pk);
        tmem_st16(tS + 64 * h + 16, pk);
      } else {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = 64 * h + 32 * ch;    // first query (column) of this chunk
          uint32_t sr[32], pk[16];
          tmem_ld32_wait(tS + c0, sr);
          p_chunk(sr, c0, true, pv + 16 * ch, pk);
          tmem_st16(tS + 64 * h + 16 * ch, pk);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_done));

      // dS^T = P^T * (dP^T - D), stored over the first half of this warp's dP^T columns.
      ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->dp_full), it & 1, abort, p.status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * h + 32 * ch;
        uint32_t dr[32], pd[16];
        tmem_ld32_wait(tDP + c0, dr);
        ds_chunk(dr, pv + 16 * ch, pd);
        tmem_st16(tDP + 64 * h + 16 * ch, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->ds_ready));
    }
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->acc_final), 0, abort, p.status));
    }
    if (Fused && ok) {
      tc_fence_after();
      dq_to_box();
      fence_proxy_async_smem();
      __syncwarp();
      box_to_acc(nq - 1);
    }
    const int kg = j * kBlockM + r;
    if (ok) {
      tc_fence_after();
      uint8_t* dv_row = static_cast<uint8_t*>(p.dv) + (static_cast<long long>(bh) * p.N + kg) * D * 2;
      uint8_t* dk_row = static_cast<uint8_t*>(p.dk) + (static_cast<long long>(bh) * p.N + kg) * D * 2;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = h * (D / 2) + 32 * c;
        uint32_t a[32];
        tmem_ld32_wait(tbase + lane_off + Cfg::kColAcc0 + col, a);
        if (kg < p.N) store_row32<F16>(dv_row + col * 2, a, 1.0f);
        tmem_ld32_wait(tbase + lane_off + Cfg::kColAcc1 + col, a);
        if (kg < p.N) store_row32<F16>(dk_row + col * 2, a, p.scale);
      }
    }
    // The reduce-adds in flight read this block's shared memory: they finish first.
    if constexpr (Fused) {
      if (lane == 0) bulk_wait_group_0();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, Cfg::kTmemCols);
  }
}

// ------------------------------------------------------------------------------------
// Query-outer pass: dQ_i.
// ------------------------------------------------------------------------------------
template <int D, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const AttnBwdParams p) {
  using Cfg = AttnBwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  AttnBwdBarriers* bars = reinterpret_cast<AttnBwdBarriers*>(smem + Cfg::kDqSmemBars);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int bh, i;
  bwd_work(p, false, &bh, &i);
  const int nk = p.causal ? i + 1 : p.nblk;  // key tiles j > i are all above the diagonal

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->fixed_full), 1);
    mbar_init(smem_u32(&bars->fixed1_full), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->p_done), 8);    // one arrival per element-wise warp
    mbar_init(smem_u32(&bars->ds_ready), 8);
    mbar_init(smem_u32(&bars->acc_final), 1);
    mbar_init(smem_u32(&bars->mma_drain), 1);
    for (int s = 0; s < Cfg::kDqSlotsK; ++s) {
      mbar_init(smem_u32(&bars->stage_full[s]), 1);
      mbar_init(smem_u32(&bars->stage_empty[s]), 1);
    }
    for (int s = 0; s < Cfg::kDqSlotsV; ++s) {
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->v_empty[s]), 1);
    }
    bars->abort = 0;
    mbar_init_fence();
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(smem_u32(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  volatile int* abort = &bars->abort;
  auto k_addr = [&](int it) {
    return sbase + Cfg::kDqSmemK + (it % Cfg::kDqSlotsK) * Cfg::kTileBytes;
  };
  auto v_addr = [&](int it) { return sbase + Cfg::kDqSmemV + (it % Cfg::kDqSlotsV) * Cfg::kTileBytes; };

  if (warp >= 10) {
    // idle
  } else if (warp == kBwdWarpLoad) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      // Q_i, then K_0 (all the first S needs), then dO_i, then V_0, K_1, V_1, ...
      const uint32_t fbar = smem_u32(&bars->fixed_full);
      const uint32_t fbar1 = smem_u32(&bars->fixed1_full);
      mbar_arrive_expect_tx(fbar, Cfg::kTileBytes);
#pragma unroll
      for (int b = 0; b < Cfg::kBoxes; ++b)
        tma_load_3d(sbase + Cfg::kSmemFixed0 + b * kBoxBytes, &tm_q, fbar, b * kBoxCols, i * kBlockM, bh);
      bool do_issued = false;
      // K_it and V_it in turn (V_it's slot frees before K_it+1's: dP is done before dQ).
      int issued_k = 0, issued_v = 0;
      for (int it = 0; it < nk; ++it) {
        const int sk = it % Cfg::kDqSlotsK;
        if (!bwd_wait(smem_u32(&bars->stage_empty[sk]), ((it / Cfg::kDqSlotsK) & 1) ^ 1, abort,
                       p.status))
          break;
        const uint32_t kfull = smem_u32(&bars->stage_full[sk]);
        mbar_arrive_expect_tx(kfull, Cfg::kTileBytes);
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_load_3d(k_addr(it) + b * kBoxBytes, &tm_k, kfull, b * kBoxCols, it * kBlockM, bh);
        issued_k = it + 1;
        if (!do_issued) {
          mbar_arrive_expect_tx(fbar1, Cfg::kTileBytes);
#pragma unroll
          for (int b = 0; b < Cfg::kBoxes; ++b)
            tma_load_3d(sbase + Cfg::kSmemFixed1 + b * kBoxBytes, &tm_do, fbar1, b * kBoxCols,
                        i * kBlockM, bh);
          do_issued = true;
        }
        const int sv = it % Cfg::kDqSlotsV;
        if (!bwd_wait(smem_u32(&bars->v_empty[sv]), ((it / Cfg::kDqSlotsV) & 1) ^ 1, abort,
                      p.status))
          break;
        const uint32_t vfull = smem_u32(&bars->v_full[sv]);
        mbar_arrive_expect_tx(vfull, Cfg::kTileBytes);
        issued_v = it + 1;
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b)
          tma_load_3d(v_addr(it) + b * kBoxBytes, &tm_v, vfull, b * kBoxCols, it * kBlockM, bh);
      }
      int no_abort = 0;
      bwd_wait(fbar, 0, &no_abort, p.status);
      if (do_issued) bwd_wait(fbar1, 0, &no_abort, p.status);
      for (int it = max(0, issued_k - Cfg::kDqSlotsK); it < issued_k; ++it)
        bwd_wait(smem_u32(&bars->stage_full[it % Cfg::kDqSlotsK]), (it / Cfg::kDqSlotsK) & 1,
                  &no_abort, p.status);
      for (int it = max(0, issued_v - Cfg::kDqSlotsV); it < issued_v; ++it)
        bwd_wait(smem_u32(&bars->v_full[it % Cfg::kDqSlotsV]), (it / Cfg::kDqSlotsV) & 1,
                 &no_abort, p.status);
    }
  } else if (warp == kBwdWarpMma) {
    constexpr uint32_t kIdescS = idesc_f16kind(kBlockM, kBlockM, false, F16);
    constexpr uint32_t kIdescAcc = idesc_f16kind(kBlockM, D, true, F16);
    const uint64_t dQ = desc_sw128(sbase + Cfg::kSmemFixed0, 16, 1024);   // A of S
    const uint64_t dDO = desc_sw128(sbase + Cfg::kSmemFixed1, 16, 1024);  // A of dP
    const uint32_t tS = tbase + Cfg::kColS, tDP = tbase + Cfg::kColDP, tDQ = tbase + Cfg::kColAcc0;
    auto wait_bar = [&](uint64_t* bar, int parity) {
      const bool r = __all_sync(0xffffffffu, bwd_wait(smem_u32(bar), parity, abort, p.status));
      if (r) tc_fence_after();
      return r;
    };
    auto k_desc = [&](int it, uint32_t lbo) { return desc_sw128(k_addr(it), lbo, 1024); };
    auto v_desc = [&](int it) { return desc_sw128(v_addr(it), 16, 1024); };
    auto wait_k = [&](int it) {
      return wait_bar(&bars->stage_full[it % Cfg::kDqSlotsK], (it / Cfg::kDqSlotsK) & 1);
    };
    auto wait_v = [&](int it) {
      return wait_bar(&bars->v_full[it % Cfg::kDqSlotsV], (it / Cfg::kDqSlotsV) & 1);
    };
    auto release_v = [&](int it) { mma_commit_elect(smem_u32(&bars->v_empty[it % Cfg::kDqSlotsV])); };
    // S = Q_i K_j^T into tS, or dP = dO_i V_j^T into tDP: queries on lanes, keys on
    // columns; the streamed tile is the K-major B operand.
    auto issue_n = [&](uint32_t tD, uint64_t dA, uint64_t dB) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off16 = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss_elect(tD, dA + off16, dB + off16, kIdescS, kk > 0 ? 1u : 0u);
      }
    };
    // Software pipeline on the tensor pipe, per key tile it:
    //   S(it+1) (once the element-wise warps hold S(it) in registers)  |
    //   dQ += dS(it) K_it (dS stored over dP(it))  |  dP(it+1)
    // so the next S is computed while dS(it) is being formed.
    bool ok = wait_bar(&bars->fixed_full, 0) && wait_k(0);
    if (ok) {
      issue_n(tS, dQ, k_desc(0, 16));
      mma_commit_elect(smem_u32(&bars->s_full));
      if ((ok = wait_bar(&bars->fixed1_full, 0) && wait_v(0))) {
        issue_n(tDP, dDO, v_desc(0));
        mma_commit_elect(smem_u32(&bars->dp_full));
        release_v(0);
      }
    }
    for (int it = 0; ok && it < nk; ++it) {
      const bool more = it + 1 < nk;
      if (more) {
        if (!(ok = wait_bar(&bars->p_done, it & 1))) break;
        if (!(ok = wait_k(it + 1))) break;
        issue_n(tS, dQ, k_desc(it + 1, 16));
        mma_commit_elect(smem_u32(&bars->s_full));
      }
      if (!(ok = wait_bar(&bars->ds_ready, it & 1))) break;
      // dQ += dS K_j: dS (16 keys = 8 packed columns per step) from the dP columns.
      const uint64_t dKmn = k_desc(it, kBoxBytes);
#pragma unroll
      for (int kk = 0; kk < kBlockM / 16; ++kk) {
        const uint32_t acol = (kk >> 2) * 64 + (kk & 3) * 8;
        mma_bf16_ts_elect(tDQ, tDP + acol, dKmn + ((kk * 2048) >> 4), kIdescAcc,
                          (it > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_elect(smem_u32(&bars->stage_empty[it % Cfg::kDqSlotsK]));
      if (more) {
        if (!(ok = wait_v(it + 1))) break;
        issue_n(tDP, dDO, v_desc(it + 1));
        mma_commit_elect(smem_u32(&bars->dp_full));
        release_v(it + 1);
      }
    }
    if (ok) mma_commit_elect(smem_u32(&bars->acc_final));
    mma_commit_elect(smem_u32(&bars->mma_drain));
    int no_abort = 0;
    bwd_wait(smem_u32(&bars->mma_drain), 0, &no_abort, p.status);
    __syncwarp();
  } else {
    const int h = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query within the tile
    const int qg = i * kBlockM + r;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + Cfg::kColS, tDP = tbase + lane_off + Cfg::kColDP;
    const float sl2 = p.scale_log2;
    const long long srow = static_cast<long long>(bh) * p.n_pad + qg;
    const float lse2 = p.lse2[srow];
    const float dd = p.dd[srow];
    bool ok = true;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const uint64_t negl2 = f2_pack(-lse2, -lse2);
    const uint64_t negd2 = f2_pack(-dd, -dd);
    for (int it = 0; it < nk; ++it) {
      ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->s_full), it & 1, abort, p.status));
      if (!ok) break;
      tc_fence_after();
      const int key0 = it * kBlockM;
      // Keys past N, and (causal) keys after the query, drop out.
      const bool need_mask = (p.causal && it == i) || key0 + kBlockM > p.N;
      int lim = p.N - 1 - key0;
      if (p.causal) lim = min(lim, qg - key0);
      // P = exp2(S * scale * log2 e - LSE * log2 e), in registers.
      uint64_t pv[32];
      if (!need_mask) {
        // The second half of this warp's S loads while P of the first half is formed.
        uint32_t sr0[32];
        tmem_ld32_wait(tS + 64 * h, sr0);
        uint32_t sr[32];
        tmem_ld32_exp_lse_chunk(tS + 64 * h + 32, sr, sr0, sl2x2, negl2, pv);
        if (it + 1 < nk) {  // S(it) is in registers: the next S may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->p_done));
        }
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2,
                           negl2),
                    x0, x1);
          pv[16 + (c >> 1)] = f2_pack(ex2_approx(x0), ex2_approx(x1));
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = 64 * h + 32 * ch;   // first key (column) of this chunk
          uint32_t sr[32];
          tmem_ld32_wait(tS + c0, sr);
          if (ch == 1 && it + 1 < nk) {  // S(it) is in registers: the next S may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_done));
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2,
                             negl2),
                      x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (need_mask) {
              if (c0 + c > lim) p0 = 0.f;
              if (c0 + c + 1 > lim) p1 = 0.f;
            }
            pv[16 * ch + (c >> 1)] = f2_pack(p0, p1);
          }
        }
      }
      // dS = P * (dP - D), stored (16-bit) over the first half of this warp's dP columns.
      ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->dp_full), it & 1, abort, p.status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * h + 32 * ch;
        uint32_t dr[32];
        tmem_ld32_wait(tDP + c0, dr);
        uint32_t pd[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const uint64_t ds = f2_mul(
              pv[16 * ch + (c >> 1)],
              f2_add(f2_pack(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), negd2));
          float d0, d1;
          f2_unpack(ds, d0, d1);
          pd[c >> 1] = pack_elem2<F16>(d0, d1);
        }
        tmem_st16(tDP + 64 * h + 16 * ch, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->ds_ready));
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, bwd_wait(smem_u32(&bars->acc_final), 0, abort, p.status));
    }
    if (ok) {
      tc_fence_after();
      uint8_t* dq_row = static_cast<uint8_t*>(p.dq) + (static_cast<long long>(bh) * p.N + qg) * D * 2;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = h * (D / 2) + 32 * c;
        uint32_t a[32];
        tmem_ld32_wait(tbase + lane_off + Cfg::kColAcc0 + col, a);
        if (qg < p.N) store_row32<F16>(dq_row + col * 2, a, p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, Cfg::kTmemCols);
  }
}

// dQ = scale * accumulator, rounded to 16 bits, for the N real rows of each head; a thread
// takes 8 columns of one row (two 16-byte loads, one 16-byte store).
template <bool F16>
__global__ void __launch_bounds__(256) attn_bwd_dq_finalize_kernel(const float* __restrict__ acc,
                                                                   uint16_t* __restrict__ dq,
                                                                   long long rows, int N,
                                                                   int n_pad, float scale) {
  const long long step = static_cast<long long>(gridDim.x) * 256;
  for (long long t = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; t < rows * 8;
       t += step) {
    const long long row = t >> 3;  // bh * N + q
    const int c8 = static_cast<int>(t & 7) * 8;
    const long long bh = row / N;
    const long long q = row - bh * N;
    const float4* src = reinterpret_cast<const float4*>(acc + (bh * n_pad + q) * 64 + c8);
    const float4 a = src[0], b = src[1];
    *reinterpret_cast<uint4*>(dq + row * 64 + c8) = make_uint4(
        pack_elem2<F16>(a.x * scale, a.y * scale), pack_elem2<F16>(a.z * scale, a.w * scale),
        pack_elem2<F16>(b.x * scale, b.y * scale), pack_elem2<F16>(b.z * scale, b.w * scale));
  }
}

template <int D, bool F16>
cudaError_t launch_attn_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq_acc,
                            const CUtensorMap& taug, const void* o, const void* dout,
                            const float* lse, float* ws, const AttnBwdParams& p0,
                            cudaStream_t stream, const BwdFork* fork) {
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(sizeof(AttnBwdBarriers) <= 512, "barrier block");
  constexpr bool kFused = (D == 64);
  AttnBwdParams p = p0;
  const long long rows = static_cast<long long>(p.BH) * p.n_pad;
  // Workspace: d = 128 LSE * log2(e) and D per row, then the statistics terms (16 bf16
  // per row); d = 64 the terms and then the dQ accumulator (64 fp32 per row).
  p.lse2 = kFused ? nullptr : ws;
  p.dd = kFused ? nullptr : ws + rows;
  p.aug = reinterpret_cast<uint16_t*>(kFused ? ws : ws + 2 * rows);
  p.dq_acc = kFused ? ws + 8 * rows : nullptr;
  attn_bwd_prep_kernel<D, F16><<<static_cast<unsigned>((rows + 8 * kPrepRows<D> - 1) / (8 * kPrepRows<D>)),
                                 256, 0, stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse,
      const_cast<float*>(p.lse2), const_cast<float*>(p.dd), p.BH, p.N, p.n_pad, p.dq_acc, p.aug,
      1.0f / p.scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.BH) * p.nblk);
  if constexpr (kFused) {
    // One pass over the key tiles, then dQ from its accumulator.
    using C1 = AttnBwd1Cfg;
    static_assert(C1::kSmemBytes <= 227 * 1024, "shared memory");
    if ((e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, F16, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, C1::kSmemBytes)) !=
        cudaSuccess)
      return e;
    attn_bwd_dkdv_kernel<D, F16, true><<<grid, kBwdThreads, C1::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, tdq_acc, taug, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long out_rows = static_cast<long long>(p.BH) * p.N;
    const long long fin_blocks = std::min<long long>((out_rows * 8 + 255) / 256, 1LL << 20);
    attn_bwd_dq_finalize_kernel<F16><<<static_cast<unsigned>(fin_blocks), 256, 0, stream>>>(
        p.dq_acc, static_cast<uint16_t*>(p.dq), out_rows, p.N, p.n_pad, p.scale);
    return cudaGetLastError();
  } else {
    // Two passes: dK, dV key-outer on `stream`, dQ query-outer on the side stream.
    using Cfg = AttnBwdCfg<D>;
    static_assert(Cfg::kSmemBytes <= 227 * 1024 && Cfg::kDqSmemBytes <= 227 * 1024,
                  "shared memory");
    if ((e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, F16, false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes)) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, F16>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfg::kDqSmemBytes)) != cudaSuccess)
      return e;
    // The fork point is the prep's completion, recorded before the key-outer launch.
    if (fork != nullptr && (e = cudaEventRecord(fork->fork, stream)) != cudaSuccess) return e;
    attn_bwd_dkdv_kernel<D, F16, false><<<grid, kBwdThreads, Cfg::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, tdq_acc, taug, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (fork == nullptr) {
      attn_bwd_dq_kernel<D, F16><<<grid, kBwdThreads, Cfg::kDqSmemBytes, stream>>>(tq, tk, tv,
                                                                                  tdo, p);
      return cudaGetLastError();
    }
    if ((e = cudaStreamWaitEvent(fork->side, fork->fork, 0)) != cudaSuccess) return e;
    attn_bwd_dq_kernel<D, F16><<<grid, kBwdThreads, Cfg::kDqSmemBytes, fork->side>>>(
        tq, tk, tv, tdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaEventRecord(fork->join, fork->side)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, fork->join, 0);
  }
}

}  // namespace osfa
