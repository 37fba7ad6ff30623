// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers with bounded waits,
// TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, commit, ld/st) and a few
// scalar helpers.  Written from the PTX ISA's descriptions of these instructions.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace osfa {

// Status word bits (the word lives in static device memory of the library).
enum : unsigned { kStatusTimeout = 1u };

// Bounded waits give up after this many nanoseconds of %globaltimer.  A correct
// run never waits on one barrier for more than a few milliseconds.
#ifndef OSFA_WAIT_LIMIT_NS
#define OSFA_WAIT_LIMIT_NS 1000000000ull
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with parity `parity` of barrier `bar` has completed.
// Gives up when `*abort` becomes non-zero (another role of the block gave up) or
// after `limit_ns`; on a time-out it records kStatusTimeout in `*status`, sets
// `*abort` and returns false.  Never traps.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned* status,
                                          uint64_t limit_ns = OSFA_WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, kStatusTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_group_0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Waits until every committed bulk copy of this thread has finished READING its source
// (shared memory may then be reused or released); the writes complete asynchronously,
// before the kernel is complete.
__device__ __forceinline__ void bulk_wait_group_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA store) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-uniform issue: every lane of the warp executes these with the same operands
// and elect.sync lets exactly one lane issue the instruction.  Keeping the issue loop
// warp-uniform keeps its operands in uniform registers; a single-lane branch around
// the loop made each MMA cost more issue cycles than the tensor core spends on it.

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_bf16_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_bf16_ts_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 4 tcgen05.mma (A and B from shared memory) into one accumulator under a single
// elect.sync: a[k], b[k] are the k-th operand descriptors; the first product accumulates
// when `acc` is non-zero, the others always.
__device__ __forceinline__ void mma_ss4_elect(uint32_t d_tmem, const uint64_t* a, const uint64_t* b,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %2, 0;\n\t"
      "setp.eq.b32 t, %2, %2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %1, t;\n\t"
      "}"
      :: "r"(d_tmem), "r"(idesc), "r"(acc), "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3])
      : "memory");
}

// 8 tcgen05.mma (A and B from shared memory) into one accumulator under a single
// elect.sync: a[k], b[k] are the k-th operand descriptors; the first product accumulates
// when `acc` is non-zero, the others always.
__device__ __forceinline__ void mma_ss8_elect(uint32_t d_tmem, const uint64_t* a, const uint64_t* b,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %2, 0;\n\t"
      "setp.eq.b32 t, %2, %2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %11, %12, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %13, %14, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %15, %16, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %17, %18, %1, t;\n\t"
      "}"
      :: "r"(d_tmem), "r"(idesc), "r"(acc), "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]), "l"(a[4]), "l"(b[4]), "l"(a[5]), "l"(b[5]), "l"(a[6]), "l"(b[6]), "l"(a[7]), "l"(b[7])
      : "memory");
}

// 8 tcgen05.mma (A from TMEM, B from shared memory) into one accumulator under a single
// elect.sync; a[k]: TMEM address of the k-th A operand, b[k]: descriptor of the k-th B.
__device__ __forceinline__ void mma_ts8_elect(uint32_t d_tmem, const uint32_t* a, const uint64_t* b,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %2, 0;\n\t"
      "setp.eq.b32 t, %2, %2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%11], %12, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%13], %14, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%15], %16, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%17], %18, %1, t;\n\t"
      "}"
      :: "r"(d_tmem), "r"(idesc), "r"(acc), "r"(a[0]), "l"(b[0]), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]), "l"(b[3]), "r"(a[4]), "l"(b[4]), "r"(a[5]), "l"(b[5]), "r"(a[6]), "l"(b[6]), "r"(a[7]), "l"(b[7])
      : "memory");
}


// 4 tcgen05.mma (A from TMEM, B from shared memory) into one accumulator under a single
// elect.sync; a[k]: TMEM address of the k-th A operand, b[k]: descriptor of the k-th B.
__device__ __forceinline__ void mma_ts4_elect(uint32_t d_tmem, const uint32_t* a, const uint64_t* b,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %2, 0;\n\t"
      "setp.eq.b32 t, %2, %2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %1, t;\n\t"
      "}"
      :: "r"(d_tmem), "r"(idesc), "r"(acc), "r"(a[0]), "l"(b[0]), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]), "l"(b[3])
      : "memory");
}

// 16 tcgen05.mma (A from TMEM, B from shared memory) into one accumulator under a single
// elect.sync; a[k]: TMEM address of the k-th A operand, b[k]: descriptor of the k-th B.
__device__ __forceinline__ void mma_ts16_elect(uint32_t d_tmem, const uint32_t* a, const uint64_t* b,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %2, 0;\n\t"
      "setp.eq.b32 t, %2, %2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%11], %12, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%13], %14, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%15], %16, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%17], %18, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%19], %20, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%21], %22, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%23], %24, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%25], %26, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%27], %28, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%29], %30, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%31], %32, %1, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%33], %34, %1, t;\n\t"
      "}"
      :: "r"(d_tmem), "r"(idesc), "r"(acc), "r"(a[0]), "l"(b[0]), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]), "l"(b[3]), "r"(a[4]), "l"(b[4]), "r"(a[5]), "l"(b[5]), "r"(a[6]), "l"(b[6]), "r"(a[7]), "l"(b[7]), "r"(a[8]), "l"(b[8]), "r"(a[9]), "l"(b[9]), "r"(a[10]), "l"(b[10]), "r"(a[11]), "l"(b[11]), "r"(a[12]), "l"(b[12]), "r"(a[13]), "l"(b[13]), "r"(a[14]), "l"(b[14]), "r"(a[15]), "l"(b[15])
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation the electing thread issued before
// has completed (one lane of the warp, elected as for the MMAs).
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Loads 32 lanes x 32 consecutive 32-bit TMEM columns and waits for them: thread i
// of the warp gets lane (taddr.lane + i), columns taddr.col .. taddr.col + 31.  The
// load and its wait sit in one asm statement so that no use of r[] can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Loads 32 lanes x 128 consecutive 32-bit TMEM columns and waits for them: thread i of
// the warp gets lane (taddr.lane + i), columns taddr.col .. taddr.col + 127 (the load and
// its wait in one asm statement, so that no use of r[] can be scheduled before the data
// has arrived).  Also returns in `mx` the maximum of the 128 values this thread loaded
// (tcgen05.ld.red, sm_103a: the reduction is done by the load, not by instructions of
// the thread; -inf values take part as the ordinary smallest value).
__device__ __forceinline__ void tmem_ld128_max_wait(uint32_t taddr, uint32_t* r, float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x128.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, %128, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127]), "=f"(mx)
      : "r"(taddr)
      : "memory");
}

// 64-column form of tmem_ld128_max_wait.
__device__ __forceinline__ void tmem_ld64_max_wait(uint32_t taddr, uint32_t* r, float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x64.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, %64, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=f"(mx)
      : "r"(taddr)
      : "memory");
}

// Stores 32 lanes x 32 consecutive 32-bit TMEM columns (layout as the load); complete
// after tmem_wait_st().
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Stores 32 lanes x 16 consecutive 32-bit TMEM columns; complete after tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Register-budget hand-off between warpgroups (all four warps of a warpgroup execute
// the same one): the softmax warpgroups take registers the issue warps give back.
template <int N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- scalar helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packs two fp32 into bf16x2 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed pairs of fp32 (sm_100 family: one instruction works on both halves).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace osfa
