// combine.cu -- merge of split-KV partial results into O and LSE.
//
// Each split s of a query row holds O_s = (sum over its keys of p v) / l_s and
// LSE_s = m_s + ln l_s.  Results normalised separately cannot be averaged (lihaoran.work
// FlashAttention note, section "为什么不能平均各块的softmax"); they are brought to a common
// reference M = max_s LSE_s with the merge rule of "Softmax 数值稳定性与 IO-Aware
// Attention", §4.1: w_s = exp(LSE_s - M) (0 for an empty split, LSE_s = -inf),
// O = sum_s w_s O_s / sum_s w_s, LSE = M + ln sum_s w_s.
//
// One warp per query row; lane t holds output columns [t * D/32, (t+1) * D/32).  The
// partials are read once (HBM-bound: splits * (D + 1) * 4 bytes per row).
//
// The kernel is a programmatic dependent of the split-mode attention launch: its blocks
// may be scheduled as the attention blocks drain (the attention kernel signals
// griddepcontrol.launch_dependents when it starts), and griddepcontrol.wait holds them
// until the whole attention grid has completed and its partials are visible.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace osfa {
namespace {

template <int D, bool F16>
__global__ void __launch_bounds__(256)
    splitkv_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                           void* __restrict__ o, float* __restrict__ lse, int BH, int N,
                           int n_pad, int splits) {
  constexpr int kPer = D / 32;  // columns per lane: 2 or 4
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(BH) * N) return;
  const int bh = static_cast<int>(row / N);
  const int i = static_cast<int>(row % N);
  auto part = [&](int s) { return (static_cast<int64_t>(s) * BH + bh) * n_pad + i; };

  float M = -INFINITY;
  for (int s = lane; s < splits; s += 32) M = fmaxf(M, ws_lse[part(s)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float acc[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ls = ws_lse[part(s)];
    if (ls == -INFINITY) continue;  // empty split: weight 0
    const float w = __expf(ls - M);
    wsum += w;
    const float* src = ws_o + part(s) * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
    }
  }
  const float inv = 1.0f / wsum;
  uint32_t packed[kPer / 2];
#pragma unroll
  for (int c = 0; c < kPer / 2; ++c) {
    const float lo = acc[2 * c] * inv, hi = acc[2 * c + 1] * inv;
    uint32_t r;
    if constexpr (F16)
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    packed[c] = r;
  }
  uint16_t* dst = static_cast<uint16_t*>(o) + row * D + lane * kPer;
  if constexpr (kPer == 4)
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  else
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  if (lse != nullptr && lane == 0) lse[row] = M + logf(wsum);
}

}  // namespace

cudaError_t launch_splitkv_combine(const float* ws_o, const float* ws_lse, void* o, float* lse,
                                   int BH, int N, int n_pad, int d, int splits, bool f16,
                                   cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (d == 64)
    return f16 ? cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<64, true>, ws_o, ws_lse, o, lse, BH, N, n_pad, splits)
               : cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<64, false>, ws_o, ws_lse, o, lse, BH, N, n_pad, splits);
  return f16 ? cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<128, true>, ws_o, ws_lse, o, lse, BH, N, n_pad, splits)
             : cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<128, false>, ws_o, ws_lse, o, lse, BH, N, n_pad, splits);
}

}  // namespace osfa
