// attn_f32.cu -- fp32 attention forward on CUDA cores (any head dimension 1..128).
//
// The same online-softmax tile loop as the tensor-core kernel ("Softmax 数值稳定性与
// IO-Aware Attention：从在线归一化到 FlashAttention", §七), in fp32 throughout: for each
// query row, m = -inf, l = 0, O = 0; for each tile of 32 keys S = scale q K^T, m_new =
// max(m, rowmax S), P = exp(S - m_new), alpha = exp(m - m_new), l = alpha l + rowsum P,
// O = alpha O + P V; finally O = O / l, LSE = m + ln l.
//
// One warp owns one query row at a time: lane t scores key (tile + t), the warp
// reduces max and sum with shuffles, and lane t accumulates output dimensions
// t, t + 32, t + 64, t + 96.  A block of 4 warps shares each K/V tile through shared
// memory across kRowsPerBlock query rows.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace osfa {

namespace {

constexpr int kKeysPerTile = 32;
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;
constexpr int kMaxD = 128;

__global__ void __launch_bounds__(kWarps * 32)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, float* __restrict__ o,
                        float* __restrict__ lse, int N, int d, float scale, int causal) {
  __shared__ float sk[kKeysPerTile][kMaxD + 1];  // +1: lane t reads row t, conflict-free
  __shared__ float sv[kKeysPerTile][kMaxD];
  __shared__ float sq[kRowsPerBlock][kMaxD];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nrb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t bh = blockIdx.x / nrb;
  const int row0 = (blockIdx.x % nrb) * kRowsPerBlock;
  const float* qh = q + bh * N * d;
  const float* kh = k + bh * N * d;
  const float* vh = v + bh * N * d;

  for (int i = threadIdx.x; i < kRowsPerBlock * d; i += blockDim.x) {
    const int r = i / d, c = i % d;
    sq[r][c] = (row0 + r < N) ? qh[static_cast<int64_t>(row0 + r) * d + c] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][4];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  }

  const int last_row = min(N - 1, row0 + kRowsPerBlock - 1);
  const int key_end = causal ? last_row + 1 : N;
  for (int key0 = 0; key0 < key_end; key0 += kKeysPerTile) {
    __syncthreads();
    for (int i = threadIdx.x; i < kKeysPerTile * d; i += blockDim.x) {
      const int r = i / d, c = i % d;
      const bool in = key0 + r < N;
      sk[r][c] = in ? kh[static_cast<int64_t>(key0 + r) * d + c] : 0.f;
      sv[r][c] = in ? vh[static_cast<int64_t>(key0 + r) * d + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int lr = warp * kRowsPerWarp + r;
      const int row = row0 + lr;
      const int key = key0 + lane;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s = fmaf(sq[lr][c], sk[lane][c], s);
      s *= scale;
      const bool visible = key < N && (!causal || key <= row);
      s = visible ? s : -INFINITY;
      float tmax = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float m_new = fmaxf(m[r], tmax);
      if (m_new == -INFINITY) continue;  // every key of this tile is masked for this row
      const float p = expf(s - m_new);   // 0 for masked keys
      const float alpha = expf(m[r] - m_new);
      float psum = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l[r] = alpha * l[r] + psum;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] *= alpha;
      for (int j = 0; j < kKeysPerTile; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = lane + 32 * c;
          if (col < d) acc[r][c] = fmaf(pj, sv[j][col], acc[r][c]);
        }
      }
      m[r] = m_new;
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int row = row0 + warp * kRowsPerWarp + r;
    if (row >= N) continue;
    const float inv = 1.0f / l[r];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int col = lane + 32 * c;
      if (col < d) o[(bh * N + row) * d + col] = acc[r][c] * inv;
    }
    if (lse != nullptr && lane == 0) lse[bh * N + row] = m[r] + logf(l[r]);
  }
}

}  // namespace

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int BH, int N, int d, float scale, int causal, cudaStream_t stream) {
  const long long grid = static_cast<long long>((N + kRowsPerBlock - 1) / kRowsPerBlock) * BH;
  attn_fwd_f32_kernel<<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(q, k, v, o, lse, N, d, scale, causal);
  return cudaGetLastError();
}

}  // namespace osfa
