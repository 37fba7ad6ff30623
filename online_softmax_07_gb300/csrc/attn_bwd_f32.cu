// attn_bwd_f32.cu -- fp32 attention backward on CUDA cores (any head dimension 1..128).
//
// The gradients of the fp32 forward (attn_f32.cu) for an upstream dO, recomputing the
// probabilities from the kept LSE ("Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到
// FlashAttention", §7.2), in fp32 throughout:
//   P_ij = exp(scale q_i . k_j - LSE_i),  dP_ij = dO_i . v_j,  D_i = dO_i . O_i,
//   dS_ij = P_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij k_j,
//   dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i.
// Two passes, no atomics: a warp per key row accumulates dK_j and dV_j over the queries
// that see the key; a warp per query row accumulates dQ_i over the keys it sees.  Lane t
// holds dimensions t, t + 32, t + 64, t + 96; dot products are reduced with shuffles.
// This path serves the fp32 configuration (small problems); the bf16/fp16 backward runs
// on the tensor cores (attn_bwd_impl.cuh).
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace osfa {

namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
  return x;
}

// Loads row r of a [N, d] matrix into the lane's four slots (0 past d).
__device__ __forceinline__ void load_row(const float* base, int d, float* out, int lane) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = lane + 32 * c;
    out[c] = col < d ? base[col] : 0.f;
  }
}

__device__ __forceinline__ float dot4(const float* a, const float* b) {
  return warp_sum(a[0] * b[0] + a[1] * b[1] + a[2] * b[2] + a[3] * b[3]);
}

// D_i = dO_i . O_i, one warp per row.
__global__ void __launch_bounds__(kWarps * 32)
    bwd_f32_d_kernel(const float* __restrict__ o, const float* __restrict__ dout,
                     float* __restrict__ dd, long long rows, int d) {
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float a[4], b[4];
  load_row(o + row * d, d, a, lane);
  load_row(dout + row * d, d, b, lane);
  const float s = dot4(a, b);
  if (lane == 0) dd[row] = s;
}

// dK_j, dV_j: warp per key row j of head bh.
__global__ void __launch_bounds__(kWarps * 32)
    bwd_f32_dkdv_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, const float* __restrict__ dout,
                        const float* __restrict__ lse, const float* __restrict__ dd,
                        float* __restrict__ dk, float* __restrict__ dv, long long BH, int N,
                        int d, float scale, int causal) {
  const long long gw = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= BH * N) return;
  const long long bh = gw / N;
  const int j = static_cast<int>(gw - bh * N);
  const float* qh = q + bh * N * d;
  const float* doh = dout + bh * N * d;
  float kj[4], vj[4], ak[4] = {0.f, 0.f, 0.f, 0.f}, av[4] = {0.f, 0.f, 0.f, 0.f};
  load_row(k + gw * d, d, kj, lane);
  load_row(v + gw * d, d, vj, lane);
  for (int i = causal ? j : 0; i < N; ++i) {
    float qi[4], gi[4];
    load_row(qh + static_cast<long long>(i) * d, d, qi, lane);
    load_row(doh + static_cast<long long>(i) * d, d, gi, lane);
    const float pij = expf(scale * dot4(qi, kj) - lse[bh * N + i]);
    const float ds = pij * (dot4(gi, vj) - dd[bh * N + i]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      av[c] = fmaf(pij, gi[c], av[c]);
      ak[c] = fmaf(ds, qi[c], ak[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = lane + 32 * c;
    if (col < d) {
      dv[gw * d + col] = av[c];
      dk[gw * d + col] = scale * ak[c];
    }
  }
}

// dQ_i: warp per query row i of head bh.
__global__ void __launch_bounds__(kWarps * 32)
    bwd_f32_dq_kernel(const float* __restrict__ q, const float* __restrict__ k,
                      const float* __restrict__ v, const float* __restrict__ dout,
                      const float* __restrict__ lse, const float* __restrict__ dd,
                      float* __restrict__ dq, long long BH, int N, int d, float scale,
                      int causal) {
  const long long gw = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= BH * N) return;
  const long long bh = gw / N;
  const int i = static_cast<int>(gw - bh * N);
  const float* kh = k + bh * N * d;
  const float* vh = v + bh * N * d;
  float qi[4], gi[4], aq[4] = {0.f, 0.f, 0.f, 0.f};
  load_row(q + gw * d, d, qi, lane);
  load_row(dout + gw * d, d, gi, lane);
  const float lse_i = lse[gw];
  const float dd_i = dd[gw];
  const int jend = causal ? i + 1 : N;
  for (int j = 0; j < jend; ++j) {
    float kj[4], vj[4];
    load_row(kh + static_cast<long long>(j) * d, d, kj, lane);
    load_row(vh + static_cast<long long>(j) * d, d, vj, lane);
    const float pij = expf(scale * dot4(qi, kj) - lse_i);
    const float ds = pij * (dot4(gi, vj) - dd_i);
#pragma unroll
    for (int c = 0; c < 4; ++c) aq[c] = fmaf(ds, kj[c], aq[c]);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = lane + 32 * c;
    if (col < d) dq[gw * d + col] = scale * aq[c];
  }
}

}  // namespace

cudaError_t launch_attn_bwd_f32(const float* q, const float* k, const float* v, const float* o,
                                const float* lse, const float* dout, float* dq, float* dk,
                                float* dv, float* dd, int BH, int N, int d, float scale,
                                int causal, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  const unsigned grid = static_cast<unsigned>((rows + kWarps - 1) / kWarps);
  bwd_f32_d_kernel<<<grid, kWarps * 32, 0, stream>>>(o, dout, dd, rows, d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_f32_dkdv_kernel<<<grid, kWarps * 32, 0, stream>>>(q, k, v, dout, lse, dd, dk, dv, BH, N, d,
                                                        scale, causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_f32_dq_kernel<<<grid, kWarps * 32, 0, stream>>>(q, k, v, dout, lse, dd, dq, BH, N, d, scale,
                                                      causal);
  return cudaGetLastError();
}

}  // namespace osfa
