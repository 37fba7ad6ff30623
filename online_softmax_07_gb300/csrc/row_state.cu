// row_state.cu -- per-row online-softmax state (m, l) of an fp32 [rows, len] array.
//
// "Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention", §4.2: each
// thread reduces its own elements to a local state (m, l); the states are merged by
// warp shuffles, each warp's result goes through shared memory, and the first warp
// merges the block's states.  The merge is §4.1's m = max(m_a, m_b),
// l = l_a e^(m_a - m) + l_b e^(m_b - m); an empty side (m = -inf) contributes nothing.
//
// The work is bound by HBM bandwidth (the page notes that softmax is limited by
// memory access and reduction, not by the exponential), so the kernel streams each
// row once with 16-byte loads, several in flight per thread.  A row may start at any
// float offset (len need not be a multiple of 4): the first elements up to the next
// 16-byte boundary and the last ragged elements are read one by one.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace osfa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBlockThreads = 512;
constexpr int kUnroll = 8;  // 16-byte loads in flight per thread per batch

struct State {
  float m;
  float l;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(x - m) with the difference taken first in fp32 (exact when x and m are close,
// which keeps rows such as 1000 + N(0, 9) accurate).
__device__ __forceinline__ float exp_diff(float x, float m) { return ex2f((x - m) * kLog2e); }

__device__ __forceinline__ State merge(State a, State b) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  if (a.m >= b.m) return {a.m, a.l + b.l * exp_diff(b.m, a.m)};
  return {b.m, b.l + a.l * exp_diff(a.m, b.m)};
}

__device__ __forceinline__ State warp_merge(State s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    State o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
    o.l = __shfl_xor_sync(0xffffffffu, s.l, off);
    s = merge(s, o);
  }
  return s;
}

// Folds a batch of values into the running state: one max over the batch, then one
// rescale of l (the per-element recurrence of §四 grouped kUnroll * 4 at a time).
template <int NV>
__device__ __forceinline__ void fold(State& st, const float (&x)[NV], int count) {
  float bm = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (i < count) bm = fmaxf(bm, x[i]);
  if (bm == -INFINITY) return;
  const float m_new = fmaxf(st.m, bm);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (i < count) acc[i & 3] += exp_diff(x[i], m_new);
  const float scale_old = (st.m == -INFINITY) ? 0.f : exp_diff(st.m, m_new);
  st.l = st.l * scale_old + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
  st.m = m_new;
}

// One block per row.
__global__ void __launch_bounds__(kBlockThreads)
    row_state_block_kernel(const float* __restrict__ x, float* __restrict__ m_out,
                           float* __restrict__ l_out, int len) {
  const int64_t row = blockIdx.x;
  const float* xr = x + row * static_cast<int64_t>(len);
  const int tid = threadIdx.x;
  // Elements before the first 16-byte boundary of this row.
  const int head = min(len, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(xr) & 15)) & 15) >> 2));
  const int nvec = (len - head) >> 2;
  const int tail0 = head + 4 * nvec;
  const float4* xv = reinterpret_cast<const float4*>(xr + head);

  State st = {-INFINITY, 0.f};
  {
    float e[1];
    // head and tail elements (at most 3 + 3), one per thread
    const int extra = head + (len - tail0);
    if (tid < extra) {
      e[0] = xr[tid < head ? tid : tail0 + (tid - head)];
      fold<1>(st, e, 1);
    }
  }
  for (int base = 0; base < nvec; base += kUnroll * kBlockThreads) {
    float v[4 * kUnroll];
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kBlockThreads + tid;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nvec) {
        f = __ldcs(xv + i);
        cnt = 4 * (u + 1);
      }
      v[4 * u] = f.x;
      v[4 * u + 1] = f.y;
      v[4 * u + 2] = f.z;
      v[4 * u + 3] = f.w;
    }
    fold<4 * kUnroll>(st, v, cnt);
  }

  st = warp_merge(st);
  __shared__ State warp_states[kBlockThreads / 32];
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) warp_states[warp] = st;
  __syncthreads();
  if (warp == 0) {
    st = (lane < kBlockThreads / 32) ? warp_states[lane] : State{-INFINITY, 0.f};
    st = warp_merge(st);
    if (lane == 0) {
      m_out[row] = st.m;
      l_out[row] = st.l;
    }
  }
}

// One warp per row, for short rows.
__global__ void __launch_bounds__(256)
    row_state_warp_kernel(const float* __restrict__ x, float* __restrict__ m_out,
                          float* __restrict__ l_out, int rows, int len) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* xr = x + row * static_cast<int64_t>(len);
  State st = {-INFINITY, 0.f};
  for (int base = 0; base < len; base += 32 * 8) {
    float v[8];
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * 32 + lane;
      v[u] = 0.f;
      if (i < len) {
        v[u] = __ldcs(xr + i);
        cnt = u + 1;
      }
    }
    fold<8>(st, v, cnt);
  }
  st = warp_merge(st);
  if (lane == 0) {
    m_out[row] = st.m;
    l_out[row] = st.l;
  }
}

// ---------------------------------------------------------------------------------------
// Normalised row softmax y = exp(x - m) / l ("Softmax 数值稳定性与 IO-Aware Attention", §三,
// pass three), with the state (m, l) from the same reduction as above.

// Long rows, low registers: pass one streams the row for (m, l); pass two reads it
// again (from L2: the row was just read and only ~rows-in-flight x len x 4 bytes are
// live) and writes y.  512-thread blocks (several per SM) keep enough loads in flight:
// on 4096 x 32768 they reach the measured copy bandwidth, where 256-thread blocks
// stayed at 86 % of it and 1024-thread blocks at 84 %.
constexpr int kL2Threads = 512;

__global__ void __launch_bounds__(kL2Threads)
    softmax_rows_l2_kernel(const float* x, float* y, float* __restrict__ m_out,
                           float* __restrict__ l_out, int len) {  // y may alias x
  __shared__ State warp_states[kL2Threads / 32];
  const int64_t row = blockIdx.x;
  const float* xr = x + row * static_cast<int64_t>(len);
  float* yr = y + row * static_cast<int64_t>(len);
  const int tid = threadIdx.x;
  const int head =
      min(len, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(xr) & 15)) & 15) >> 2));
  const int nvec = (len - head) >> 2;
  const int tail0 = head + 4 * nvec;
  const int extra = head + (len - tail0);
  const float4* xv = reinterpret_cast<const float4*>(xr + head);
  const bool y_vec = ((reinterpret_cast<uintptr_t>(yr) ^ reinterpret_cast<uintptr_t>(xr)) & 15) == 0;

  State st = {-INFINITY, 0.f};
  float e0 = 0.f;
  if (tid < extra) {
    e0 = xr[tid < head ? tid : tail0 + (tid - head)];
    float e[1] = {e0};
    fold<1>(st, e, 1);
  }
  for (int base = 0; base < nvec; base += kUnroll * kL2Threads) {
    float v[4 * kUnroll];
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kL2Threads + tid;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nvec) {
        f = xv[i];
        cnt = 4 * (u + 1);
      }
      v[4 * u] = f.x;
      v[4 * u + 1] = f.y;
      v[4 * u + 2] = f.z;
      v[4 * u + 3] = f.w;
    }
    fold<4 * kUnroll>(st, v, cnt);
  }
  // block merge
  st = warp_merge(st);
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) warp_states[warp] = st;
  __syncthreads();
  st = (lane < kL2Threads / 32) ? warp_states[lane] : State{-INFINITY, 0.f};
  st = warp_merge(st);
  if (tid == 0) {
    if (m_out != nullptr) m_out[row] = st.m;
    if (l_out != nullptr) l_out[row] = st.l;
  }
  const float m = st.m, inv_l = 1.0f / st.l;
  auto out = [&](float xv_) { return exp_diff(xv_, m) * inv_l; };
  if (tid < extra) yr[tid < head ? tid : tail0 + (tid - head)] = out(e0);
  float* yv = yr + head;
  for (int base = 0; base < nvec; base += kUnroll * kL2Threads) {
    float4 f[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kL2Threads + tid;
      if (i < nvec) f[u] = __ldcs(xv + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kL2Threads + tid;
      if (i >= nvec) continue;
      const float4 r = make_float4(out(f[u].x), out(f[u].y), out(f[u].z), out(f[u].w));
      if (y_vec) {
        __stcs(reinterpret_cast<float4*>(yv) + i, r);
      } else {
        yv[4 * i] = r.x;
        yv[4 * i + 1] = r.y;
        yv[4 * i + 2] = r.z;
        yv[4 * i + 3] = r.w;
      }
    }
  }
}

// One warp per row, for short rows: the row stays in registers (up to 32 per lane).
__global__ void __launch_bounds__(256)
    softmax_rows_warp_kernel(const float* x, float* y,  // y may alias x
                             float* __restrict__ m_out, float* __restrict__ l_out, int rows,
                             int len) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* xr = x + row * static_cast<int64_t>(len);
  float* yr = y + row * static_cast<int64_t>(len);
  float v[32];
  int cnt = 0;
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    const int i = u * 32 + lane;
    v[u] = 0.f;
    if (i < len) {
      v[u] = __ldcs(xr + i);
      cnt = u + 1;
    }
  }
  State st = {-INFINITY, 0.f};
  fold<32>(st, v, cnt);
  st = warp_merge(st);
  if (lane == 0) {
    if (m_out != nullptr) m_out[row] = st.m;
    if (l_out != nullptr) l_out[row] = st.l;
  }
  const float inv_l = 1.0f / st.l;
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    const int i = u * 32 + lane;
    if (i < len) __stcs(yr + i, exp_diff(v[u], st.m) * inv_l);
  }
}

}  // namespace

cudaError_t launch_row_state(const float* x, float* m_out, float* l_out, int rows, int len,
                             cudaStream_t stream) {
  if (len <= 1024) {
    const unsigned grid = static_cast<unsigned>((static_cast<long long>(rows) + 7) / 8);
    row_state_warp_kernel<<<grid, 256, 0, stream>>>(x, m_out, l_out, rows, len);
  } else {
    row_state_block_kernel<<<static_cast<unsigned>(rows), kBlockThreads, 0, stream>>>(x, m_out,
                                                                                     l_out, len);
  }
  return cudaGetLastError();
}

cudaError_t launch_softmax_rows(const float* x, float* y, float* m_out, float* l_out, int rows,
                                int len, cudaStream_t stream) {
  if (len <= 1024) {
    const unsigned grid = static_cast<unsigned>((static_cast<long long>(rows) + 7) / 8);
    softmax_rows_warp_kernel<<<grid, 256, 0, stream>>>(x, y, m_out, l_out, rows, len);
  } else {
    softmax_rows_l2_kernel<<<static_cast<unsigned>(rows), kL2Threads, 0, stream>>>(
        x, y, m_out, l_out, len);
  }
  return cudaGetLastError();
}

}  // namespace osfa
