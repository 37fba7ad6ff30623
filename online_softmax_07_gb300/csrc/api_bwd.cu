// api_bwd.cu -- the backward entry points declared in include/fa.h: argument checks,
// TMA descriptors and dispatch to the three backward launches (attn_bwd_impl.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_bwd.cuh"
#include "fa.h"
#include "host_util.h"
#include "kernels.h"

namespace osfa {
namespace {

long long bwd_n_pad(int N) { return (static_cast<long long>(N) + kBlockM - 1) / kBlockM * kBlockM; }

// Per (head, padded query row): the tensor-core path keeps fp32 LSE * log2(e) and D at
// d = 128 (8 bytes), and at d = 64 its bf16 statistics terms and fp32 dQ accumulator
// (32 + 256 bytes); the fp32 path needs D for each real row (B * H * N floats), within 8
// bytes a row.
// 0 for sizes fa_bwd rejects (more than INT_MAX tiles).
long long bwd_ws_bytes(long long BH, int N, int d, fa_dtype dtype) {
  const long long n_pad = bwd_n_pad(N);
  if (BH * (n_pad / kBlockM) > INT_MAX) return 0;
  if (dtype == FA_F32) return 2 * BH * n_pad * 4;
  return bwd_tc_ws_bytes(BH, n_pad, d);
}

// TMA map of the d = 64 dQ accumulator: [BH, n_pad, 64] fp32, boxes of 32 rows x 32
// columns (128 bytes), 128-byte swizzle (the reduction warps' staging layout).
bool encode_dq_acc(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const float* base,
                   int BH, int n_pad) {
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(n_pad), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {64 * 4, static_cast<cuuint64_t>(n_pad) * 64 * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// TMA map of the d = 64 statistics terms: [BH, n_pad, 16] bf16 (32-byte rows), boxes of
// 128 rows, 32-byte swizzle (the B operand layout of the statistics step).
bool encode_aug(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, int BH,
                int n_pad) {
  const cuuint64_t dims[3] = {16, static_cast<cuuint64_t>(n_pad), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {16 * 2, static_cast<cuuint64_t>(n_pad) * 16 * 2};
  const cuuint32_t box[3] = {16, static_cast<cuuint32_t>(kBlockM), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The query-outer pass's stream and its fork / join events, created once per device.
// Enqueueing is serialised by the mutex, so that each event's latest record is the one
// the following wait refers to.  Backward calls on different caller streams share the
// side stream, so their dQ passes run in call order.
constexpr int kMaxDevices = 64;
std::mutex g_fork_mu;
BwdFork g_fork[kMaxDevices];
bool g_fork_ready[kMaxDevices] = {};

cudaError_t fork_of_current_device(BwdFork** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  BwdFork& f = g_fork[dev];
  if (!g_fork_ready[dev]) {
    e = cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      // Release what was created, so that a later call starts afresh.
      if (f.side != nullptr) cudaStreamDestroy(f.side);
      if (f.fork != nullptr) cudaEventDestroy(f.fork);
      if (f.join != nullptr) cudaEventDestroy(f.join);
      f = BwdFork();
      return e;
    }
    g_fork_ready[dev] = true;
  }
  *out = &f;
  return cudaSuccess;
}

}  // namespace
}  // namespace osfa

using namespace osfa;

extern "C" {

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 0 || H < 0 || N < 0) return 0;
  return static_cast<size_t>(bwd_ws_bytes(static_cast<long long>(B) * H, N, 64, FA_BF16));
}

size_t fa_bwd_workspace_bytes_dt(int B, int H, int N, int d, fa_dtype dtype) {
  if (B < 0 || H < 0 || N < 0) return 0;
  if (dtype == FA_F32 ? (d < 1 || d > 128)
                      : ((dtype != FA_BF16 && dtype != FA_F16) || (d != 64 && d != 128)))
    return 0;
  return static_cast<size_t>(bwd_ws_bytes(static_cast<long long>(B) * H, N, d, dtype));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes, fa_dtype dtype,
                 cudaStream_t stream) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
  if (dtype != FA_BF16 && dtype != FA_F16 && dtype != FA_F32) return FA_ERR_UNSUPPORTED;
  const bool f32 = dtype == FA_F32;
  if (f32 ? (d < 1 || d > 128) : (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT_MAX) return FA_ERR_INVALID;
  if (BH == 0 || N == 0) return FA_OK;
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (ptr == nullptr) return FA_ERR_INVALID;
  if (lse == nullptr) return FA_ERR_INVALID;
  for (const void* ptr : ptrs)
    if (!aligned(ptr, f32 ? 4 : 16)) return FA_ERR_ALIGN;
  if (!aligned(lse, 4) || !aligned(workspace, 16)) return FA_ERR_ALIGN;
  const long long nblk = bwd_n_pad(N) / kBlockM;
  if (nblk * BH > INT_MAX) return FA_ERR_INVALID;
  if (workspace_bytes < static_cast<size_t>(bwd_ws_bytes(BH, N, d, dtype))) return FA_ERR_INVALID;
  if (f32) {
    // CUDA cores, warp per row: D (fp32, first B*H*N floats of the workspace), then the
    // key pass and the query pass.
    if ((BH * N + 3) / 4 > INT_MAX) return FA_ERR_INVALID;
    return from_cuda(launch_attn_bwd_f32(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<const float*>(o), lse, static_cast<const float*>(dout),
        static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv),
        static_cast<float*>(workspace), static_cast<int>(BH), N, d, scale, causal, stream));
  }

  unsigned* status = nullptr;
  cudaError_t e = status_word(&status);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((e = encode_fn(&enc)) != cudaSuccess) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo, tacc, taug;
  const int bh = static_cast<int>(BH);
  const bool f16 = dtype == FA_F16;
  if (!encode_bhnd(enc, &tq, q, bh, N, d, f16, kBlockM) ||
      !encode_bhnd(enc, &tk, k, bh, N, d, f16, kBlockM) ||
      !encode_bhnd(enc, &tv, v, bh, N, d, f16, kBlockM) ||
      !encode_bhnd(enc, &tdo, dout, bh, N, d, f16, kBlockM))
    return FA_ERR_CUDA;
  const int n_pad = static_cast<int>(nblk * kBlockM);
  // The workspace holds the statistics terms (32 bytes per row): at d = 64 first, followed
  // by the dQ accumulator (256 bytes per row); at d = 128 after LSE * log2(e) and D.
  const float* ws_f = static_cast<const float*>(workspace);
  if (!encode_aug(enc, &taug, d == 64 ? ws_f : ws_f + 2 * BH * n_pad, bh, n_pad))
    return FA_ERR_CUDA;
  if (d == 64 && !encode_dq_acc(enc, &tacc, ws_f + 8 * BH * n_pad, bh, n_pad)) return FA_ERR_CUDA;
  if (d != 64) tacc = tq;  // not read at d = 128
  AttnBwdParams p;
  p.lse2 = nullptr;  // set by the launcher from the workspace
  p.dd = nullptr;
  p.aug = nullptr;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = status;
  p.N = N;
  p.BH = bh;
  p.dq_acc = nullptr;  // set by the launcher (d = 64)
  p.nblk = static_cast<int>(nblk);
  p.n_pad = n_pad;
  // Heads scheduled together: as many as keep what each pass streams per head within
  // about 64 MB of L2 (two [N, d] tensors, and at d = 64 the head's fp32 dQ accumulator
  // rows, which every key tile's block adds into).
  const long long stream_head_bytes = 2LL * N * d * 2 + (d == 64 ? 256LL * N : 0LL);
  p.head_group = static_cast<int>(
      std::max(1LL, std::min(BH, (64LL << 20) / std::max(1LL, stream_head_bytes))));
  p.causal = causal;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  float* ws = static_cast<float*>(workspace);
  std::lock_guard<std::mutex> lock(g_fork_mu);
  BwdFork* fk = nullptr;
  if ((e = fork_of_current_device(&fk)) != cudaSuccess) return FA_ERR_CUDA;
  if (d == 64)
    e = f16 ? launch_attn_bwd<64, true>(tq, tk, tv, tdo, tacc, taug, o, dout, lse, ws, p, stream, fk)
            : launch_attn_bwd<64, false>(tq, tk, tv, tdo, tacc, taug, o, dout, lse, ws, p, stream, fk);
  else
    e = f16 ? launch_attn_bwd<128, true>(tq, tk, tv, tdo, tacc, taug, o, dout, lse, ws, p, stream, fk)
            : launch_attn_bwd<128, false>(tq, tk, tv, tdo, tacc, taug, o, dout, lse, ws, p, stream, fk);
  return from_cuda(e);
}

}  // extern "C"
