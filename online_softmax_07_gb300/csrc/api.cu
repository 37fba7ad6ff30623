// api.cu -- the C ABI declared in include/fa.h: argument checks, TMA descriptor set-up
// and dispatch to the kernels.  No device memory is allocated here: the status word
// the kernels report bounded-wait time-outs in is a static device variable.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_tc.cuh"
#include "fa.h"
#include "host_util.h"
#include "kernels.h"
#include "ptx.cuh"

namespace osfa {
namespace {

__device__ unsigned g_device_status;

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;
std::mutex g_mutex;
unsigned* g_status_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

// Address of this device's status word (looked up once per device).
cudaError_t status_word(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

cudaError_t encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return cudaSuccess;
}

// A [BH, N, d] bf16 or fp16 tensor seen by TMA as 3-D (d innermost), boxes of box_rows
// rows x 64 columns (128 bytes) with the 128-byte swizzle.  Rows past N read as zero and
// are not written by stores.
bool encode_bhnd(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base,
                 int BH, int N, int d, bool f16, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(box_rows),
                             1};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

namespace {

__global__ void wait_timeout_selftest_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // expects one arrival that never comes
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned* status, unsigned long long limit_ns,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace osfa

using namespace osfa;

extern "C" {

const char* fa_status_str(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or dtype";
    case FA_ERR_ALIGN: return "misaligned pointer";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case FA_ERR_TOO_LARGE: return "problem needs more than the library's 64 MiB static scratch";
  }
  return "unknown status";
}

}  // extern "C"

namespace osfa {

// Checks shared by the tensor-core entry points (bf16/fp16, d in {64, 128}).
fa_status check_tc_args(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, int B, int H, int N, int d, float scale, int causal,
                        fa_dtype dtype) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
  if (dtype != FA_BF16 && dtype != FA_F16) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > INT_MAX) return FA_ERR_INVALID;
  if (static_cast<long long>(B) * H == 0 || N == 0) return FA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID;
  if (lse != nullptr && !aligned(lse, 4)) return FA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return FA_ERR_ALIGN;
  return FA_OK;
}

namespace {

long long nqb_of(int N) { return (static_cast<long long>(N) + 2 * kBlockM - 1) / (2 * kBlockM); }

// Launches the tensor-core kernel; with splits > 1 it writes partials to ws_o / ws_lse
// (caller-sized) and the combine kernel then writes o and lse.
fa_status run_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, fa_dtype dtype, int splits, float* ws_o,
                 float* ws_lse, cudaStream_t stream, int block_n = kDefaultBlockN) {
  const long long BH = static_cast<long long>(B) * H;
  const long long nqb = nqb_of(N);
  if (nqb * BH * splits > INT_MAX) return FA_ERR_INVALID;
  unsigned* status = nullptr;
  cudaError_t e = status_word(&status);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((e = encode_fn(&enc)) != cudaSuccess) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, to;
  const int bh = static_cast<int>(BH);
  const bool f16 = dtype == FA_F16;
  if (!encode_bhnd(enc, &tq, q, bh, N, d, f16, kBlockM) ||
      !encode_bhnd(enc, &tk, k, bh, N, d, f16, block_n) ||
      !encode_bhnd(enc, &tv, v, bh, N, d, f16, block_n) ||
      !encode_bhnd(enc, &to, o, bh, N, d, f16, kBlockM))
    return FA_ERR_CUDA;
  AttnTcParams p;
  p.lse = lse;
  p.status = status;
  p.N = N;
  p.BH = bh;
  p.nqb = static_cast<int>(nqb);
  // Heads scheduled together: as many as keep their K and V within about 32 MB of the
  // 129 MB L2 (a sweep of 8-128 MB on GB300: 32 MB within 1 % of the best budget on every
  // shape measured, and the one at which B2 H16 N8192 causal reads Q, K and V from DRAM
  // only once; 16 MB and below lengthen the causal tail).
  const long long kv_head_bytes = 2LL * N * d * 2;
  p.head_group = static_cast<int>(
      std::max(1LL, std::min(BH, (32LL << 20) / std::max(1LL, kv_head_bytes))));
  p.causal = causal;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.splits = splits;
  p.n_pad = static_cast<int>(nqb * 2 * kBlockM);
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  if (block_n == 64)  // block-size study kernels (bf16)
    e = d == 64 ? launch_attn_tc<64, 64, false>(tq, tk, tv, to, p, stream)
                : launch_attn_tc<128, 64, false>(tq, tk, tv, to, p, stream);
  else if (block_n == 192)
    e = launch_attn_tc<64, 192, false>(tq, tk, tv, to, p, stream);
  else if (block_n == 256)
    e = launch_attn_tc<64, 256, false>(tq, tk, tv, to, p, stream);
  else if (d == 64)
    e = f16 ? launch_attn_tc<64, 128, true>(tq, tk, tv, to, p, stream)
            : launch_attn_tc<64, 128, false>(tq, tk, tv, to, p, stream);
  else
    e = f16 ? launch_attn_tc<128, 128, true>(tq, tk, tv, to, p, stream)
            : launch_attn_tc<128, 128, false>(tq, tk, tv, to, p, stream);
  if (e != cudaSuccess || splits == 1) return from_cuda(e);
  return from_cuda(launch_splitkv_combine(ws_o, ws_lse, o, lse, bh, N, p.n_pad, d, splits, f16,
                                          stream));
}

// Workspace of the split-KV forward: fp32 partial O then fp32 partial LSE.
long long splitkv_ws_bytes(long long BH, int N, int d, int splits) {
  const long long n_pad = nqb_of(N) * 2 * kBlockM;
  return static_cast<long long>(splits) * BH * n_pad * (d + 1) * 4;
}

}  // namespace
}  // namespace osfa

extern "C" {

fa_status fa_fwd_dt(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int N, int d, float scale, int causal, fa_dtype dtype,
                    cudaStream_t stream) {
  if (dtype == FA_F32) {
    if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
    if (d < 1 || d > 128) return FA_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    if (BH > INT_MAX) return FA_ERR_INVALID;
    if (BH == 0 || N == 0) return FA_OK;  // empty problem
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID;
    if (lse != nullptr && !aligned(lse, 4)) return FA_ERR_ALIGN;
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(o, 4)) return FA_ERR_ALIGN;
    if ((static_cast<long long>(N) + 15) / 16 * BH > INT_MAX) return FA_ERR_INVALID;
    return from_cuda(launch_attn_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                     static_cast<const float*>(v), static_cast<float*>(o), lse,
                                     static_cast<int>(BH), N, d, scale, causal, stream));
  }
  fa_status st = check_tc_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype);
  if (st != FA_OK || static_cast<long long>(B) * H == 0 || N == 0) return st;
  return run_tc(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 1, nullptr, nullptr, stream);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits) {
  if (B < 0 || H < 0 || N < 0 || num_splits < 1 || (d != 64 && d != 128)) return 0;
  return static_cast<size_t>(splitkv_ws_bytes(static_cast<long long>(B) * H, N, d, num_splits));
}

int fa_fwd_splitkv_splits_for(int B, int H, int N, int causal, int sms) {
  if (B <= 0 || H <= 0 || N <= 0 || (causal != 0 && causal != 1) || sms <= 0) return 1;
  const long long blocks = nqb_of(N) * B * H;
  const long long kv_tiles = (static_cast<long long>(N) + kDefaultBlockN - 1) / kDefaultBlockN;
  // Causal: floor(2 sms / blocks + 0.2), the longest block over the average work per SM;
  // not causal: as many pieces as still run in one wave.  (Measured on GB300, 152 SMs:
  // causal 64 blocks best at 4 splits, 128 and 160 at 2, 256 at 1-2; not causal 32
  // blocks best at 4, 128 at 1.)
  long long s = causal ? (20LL * sms + 2 * blocks) / (10 * blocks) : sms / blocks;
  s = std::min<long long>(s, std::max<long long>(1, kv_tiles / 2));
  return static_cast<int>(std::max<long long>(1, std::min<long long>(s, kMaxSplits)));
}

int fa_fwd_splitkv_default_splits(int B, int H, int N, int causal) {
  int dev = 0, sms = 0;
  // Without the device's SM count no split can be shown to pay: one split.
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 1;
  return fa_fwd_splitkv_splits_for(B, H, N, causal, sms);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal, int num_splits,
                         void* workspace, size_t workspace_bytes, fa_dtype dtype,
                         cudaStream_t stream) {
  fa_status st = check_tc_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype);
  if (st != FA_OK) return st;
  if (num_splits < 1 || num_splits > kMaxSplits) return FA_ERR_INVALID;
  if (static_cast<long long>(B) * H == 0 || N == 0) return FA_OK;
  if (num_splits == 1)
    return run_tc(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 1, nullptr, nullptr, stream);
  const long long BH = static_cast<long long>(B) * H;
  if (workspace == nullptr) return FA_ERR_INVALID;
  if (!aligned(workspace, 16)) return FA_ERR_ALIGN;
  if (static_cast<long long>(workspace_bytes) < splitkv_ws_bytes(BH, N, d, num_splits))
    return FA_ERR_INVALID;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_lse = ws_o + static_cast<long long>(num_splits) * BH * nqb_of(N) * 2 * kBlockM * d;
  return run_tc(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, num_splits, ws_o, ws_lse,
                stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, cudaStream_t stream) {
  return fa_fwd_dt(q, k, v, o, lse, B, H, N, d, scale, causal, FA_BF16, stream);
}

fa_status fa_fwd_block(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, int causal, fa_dtype dtype, int block_n,
                       cudaStream_t stream) {
  if (block_n == 0 || block_n == kDefaultBlockN)
    return fa_fwd_dt(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream);
  if (block_n != 64 && block_n != 192 && block_n != 256) return FA_ERR_INVALID;
  fa_status st = check_tc_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype);
  if (st != FA_OK) return st;
  if (dtype != FA_BF16 || (block_n >= 192 && d != 64)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H == 0 || N == 0) return FA_OK;
  return run_tc(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 1, nullptr, nullptr, stream,
                block_n);
}

fa_status online_softmax_rows(const float* x, float* m_out, float* l_out, int rows, int len,
                              cudaStream_t stream) {
  if (rows < 0 || len < 0) return FA_ERR_INVALID;
  if (rows == 0) return FA_OK;
  if (len == 0) return FA_ERR_INVALID;
  if (x == nullptr || m_out == nullptr || l_out == nullptr) return FA_ERR_INVALID;
  if (!aligned(x, 4) || !aligned(m_out, 4) || !aligned(l_out, 4)) return FA_ERR_ALIGN;
  return from_cuda(launch_row_state(x, m_out, l_out, rows, len, stream));
}

fa_status online_softmax_forward(const float* x, float* y, float* m_out, float* l_out, int rows,
                                 int len, cudaStream_t stream) {
  if (rows < 0 || len < 0) return FA_ERR_INVALID;
  if (rows == 0) return FA_OK;
  if (len == 0) return FA_ERR_INVALID;
  if (x == nullptr || y == nullptr) return FA_ERR_INVALID;
  if (!aligned(x, 4) || !aligned(y, 4) || (m_out != nullptr && !aligned(m_out, 4)) ||
      (l_out != nullptr && !aligned(l_out, 4)))
    return FA_ERR_ALIGN;
  return from_cuda(launch_softmax_rows(x, y, m_out, l_out, rows, len, stream));
}

fa_status fa_last_device_error(cudaStream_t stream) {
  unsigned* status = nullptr;
  if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  unsigned value = 0;
  if (cudaMemcpy(&value, status, sizeof(value), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (value != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return (value & kStatusTimeout) ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status fa_selftest_wait_timeout(long long limit_ns, cudaStream_t stream) {
  if (limit_ns < 1 || limit_ns > 2000000000LL) return FA_ERR_INVALID;
  unsigned* status = nullptr;
  if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
  return from_cuda(
      launch_wait_timeout_selftest(status, static_cast<unsigned long long>(limit_ns), stream));
}

}  // extern "C"
