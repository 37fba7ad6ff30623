// splitkv_static.cu -- split-KV attention forward that allocates no device memory.
//
// fa_fwd_splitkv needs a workspace for the per-split partial results, and leaves it to
// the caller to provide one.  Some callers cannot allocate device memory at the point
// where they call attention: code that runs while an application's memory pool or
// arena owns all device memory (cudaMalloc there would fail or break the pool's
// accounting), plugins of inference runtimes whose plugin interface gives them no
// allocator, and latency-critical paths where cudaMalloc/cudaFree would synchronise the
// device.  This entry point gives them split-KV without any allocation: the partials go
// to a scratch array that lives in the library's static device memory.
//
// The array is reserved on every GPU that loads the library, for as long as the library
// stays loaded (kStaticScratchBytes each).  Problems whose partials need more are
// rejected with FA_ERR_TOO_LARGE before anything is launched.  Every call shares the
// array: the kernels write every partial they later read (empty chunks included), so
// nothing needs clearing between calls, but calls whose work overlaps on the GPU (other
// streams, other host threads) would overwrite each other's partials.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "host_util.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;  // fa_fwd_splitkv's limit

static __device__ __align__(256) unsigned char g_splitkv_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side name of
// the array is only a stand-in for the runtime, not a device address, so the address is
// looked up once per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_splitkv_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" fa_status fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int B, int H, int N, int d, float scale,
                                           int causal, int num_splits, fa_dtype dtype,
                                           cudaStream_t stream) {
  // Arguments are checked before anything touches the device.
  if (num_splits < 1 || num_splits > kMaxSplits) return FA_ERR_INVALID;
  const fa_status st = osfa::check_tc_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype);
  if (st != FA_OK) return st;
  if (static_cast<long long>(B) * H == 0 || N == 0) return FA_OK;  // empty: nothing launched
  // One split needs no partials, hence no scratch.
  if (num_splits == 1)
    return fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, 1, nullptr, 0, dtype,
                          stream);
  if (fa_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits) > kStaticScratchBytes)
    return FA_ERR_TOO_LARGE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return FA_ERR_CUDA;
  return fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, scratch,
                        kStaticScratchBytes, dtype, stream);
}
