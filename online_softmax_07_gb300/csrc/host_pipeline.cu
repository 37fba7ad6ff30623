// host_pipeline.cu -- fa_fwd_host: the attention forward on host-resident tensors, with the
// copies in, the kernels and the copies out of consecutive groups of (batch, head) slabs
// overlapped on three streams (internal copy-in and copy-out streams, and the caller's).
//
// Per group c, in device slot c % 3 of the caller's workspace:
//   copy-in stream:  [wait: slot's previous copies out done]  Q, K, V host -> slot
//   caller's stream: [wait: copies in done]  fa_fwd_dt on the slot
//   copy-out stream: [wait: kernel done]  O (and LSE) slot -> host
// so group c+1 is copied in while group c computes and group c-1 is copied out.  The
// streams and events are created once per device; enqueueing is serialised by a mutex,
// which keeps each event's most recent record the one a later wait refers to.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "host_util.h"

namespace osfa {
namespace {

constexpr int kSlots = 3;       // groups whose device buffers are in use at a time
constexpr int kMaxDevices = 64;

struct HostPipe {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr;             // the caller's stream reached the call
  cudaEvent_t in_done[kSlots] = {};        // slot's Q, K, V copied in
  cudaEvent_t comp_done[kSlots] = {};      // slot's kernel finished
  cudaEvent_t out_done[kSlots] = {};       // slot's O, LSE copied out
  bool used[kSlots] = {};                  // slot written by an earlier group
};

std::mutex g_mu;
HostPipe g_pipes[kMaxDevices];

// Destroys whatever streams and events of `p` exist and clears it.
void release_pipe(HostPipe& p) {
  if (p.s_in != nullptr) cudaStreamDestroy(p.s_in);
  if (p.s_out != nullptr) cudaStreamDestroy(p.s_out);
  if (p.start != nullptr) cudaEventDestroy(p.start);
  for (int i = 0; i < kSlots; ++i)
    for (cudaEvent_t ev : {p.in_done[i], p.comp_done[i], p.out_done[i]})
      if (ev != nullptr) cudaEventDestroy(ev);
  p = HostPipe();
}

cudaError_t pipe_of_current_device(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    e = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i)
      for (cudaEvent_t* ev : {&p.in_done[i], &p.comp_done[i], &p.out_done[i]})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      release_pipe(p);  // nothing half-built stays behind; the next call starts afresh
      return e;
    }
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Arguments fa_fwd_dt would accept for these shapes (pointers aside).
fa_status check_shape(int B, int H, int N, int d, float scale, int causal, fa_dtype dtype) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
  if (static_cast<long long>(B) * H > INT_MAX) return FA_ERR_INVALID;
  if (dtype == FA_F32) return (d >= 1 && d <= 128) ? FA_OK : FA_ERR_UNSUPPORTED;
  if (dtype != FA_BF16 && dtype != FA_F16) return FA_ERR_UNSUPPORTED;
  return (d == 64 || d == 128) ? FA_OK : FA_ERR_UNSUPPORTED;
}

// `chunks` groups of equal size (the last may be smaller).  The kernels of the groups run
// one after another on the caller's stream and each takes at least as long as its
// longest query block, so small groups do not pay: a separate one-head last group, to
// shorten the final copy out, made B2 H16 N8192 causal slower (1.357 vs 1.272 ms at four
// groups).
struct Layout {
  long long groups = 0, heads = 0;  // number of groups, heads per group
  size_t tensor = 0, lse = 0, slot = 0, total = 0;
};

Layout layout(long long BH, int N, int d, fa_dtype dtype, int chunks) {
  Layout L;
  const long long g = std::min<long long>(std::max(1, chunks), BH);
  L.heads = (BH + g - 1) / g;
  L.groups = (BH + L.heads - 1) / L.heads;
  const size_t es = dtype == FA_F32 ? 4 : 2;
  L.tensor = round_up(static_cast<size_t>(L.heads) * N * d * es, 256);
  L.lse = round_up(static_cast<size_t>(L.heads) * N * 4, 256);
  L.slot = 4 * L.tensor + L.lse;
  L.total = std::min<long long>(kSlots, L.groups) * L.slot;
  return L;
}

}  // namespace
}  // namespace osfa

extern "C" {

size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d, fa_dtype dtype, int chunks) {
  using namespace osfa;
  if (chunks < 1 || check_shape(B, H, N, d, 1.0f, 0, dtype) != FA_OK) return 0;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || N == 0) return 0;
  return layout(BH, N, d, dtype, chunks).total;
}

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int N, int d, float scale, int causal, fa_dtype dtype, int chunks,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace osfa;
  fa_status st = check_shape(B, H, N, d, scale, causal, dtype);
  if (st != FA_OK) return st;
  if (chunks < 1) return FA_ERR_INVALID;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || N == 0) return FA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID;
  const Layout L = layout(BH, N, d, dtype, chunks);
  if (workspace == nullptr || workspace_bytes < L.total) return FA_ERR_INVALID;
  if (!aligned(workspace, 256)) return FA_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mu);
  HostPipe* pp = nullptr;
  cudaError_t e = pipe_of_current_device(&pp);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  HostPipe& P = *pp;
  const size_t es = dtype == FA_F32 ? 4 : 2;
  const size_t head_bytes = static_cast<size_t>(N) * d * es;
  const size_t head_lse = static_cast<size_t>(N) * 4;
  auto ok = [&](cudaError_t r) { return (e = r) == cudaSuccess; };

  // The copies in (into the workspace) follow the caller's earlier work.
  if (!ok(cudaEventRecord(P.start, stream)) || !ok(cudaStreamWaitEvent(P.s_in, P.start, 0)))
    return FA_ERR_CUDA;
  int last = 0;
  for (long long c = 0; c < L.groups; ++c) {
    const int slot = static_cast<int>(c % kSlots);
    const long long h0 = c * L.heads;
    const long long hn = std::min(L.heads, BH - h0);
    uint8_t* base = static_cast<uint8_t*>(workspace) + slot * L.slot;
    void* dq = base;
    void* dk = base + L.tensor;
    void* dv = base + 2 * L.tensor;
    void* dout = base + 3 * L.tensor;
    float* dlse = lse != nullptr ? reinterpret_cast<float*>(base + 4 * L.tensor) : nullptr;
    const size_t off = static_cast<size_t>(h0) * head_bytes;
    const size_t bytes = static_cast<size_t>(hn) * head_bytes;
    if (P.used[slot] && !ok(cudaStreamWaitEvent(P.s_in, P.out_done[slot], 0))) return FA_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + off, bytes,
                            cudaMemcpyHostToDevice, P.s_in)) ||
        !ok(cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + off, bytes,
                            cudaMemcpyHostToDevice, P.s_in)) ||
        !ok(cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + off, bytes,
                            cudaMemcpyHostToDevice, P.s_in)) ||
        !ok(cudaEventRecord(P.in_done[slot], P.s_in)) ||
        !ok(cudaStreamWaitEvent(stream, P.in_done[slot], 0)))
      return FA_ERR_CUDA;
    st = fa_fwd_dt(dq, dk, dv, dout, dlse, 1, static_cast<int>(hn), N, d, scale, causal, dtype,
                   stream);
    if (st != FA_OK) return st;
    if (!ok(cudaEventRecord(P.comp_done[slot], stream)) ||
        !ok(cudaStreamWaitEvent(P.s_out, P.comp_done[slot], 0)) ||
        !ok(cudaMemcpyAsync(static_cast<uint8_t*>(o) + off, dout, bytes, cudaMemcpyDeviceToHost,
                            P.s_out)))
      return FA_ERR_CUDA;
    if (lse != nullptr &&
        !ok(cudaMemcpyAsync(lse + h0 * N, dlse, static_cast<size_t>(hn) * head_lse,
                            cudaMemcpyDeviceToHost, P.s_out)))
      return FA_ERR_CUDA;
    if (!ok(cudaEventRecord(P.out_done[slot], P.s_out))) return FA_ERR_CUDA;
    P.used[slot] = true;
    last = slot;
  }
  // Later work on the caller's stream follows the last copy out (the copy-out stream is
  // in order, so its last event covers every group).
  if (!ok(cudaStreamWaitEvent(stream, P.out_done[last], 0))) return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
