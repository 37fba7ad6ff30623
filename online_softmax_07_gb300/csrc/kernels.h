// kernels.h -- launchers shared between the kernel translation units and the C ABI
// (api.cu).  Internal to the library; the public interface is include/fa.h.
#pragma once

#include <cuda_runtime.h>

namespace osfa {

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int BH, int N, int d, float scale, int causal, cudaStream_t stream);

cudaError_t launch_attn_bwd_f32(const float* q, const float* k, const float* v, const float* o,
                                const float* lse, const float* dout, float* dq, float* dk,
                                float* dv, float* dd, int BH, int N, int d, float scale,
                                int causal, cudaStream_t stream);

cudaError_t launch_row_state(const float* x, float* m_out, float* l_out, int rows, int len,
                             cudaStream_t stream);

cudaError_t launch_softmax_rows(const float* x, float* y, float* m_out, float* l_out, int rows,
                                int len, cudaStream_t stream);

cudaError_t launch_splitkv_combine(const float* ws_o, const float* ws_lse, void* o, float* lse,
                                   int BH, int N, int n_pad, int d, int splits, bool f16,
                                   cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(unsigned* status, unsigned long long limit_ns,
                                         cudaStream_t stream);

}  // namespace osfa
