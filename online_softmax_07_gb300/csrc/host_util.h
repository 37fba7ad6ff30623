// host_util.h -- host helpers of the C ABI shared by its translation units (api.cu,
// api_bwd.cu, splitkv_static.cu).  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "fa.h"

namespace osfa {

// Device address of the status word the kernels report bounded-wait time-outs in.
cudaError_t status_word(unsigned** out);
// cuTensorMapEncodeTiled from the driver (looked up once).
cudaError_t encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out);
// TMA map of a [BH, N, d] bf16/fp16 tensor, box_rows x 64-column boxes, 128-byte swizzle.
bool encode_bhnd(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base,
                 int BH, int N, int d, bool f16, int box_rows);
bool aligned(const void* p, uintptr_t a);
fa_status from_cuda(cudaError_t e);
// Host-side argument checks of the tensor-core forward entry points (bf16/fp16, d in
// {64, 128}); FA_OK also for an empty problem.  Touches no device state.
fa_status check_tc_args(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, int B, int H, int N, int d, float scale, int causal,
                        fa_dtype dtype);

}  // namespace osfa
