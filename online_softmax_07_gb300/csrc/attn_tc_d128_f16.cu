// tcgen05 attention forward, head dimension 128, fp16, 128-key tiles (kernel body in attn_tc_impl.cuh).
#include "attn_tc_impl.cuh"

namespace osfa {
template cudaError_t launch_attn_tc<128, 128, true>(const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&,
                                                  const AttnTcParams&, cudaStream_t);
}  // namespace osfa
