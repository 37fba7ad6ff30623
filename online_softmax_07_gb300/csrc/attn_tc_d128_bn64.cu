// tcgen05 attention forward, head dimension 128, bf16, 64-key tiles (block-size study) (kernel body in attn_tc_impl.cuh).
#include "attn_tc_impl.cuh"

namespace osfa {
template cudaError_t launch_attn_tc<128, 64, false>(const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&,
                                                  const AttnTcParams&, cudaStream_t);
}  // namespace osfa
