// tcgen05 attention forward, head dimension 64, bf16, 192-key tiles (block-size study) (kernel body in attn_tc_impl.cuh).
#include "attn_tc_impl.cuh"

namespace osfa {
template cudaError_t launch_attn_tc<64, 192, false>(const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&,
                                                  const AttnTcParams&, cudaStream_t);
}  // namespace osfa
