// tcgen05 attention forward, head dimension 64, bf16, 128-key tiles (kernel body in attn_tc_impl.cuh).
#include "attn_tc_impl.cuh"

namespace osfa {
template cudaError_t launch_attn_tc<64, 128, false>(const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&,
                                                  const AttnTcParams&, cudaStream_t);
}  // namespace osfa
