// Head dimension 64 instances of the tcgen05 attention backward.
#include "attn_bwd_impl.cuh"

namespace osfa {
template cudaError_t launch_attn_bwd<64, false>(const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&,
                                               const void*, const void*,
                                               const float*, float*, const AttnBwdParams&,
                                               cudaStream_t, const BwdFork*);
template cudaError_t launch_attn_bwd<64, true>(const CUtensorMap&, const CUtensorMap&,
                                              const CUtensorMap&, const CUtensorMap&,
                                              const CUtensorMap&, const CUtensorMap&,
                                              const void*, const void*,
                                              const float*, float*, const AttnBwdParams&,
                                              cudaStream_t, const BwdFork*);
}  // namespace osfa
