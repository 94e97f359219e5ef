// Dense causal and A-shape variants of the attention engine.
#include "attn_launch.cuh"

namespace mi {
template cudaError_t launch_attn<kPatDense>(const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn<kPatAShape>(const CUtensorMap&, const CUtensorMap&,
                                             const CUtensorMap&, const AttnArgs&, int, cudaStream_t);
}  // namespace mi
