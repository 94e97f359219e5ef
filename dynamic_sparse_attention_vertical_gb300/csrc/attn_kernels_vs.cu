// Vertical-slash and block-sparse variants of the attention engine.
#include "attn_launch.cuh"

namespace mi {
template cudaError_t launch_attn<kPatVS>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                         const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn<kPatBlock>(const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const AttnArgs&, int, cudaStream_t);
}  // namespace mi
