// Dense causal, A-shape, grid-row and cross-modality variants of the attention engine.
#include "attn_launch.cuh"

namespace mi {
#define MI_ATTN_MAPS const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, \
                     const CUtensorMap&
template cudaError_t launch_attn<kPatDense>(MI_ATTN_MAPS, const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn<kPatAShape>(MI_ATTN_MAPS, const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn<kPatRows>(MI_ATTN_MAPS, const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn<kPatCross>(MI_ATTN_MAPS, const AttnArgs&, int, cudaStream_t);
#undef MI_ATTN_MAPS
}  // namespace mi
