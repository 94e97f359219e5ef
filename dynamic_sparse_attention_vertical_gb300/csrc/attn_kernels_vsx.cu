// Vertical-slash engine with block-expanded slashes (64x64 blocks along each
// selected diagonal), compiled on its own so that the variants build in parallel.
#include "attn_launch.cuh"

namespace mi {
template cudaError_t launch_attn<kPatVSExp>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const CUtensorMap&, const AttnArgs&, int,
                                            cudaStream_t);
}  // namespace mi
