// attn_launch.cuh - definition of mi::launch_attn, included by the per-pattern units.
#pragma once

#include "attention.cuh"

namespace mi {

template <int PAT>
cudaError_t launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mkr, const CUtensorMap& mvr, const AttnArgs& a,
                        int n_row_blocks, cudaStream_t st) {
  static cudaError_t attr = cudaFuncSetAttribute(
      attn_kernel<PAT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kAttnSmemBytes));
  if (attr != cudaSuccess) return attr;
  attn_kernel<PAT><<<dim3(n_row_blocks, a.heads.n), kAttnThreads, kAttnSmemBytes, st>>>(mq, mk, mv, mkr, mvr, a);
  return cudaGetLastError();
}

}  // namespace mi
