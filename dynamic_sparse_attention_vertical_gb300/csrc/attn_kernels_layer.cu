// The layer variant of the attention engine: every pattern of a layer's heads in one launch.
#include "attention.cuh"

namespace mi {

// The lighter patterns' engines as functions of their own, so that each gets its
// own register allocation and the inlined vertical-slash engine keeps its own.
template <int PAT>
__device__ __noinline__ void attn_body_call(uint8_t* smem_raw, const CUtensorMap& map_q, const CUtensorMap& map_k,
                                            const CUtensorMap& map_v, const CUtensorMap& map_kr,
                                            const CUtensorMap& map_vr, const AttnArgs& a, int r, int n, int h) {
  attn_body<PAT>(smem_raw, map_q, map_k, map_v, map_kr, map_vr, a, r, n, h);
}

// A layer's heads of every pattern in one launch: blockIdx.y is the listed head
// (dense, vertical-slash, block-sparse, A-shape in turn), blockIdx.x the row block
// counted from the last, so the heavier patterns start first and the lighter
// ones fill the end.  The slot is blockIdx.y minus a per-pattern constant, which
// the compiler can recompute instead of holding a register for it.  VSP is the
// vertical-slash engine: exact (kPatVS) or block-expanded slashes (kPatVSExp).
template <int VSP>
__global__ void __launch_bounds__(kAttnThreads, 2)
attn_layer_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_kr,
                  const __grid_constant__ CUtensorMap map_vr, const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int NRB = cdiv(a.N, kBM);
  const int r = NRB - 1 - static_cast<int>(blockIdx.x);
  const int y = static_cast<int>(blockIdx.y);
  const int h = a.heads.h[y];
  if (y >= a.layer_base[kPatVS] && y < a.layer_base[kPatBlock]) {
    // the heaviest pattern of a layer: inlined, with the kernel's own registers
    attn_body<VSP>(smem_raw, map_q, map_k, map_v, map_kr, map_vr, a, r, y - a.layer_base[kPatVS], h);
  } else if (y < a.layer_base[kPatVS]) {
    attn_body_call<kPatDense>(smem_raw, map_q, map_k, map_v, map_kr, map_vr, a, r, y - a.layer_base[kPatDense], h);
  } else if (y < a.layer_base[kPatAShape]) {
    attn_body_call<kPatBlock>(smem_raw, map_q, map_k, map_v, map_kr, map_vr, a, r, y - a.layer_base[kPatBlock], h);
  } else {
    attn_body_call<kPatAShape>(smem_raw, map_q, map_k, map_v, map_kr, map_vr, a, r, y - a.layer_base[kPatAShape],
                               h);
  }
}

cudaError_t launch_attn_layer(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                              const CUtensorMap& mkr, const CUtensorMap& mvr, const AttnArgs& a,
                              int n_row_blocks, cudaStream_t st) {
  static cudaError_t attr = cudaFuncSetAttribute(attn_layer_kernel<kPatVS>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kAttnSmemBytes));
  static cudaError_t attr_x = cudaFuncSetAttribute(attn_layer_kernel<kPatVSExp>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kAttnSmemBytes));
  if (attr != cudaSuccess) return attr;
  if (attr_x != cudaSuccess) return attr_x;
  const dim3 grid(n_row_blocks, a.heads.n);
  if (a.expand)
    attn_layer_kernel<kPatVSExp><<<grid, kAttnThreads, kAttnSmemBytes, st>>>(mq, mk, mv, mkr, mvr, a);
  else
    attn_layer_kernel<kPatVS><<<grid, kAttnThreads, kAttnSmemBytes, st>>>(mq, mk, mv, mkr, mvr, a);
  return cudaGetLastError();
}

}  // namespace mi
