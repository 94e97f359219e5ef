// block.cuh - block selection for block-sparse heads.
//
// Pattern: MInference talk slides (boteman.cn), "A-shape, Vertical-Slash and
// block-sparse patterns"; kernel call block_sparse_attention(q, k, v, topk)
// in the README mirror (gittoolsai.com), "Kernel-only usage".  Selection
// reading: mean-pool each 64-row block of Q and K, score sigma[r, c] =
// Qbar_r . Kbar_c for c <= r, keep the top-min(topk, r+1) blocks (larger
// score, then lower c), ascending.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace mi {

// Mean of 64 consecutive rows (of the rows left in a last, partial block), fp32:
// one warp per (head, block); lane l owns dims 4l..4l+3 and adds the rows in
// order.  Output head o reads source head heads.h[o] (use_list) or o; heads are
// ld rows apart.
__global__ void block_pool_kernel(const __nv_bfloat16* src, int N, int64_t ld, int n_out, int NB,
                                  HeadList heads, int use_list, float* out) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= n_out * NB) return;
  const int o = gw / NB, blk = gw - o * NB;
  const int h = use_list ? heads.h[o] : o;
  const __nv_bfloat16* base = src + ((size_t)h * ld + (size_t)blk * kBlk) * kD + lane * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int rows = min(kBlk, N - blk * kBlk);
  for (int r = 0; r < rows; ++r) {
    const uint2 raw = *reinterpret_cast<const uint2*>(base + (size_t)r * kD);
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    acc[0] += __low2float(p0);
    acc[1] += __high2float(p0);
    acc[2] += __low2float(p1);
    acc[3] += __high2float(p1);
  }
  const float inv = 1.f / static_cast<float>(rows);
  const float4 res = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<float4*>(out + ((size_t)o * NB + blk) * kD + lane * 4) = res;
}

// Per (query block r, listed head): sigma over c <= r, then top-k into blk_idx
// (rows of ld >= topk entries, padded with -1).
__global__ void __launch_bounds__(256)
block_select_kernel(const float* qbar, const float* kbar, int NB, int group, HeadList heads,
                    int topk, int ld, int32_t* blk_idx) {
  extern __shared__ float sig[];  // [NB]
  __shared__ SelectSmem sm;
  __shared__ __align__(16) float qrow[kD];
  const int r = blockIdx.x, slot = blockIdx.y;
  const int g = heads.h[slot] / group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kD) qrow[tid] = qbar[((size_t)slot * NB + r) * kD + tid];
  __syncthreads();
  const float4 qv = *reinterpret_cast<const float4*>(qrow + lane * 4);
  for (int c = warp; c <= r; c += 8) {
    const float4 kv = *reinterpret_cast<const float4*>(kbar + ((size_t)g * NB + c) * kD + lane * 4);
    float d = qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) sig[c] = d;
  }
  __syncthreads();
  int32_t* out = blk_idx + ((size_t)slot * NB + r) * ld;
  const int kk = min(topk, r + 1);  // >= 1
  const float* sp = sig;
  topk_select_sorted<256>([sp](int i) { return float_key(sp[i]); }, r + 1, kk, out, sm);
  for (int i = kk + tid; i < ld; i += 256) out[i] = -1;
}

// With caller-given block lists: flag any row that is not ascending, out of
// [0, r] or has a value after -1 padding.
__global__ void block_validate_kernel(const int32_t* blk_idx, int NB, int topk, int n_rows,
                                      int* status) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= n_rows) return;
  const int r = row % NB;
  const int32_t* b = blk_idx + (size_t)row * topk;
  int prev = -1;
  bool pad = false;
  for (int e = 0; e < topk; ++e) {
    const int c = b[e];
    if (c == -1) {
      pad = true;
      continue;
    }
    if (pad || c < 0 || c > r || c <= prev) {
      set_status(status, MI_ERR_INDEX);
      return;
    }
    prev = c;
  }
}

}  // namespace mi
