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
#include <algorithm>

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

// Per R consecutive query blocks r0 .. r0+R-1 of one listed head (blockIdx.x,
// blockIdx.y): sigma over c <= r for each of them, then one top-k per block into
// blk_idx (rows of ld >= topk entries, padded with -1).  Each pooled key block is
// read once for the R query blocks: warp w takes c = w, w + 8, ...; lane l holds
// dims 4l..4l+3 of the R pooled queries, forms R partial dots and reduces them
// over the warp by a butterfly that leaves query block i's sum in lanes 4i..4i+3
// (9 shuffles for 8 sums).  Then warp i selects for query block r0 + i.  R <= 8;
// the host picks R so that R * NB floats fit in shared memory.
constexpr int kSelRows = 8;
__global__ void __launch_bounds__(256)
block_select_kernel(const float* qbar, const float* kbar, int NB, int group, HeadList heads,
                    int topk, int ld, int R, int32_t* blk_idx) {
  extern __shared__ float sig[];  // [R][NB]
  __shared__ alignas(16) int hist[kSelRows][256];
  // the last query blocks (the most candidates) are scheduled first
  const int r0 = (gridDim.x - 1 - blockIdx.x) * R, slot = blockIdx.y;
  const int nr = min(R, NB - r0);
  const int rmax = r0 + nr - 1;
  const int g = heads.h[slot] / group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float4 qv[kSelRows];
#pragma unroll
  for (int i = 0; i < kSelRows; ++i)
    qv[i] = (i < nr) ? *reinterpret_cast<const float4*>(qbar + ((size_t)slot * NB + r0 + i) * kD + lane * 4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
  const int mine = (b16 ? 4 : 0) + (b8 ? 2 : 0) + (b4 ? 1 : 0);  // the query block this lane ends with
  // four pooled key blocks per warp and step; the next step's are loaded while
  // this step's are reduced (the loop is bound by the loads' latency)
  float4 kv4[4];
  auto load4 = [&](int c0, float4* dst) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + 8 * u;
      dst[u] = (c <= rmax) ? *reinterpret_cast<const float4*>(kbar + ((size_t)g * NB + c) * kD + lane * 4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load4(warp, kv4);
  for (int c0 = warp; c0 <= rmax; c0 += 32) {
    float4 nx4[4];
    load4(c0 + 32, nx4);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + 8 * u;
      const float4 kv = kv4[u];
      float v[kSelRows];
#pragma unroll
      for (int i = 0; i < kSelRows; ++i) v[i] = qv[i].x * kv.x + qv[i].y * kv.y + qv[i].z * kv.z + qv[i].w * kv.w;
      float w4[4], w2[2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float keep = b16 ? v[j + 4] : v[j], send = b16 ? v[j] : v[j + 4];
        w4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float keep = b8 ? w4[j + 2] : w4[j], send = b8 ? w4[j] : w4[j + 2];
        w2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      float y = (b4 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b4 ? w2[0] : w2[1], 4);
      y += __shfl_xor_sync(0xffffffffu, y, 2);
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      if ((lane & 3) == 0 && mine < nr && c <= rmax) sig[(size_t)mine * NB + c] = y;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) kv4[u] = nx4[u];
  }
  __syncthreads();
  // one query block per warp
  if (warp < nr) {
    const int r = r0 + warp;
    int32_t* out = blk_idx + ((size_t)slot * NB + r) * ld;
    const int kk = min(topk, r + 1);  // >= 1
    const float* sp = sig + (size_t)warp * NB;
    warp_topk_sorted([sp](int j) { return float_key(sp[j]); }, r + 1, kk, out, hist[warp]);
    for (int j = kk + lane; j < ld; j += 32) out[j] = -1;
  }
}

// Query blocks per selection CTA: up to kSelRows, as many as fit max_smem bytes of scores.
inline int block_select_rows(int NB, size_t max_smem) {
  const size_t per = sizeof(float) * (size_t)NB;
  return static_cast<int>(std::max<size_t>(1, std::min<size_t>(kSelRows, max_smem / per)));
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
