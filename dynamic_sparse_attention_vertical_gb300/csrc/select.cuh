// select.cuh - block-wide top-k selection, returned in ascending index order.
//
// The pages keep the top-k vertical columns and top-k slash diagonals
// (README mirror, gittoolsai.com, "Kernel-only usage": vertical_topk, slash)
// and note that top-k on a GPU can be slow (hugging-face.cn blog "How to
// optimise the TTFT of an 8B LLM with 1M tokens to 20 s", section on
// co-designing algorithm and system).  Selection here never sorts: a 4-pass
// 8-bit radix select finds the key of the k-th largest element, then one
// ordered compaction sweep writes every element above it plus the
// lowest-indexed elements equal to it.  Ties therefore go to the lower index
// and the output comes out ascending, deterministically.
#pragma once

#include "common.cuh"

namespace mi {

struct SelectSmem {
  int hist[256];
  int wgt[32];
  int weq[32];
  int bin;
  int rem;
};

// key_at(i) -> order-preserving uint32 key of element i (see float_key).
// Requires 1 <= k <= n.  Writes the k selected indices ascending to out[0..k).
// All NT threads of the block must call it.  The function has no early exit:
// every thread runs every block barrier in it.
template <int NT, class F>
__device__ void topk_select_sorted(F key_at, int n, int k, int* out, SelectSmem& sm) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += NT) sm.hist[i] = 0;
    __syncthreads();
    for (int base = warp * 32; base < n; base += NT) {
      const int i = base + lane;
      bool act = false;
      uint32_t bin = 0;
      if (i < n) {
        const uint32_t u = key_at(i);
        act = (u & pmask) == prefix;
        bin = (u >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, act ? bin : 256u + lane);
      if (act && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[bin], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane L covers bins 255-8L .. 248-8L (descending); find the bin where
      // the count of larger keys first reaches rem
      int c[8], tot = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = sm.hist[255 - (lane * 8 + e)];
        tot += c[e];
      }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
      if (lane == __ffs(hit) - 1) {
        int cum = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (cum + c[e] >= rem) {
            sm.bin = 255 - (lane * 8 + e);
            sm.rem = rem - cum;
            break;
          }
          cum += c[e];
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sm.bin) << shift;
    pmask |= 0xFFu << shift;
    rem = sm.rem;
    __syncthreads();
  }
  // prefix is now the key of the k-th largest element; take all larger keys and
  // the first `rem` equal ones.  Warp w sweeps its own contiguous segment.
  const int seg = cdiv(cdiv(n, NW), 32) * 32;
  const int beg = min(warp * seg, n), end = min(beg + seg, n);
  int gt = 0, eq = 0;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const uint32_t u = (i < end) ? key_at(i) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, i < end && u > prefix));
    eq += __popc(__ballot_sync(0xffffffffu, i < end && u == prefix));
  }
  if (lane == 0) {
    sm.wgt[warp] = gt;
    sm.weq[warp] = eq;
  }
  __syncthreads();
  int gb = 0, eb = 0;
  for (int w = 0; w < warp; ++w) {
    gb += sm.wgt[w];
    eb += sm.weq[w];
  }
  const unsigned lt = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const uint32_t u = (i < end) ? key_at(i) : 0u;
    const bool isg = i < end && u > prefix;
    const bool ise = i < end && u == prefix;
    const unsigned bg = __ballot_sync(0xffffffffu, isg);
    const unsigned be = __ballot_sync(0xffffffffu, ise);
    const int G = gb + __popc(bg & lt), E = eb + __popc(be & lt);
    if (isg) out[G + min(E, rem)] = i;
    else if (ise && E < rem) out[G + E] = i;
    gb += __popc(bg);
    eb += __popc(be);
  }
  __syncthreads();
}

// T1: top-k of the vertical (y = 0) or slash (y = 1) scores of every listed head;
// k > N keeps all N indices, and the row is padded with -1 up to k.
__global__ void __launch_bounds__(1024)
vs_topk_kernel(const float* vsc, const float* ssc, int N, int k_v, int k_s, int32_t* v_idx,
               int32_t* s_idx, int ld_v, int ld_s) {
  __shared__ SelectSmem sm;
  const int slot = blockIdx.x;
  const bool vert = blockIdx.y == 0;
  const float* x = (vert ? vsc : ssc) + (size_t)slot * N;
  const int k = vert ? k_v : k_s;
  const int ld = vert ? ld_v : ld_s;  // row stride >= k; the rest of a row is padding
  const int kk = min(k, N);
  int32_t* out = (vert ? v_idx : s_idx) + (size_t)slot * ld;
  if (kk > 0) topk_select_sorted<1024>([x](int i) { return float_key(__ldg(x + i)); }, N, kk, out, sm);
  for (int i = kk + threadIdx.x; i < ld; i += 1024) out[i] = -1;
}

}  // namespace mi
