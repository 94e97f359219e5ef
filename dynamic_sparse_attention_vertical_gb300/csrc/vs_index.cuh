// vs_index.cuh - index structures of a vertical-slash head (one CTA per head).
//
// From the sorted column list V and offset list S the sparse attention kernel
// needs, per head:
//   offbits  bit o set for o in S             (element mask of diagonal tiles)
//   colbits  bit j set for j in V             (columns inside contiguous tiles)
//   dbits    bit delta set when some diagonal of S reaches key tile r - delta
//            from query row block r (128-row blocks, 128-key tiles); an offset
//            o = 128a + b touches distances a and, if b > 0, a + 1; distance 0
//            (the local block) is always set
//   dlist    the set distances in ascending order, dcount of them.
//   dfull    bit delta (> 0) set when every offset a 128x128 tile at distance
//            delta can meet, [128*delta - 127, 128*delta + 127] (within
//            [0, N)), is selected: such a tile is kept whole for every row.
//   clist    the valid selected columns, ascending, ccount of them; the
//            columns' K and V rows are then copied side by side
//            (vs_colgather_kernel), so that the attention kernel loads the
//            column tiles with plain TMA boxes.
// Block-expanded mode (every 64x64 block a selected diagonal crosses is kept):
//   offbits then holds D64, bit e set for the 64-block distances e = o/64 and
//            (o % 64 != 0) o/64 + 1 of the selected offsets, and e = 0;
//   dbits    bit delta set when one of the 64-block distances 2 delta - 1,
//            2 delta, 2 delta + 1 (those of the four 64x64 sub-blocks of a
//            128x128 tile at distance delta) is in D64;
//   dfull    bit delta (> 0) set when all three are.
// All are O(N/32 + k) words per head, the same for every row block.  The
// entries are validated here: a value out of [0, N) or not strictly above its
// predecessor raises MI_ERR_INDEX in the status word and is skipped; -1 is
// padding, and a value after padding is invalid.
#pragma once

#include "common.cuh"

namespace mi {

struct VsIndexArgs {
  int N, k_v, k_s, Nw, NT, NTw;
  int expanded;  // block-expanded mode
  const int32_t* v_idx;
  const int32_t* s_idx;
  uint32_t* offbits;
  uint32_t* colbits;
  uint32_t* dbits;
  uint32_t* dfull;
  int* dlist;
  int* dcount;
  int* clist;   // [n_heads, MI_MAX_KV]
  int* ccount;  // [n_heads]
  int* status;
};

// 0: padding, 1: valid, -1: invalid.
__device__ __forceinline__ int classify_entry(const int32_t* idx, int e, int N) {
  const int v = idx[e];
  if (v == -1) return 0;
  if (v < 0 || v >= N) return -1;
  if (e > 0) {
    const int p = idx[e - 1];
    if (p == -1 || p >= v) return -1;
  }
  return 1;
}

__global__ void __launch_bounds__(512) vs_index_kernel(const __grid_constant__ VsIndexArgs a) {
  __shared__ uint32_t db[512];
  __shared__ int scan[512];
  const int n = blockIdx.x, tid = threadIdx.x;
  uint32_t* off = a.offbits + (size_t)n * a.Nw;
  uint32_t* col = a.colbits + (size_t)n * a.Nw;
  for (int w = tid; w < a.Nw; w += 512) {
    off[w] = 0u;
    col[w] = 0u;
  }
  db[tid] = 0u;
  __syncthreads();
  const int32_t* si = a.s_idx + (size_t)n * a.k_s;
  for (int e = tid; e < a.k_s; e += 512) {
    const int c = classify_entry(si, e, a.N);
    if (c < 0) set_status(a.status, MI_ERR_INDEX);
    if (c != 1) continue;
    const int o = si[e];
    if (a.expanded) {
      const int b0 = o >> 6;  // 64-block distances the diagonal crosses
      atomicOr(off + (b0 >> 5), 1u << (b0 & 31));
      if ((o & 63) && 64 * (b0 + 1) < a.N) atomicOr(off + ((b0 + 1) >> 5), 1u << ((b0 + 1) & 31));
      continue;
    }
    atomicOr(off + (o >> 5), 1u << (o & 31));
    const int d0 = o >> 7;
    atomicOr(&db[d0 >> 5], 1u << (d0 & 31));
    if ((o & 127) && d0 + 1 < a.NT) atomicOr(&db[(d0 + 1) >> 5], 1u << ((d0 + 1) & 31));
  }
  if (a.expanded && tid == 0) atomicOr(off, 1u);  // distance 0: the query's own 64-block
  const int32_t* vi = a.v_idx + (size_t)n * a.k_v;
  for (int e = tid; e < a.k_v; e += 512) {
    const int c = classify_entry(vi, e, a.N);
    if (c < 0) set_status(a.status, MI_ERR_INDEX);
    if (c != 1) continue;
    const int j = vi[e];
    atomicOr(col + (j >> 5), 1u << (j & 31));
  }
  if (tid == 0) atomicOr(&db[0], 1u);
  __syncthreads();
  {
    // the valid columns, ascending (the bitmap was just built with atomics: read
    // back through L2); their count is at most k_v <= MI_MAX_KV
    __shared__ int cs[512];
    const int per = (a.Nw + 511) / 512;
    const int w0 = min(tid * per, a.Nw), w1 = min(w0 + per, a.Nw);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(__ldcg(col + w));
    cs[tid] = cnt;
    __syncthreads();
    for (int o = 1; o < 512; o <<= 1) {
      const int y = (tid >= o) ? cs[tid - o] : 0;
      __syncthreads();
      cs[tid] += y;
      __syncthreads();
    }
    int pos = cs[tid] - cnt;
    int* cl = a.clist + (size_t)n * MI_MAX_KV;
    for (int w = w0; w < w1; ++w)
      for (uint32_t m = __ldcg(col + w); m; m &= m - 1) cl[pos++] = 32 * w + __ffs(m) - 1;
    if (tid == 511) a.ccount[n] = cs[511];
  }
  if (a.expanded) {
    // 128-tile distance delta: its sub-blocks sit at 64-block distances
    // 2 delta - 1 .. 2 delta + 1 (read back through L2: built with atomics)
    const int NB = (a.N + 63) >> 6;
    for (int d = tid; d < a.NT; d += 512) {
      bool any = false;
      for (int e = 2 * d - 1; e <= 2 * d + 1; ++e)
        if (e >= 0 && e < NB && ((__ldcg(off + (e >> 5)) >> (e & 31)) & 1u)) any = true;
      if (any) atomicOr(&db[d >> 5], 1u << (d & 31));
    }
    __syncthreads();
  }
  // tile distances whose whole offset window is selected (read back through L2:
  // the bitmap was just built with atomics)
  __shared__ uint32_t dfw[512];
  dfw[tid] = 0u;
  __syncthreads();
  for (int d = 1 + tid; d < a.NT; d += 512) {
    bool all = true;
    if (a.expanded) {
      const int NB = (a.N + 63) >> 6;
      for (int e = 2 * d - 1; e <= 2 * d + 1 && all; ++e)
        all = e < NB && ((__ldcg(off + (e >> 5)) >> (e & 31)) & 1u);
    } else {
      const int lo = 128 * d - 127, hi = min(128 * d + 127, a.N - 1);  // inclusive
      for (int w = lo >> 5; w <= (hi >> 5) && all; ++w) {
        uint32_t need = 0xFFFFFFFFu;
        if (w == (lo >> 5)) need &= 0xFFFFFFFFu << (lo & 31);
        if (w == (hi >> 5)) need &= 0xFFFFFFFFu >> (31 - (hi & 31));
        all = (__ldcg(off + w) & need) == need;
      }
    }
    if (all) atomicOr(&dfw[d >> 5], 1u << (d & 31));
  }
  __syncthreads();
  if (tid < a.NTw) a.dfull[(size_t)n * a.NTw + tid] = dfw[tid];
  // dbits to global, then the ascending list of set distances
  const uint32_t word = (tid < a.NTw) ? db[tid] : 0u;
  if (tid < a.NTw) a.dbits[(size_t)n * a.NTw + tid] = word;
  scan[tid] = __popc(word);
  __syncthreads();
  for (int o = 1; o < 512; o <<= 1) {
    const int y = (tid >= o) ? scan[tid - o] : 0;
    __syncthreads();
    scan[tid] += y;
    __syncthreads();
  }
  int pos = scan[tid] - __popc(word);
  int* dl = a.dlist + (size_t)n * a.NT;
  for (uint32_t w = word; w; w &= w - 1) dl[pos++] = tid * 32 + (__ffs(w) - 1);
  if (tid == 511) a.dcount[n] = scan[511];
}

// Compacted K and V rows of the selected columns: row i of head slot n is row
// clist[n][i] of its KV head for i < ccount[n], and zero up to the next 128
// rows past it (a column tile starting below ccount may read that far; TMA
// reads past MI_MAX_KV rows as zero).  One warp per row: lanes 0-15 copy K,
// 16-31 copy V, 16 bytes each.
__global__ void vs_colgather_kernel(const __nv_bfloat16* k, const __nv_bfloat16* v, int64_t ld, int group,
                                    HeadList heads, const int* clist, const int* ccount,
                                    __nv_bfloat16* kc, __nv_bfloat16* vc) {
  const int n = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int cnt = ccount[n];
  if (i >= min(cnt + 128, MI_MAX_KV)) return;
  const int g = heads.h[n] / group;
  const __nv_bfloat16* src = (lane < 16) ? k : v;
  __nv_bfloat16* dst = ((lane < 16) ? kc : vc) + ((size_t)n * MI_MAX_KV + i) * kD + (lane & 15) * 8;
  uint4 val = make_uint4(0u, 0u, 0u, 0u);
  if (i < cnt) {
    const int j = clist[(size_t)n * MI_MAX_KV + i];
    val = *reinterpret_cast<const uint4*>(src + ((size_t)g * ld + j) * kD + (lane & 15) * 8);
  }
  *reinterpret_cast<uint4*>(dst) = val;
}

}  // namespace mi
