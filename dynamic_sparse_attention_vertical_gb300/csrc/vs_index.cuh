// vs_index.cuh - index structures of a vertical-slash head (one CTA per head).
//
// From the sorted column list V and offset list S the sparse attention kernel
// needs, per head:
//   offbits  bit o set for o in S             (element mask of diagonal tiles)
//   colbits  bit j set for j in V             (columns inside contiguous tiles)
//   dlist    key windows, dcount of them: row block r (rows 128 r ..) reads keys
//            128 r - p .. 128 r - p + 127 for every window p < 128 r, besides
//            tile 0 (keys 0 .. 127).  A window at p meets the offsets
//            p + i - 127 .. p + i in row i, so the windows must hit every
//            interval [x, x + 127] with x in [o - 127, o] for each selected
//            offset o (and o = 0, the query's own block).  The greedy hitting
//            set starts at p = 0 and moves to p + 128 while a selected offset
//            lies in (p, p + 128], else to the next selected offset.  Windows
//            are at least 128 apart, so they never overlap; unlike 128-aligned
//            tiles they need one tile, not two, for an isolated diagonal.
//   dfull    bit i set when window i is kept whole: every offset it can meet,
//            [p - 127, p + 127] (within [0, N)), is selected.
//   dbits    bit x + 128 set when some window covers key distance x = 128 r - j
//            (x in [p - 127, p]): the columns no window covers are residual.
//   clist    the valid selected columns, ascending, ccount of them; the
//            columns' K and V rows are then copied side by side
//            (vs_colgather_kernel), so that the attention kernel loads the
//            column tiles with plain TMA boxes.
// Block-expanded mode (every 64x64 block a selected diagonal crosses is kept):
//   offbits then holds D64, bit e set for the 64-block distances e = o/64 and
//            (o % 64 != 0) o/64 + 1 of the selected offsets, and e = 0; the
//            attention kernel derives each row block's needed 64-key blocks
//            from it and pairs them two per tile (dbits, dlist, dfull unused).
// All are O(N/32 + k) words per head, the same for every row block.  The
// entries are validated here: a value out of [0, N) or not strictly above its
// predecessor raises MI_ERR_INDEX in the status word and is skipped; -1 is
// padding, and a value after padding is invalid.
#pragma once

#include "common.cuh"

namespace mi {

struct VsIndexArgs {
  int N, k_v, k_s, Nw, NT, NTw;
  int Dw;        // words of dbits per head (Nw + 8: the window coverage bits)
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

// Block-wide exclusive scan of one int per thread (512 threads); returns the
// exclusive prefix and writes the total to *total.  Ends with a barrier.
__device__ __forceinline__ int scan512(int x, int* scratch, int* total) {
  const int tid = threadIdx.x;
  scratch[tid] = x;
  __syncthreads();
  for (int o = 1; o < 512; o <<= 1) {
    const int y = (tid >= o) ? scratch[tid - o] : 0;
    __syncthreads();
    scratch[tid] += y;
    __syncthreads();
  }
  const int incl = scratch[tid];
  *total = scratch[511];
  __syncthreads();
  return incl - x;
}

// Windows of the chain that starts at run ks (runs: maximal groups of selected
// offsets at most 128 apart, first offsets runA, last offsets runL).  The chain
// starts at p = runA[ks]; inside a run p moves by 128 until it reaches the run's
// last offset (the offsets are at most 128 apart there, so one lies in every
// (p, p + 128]); the next run continues the chain at p + 128 when its first
// offset is within 128 of p, else the chain jumps to that offset.  A run that
// starts more than 255 past the previous run's last offset is always jumped to
// (p is below that offset + 128), so the chain ends there and a new one starts.
// Writes the windows p < N to out (when out is not null) and returns their count.
__device__ int vs_window_chain(const int* runA, const int* runL, int R, int ks, int N, int* out) {
  int p = runA[ks], cnt = 0;
  if (p >= N) return 0;
  if (out) out[cnt] = p;
  ++cnt;
  for (int k = ks;;) {
    const int last = runL[k];
    while (p < last) {
      p += 128;
      if (p >= N) return cnt;
      if (out) out[cnt] = p;
      ++cnt;
    }
    if (++k >= R || runA[k] - runL[k - 1] > 255) return cnt;
    p = (runA[k] <= p + 128) ? p + 128 : runA[k];
    if (p >= N) return cnt;
    if (out) out[cnt] = p;
    ++cnt;
  }
}

__global__ void __launch_bounds__(512) vs_index_kernel(const __grid_constant__ VsIndexArgs a) {
  __shared__ int scan[512];
  extern __shared__ int run_smem[];  // exact mode: run first offsets [NT + 1], run last offsets [NT + 1]
  const int n = blockIdx.x, tid = threadIdx.x;
  uint32_t* off = a.offbits + (size_t)n * a.Nw;
  uint32_t* col = a.colbits + (size_t)n * a.Nw;
  uint32_t* dbh = a.dbits + (size_t)n * a.Dw;
  for (int w = tid; w < a.Nw; w += 512) {
    off[w] = 0u;
    col[w] = 0u;
  }
  for (int w = tid; w < a.Dw; w += 512) dbh[w] = 0u;
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
  }
  // expanded: distance 0, the query's own 64-block; exact: offset 0, which the
  // own-block rule keeps anyway, so that the windows start at p = 0
  if (tid == 0) atomicOr(off, 1u);
  const int32_t* vi = a.v_idx + (size_t)n * a.k_v;
  for (int e = tid; e < a.k_v; e += 512) {
    const int c = classify_entry(vi, e, a.N);
    if (c < 0) set_status(a.status, MI_ERR_INDEX);
    if (c != 1) continue;
    const int j = vi[e];
    atomicOr(col + (j >> 5), 1u << (j & 31));
  }
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
  if (a.expanded) {  // the attention pairs the needed 64-key blocks from offbits alone
    if (tid == 0) a.dcount[n] = 0;
    return;
  }
  // ---- exact mode: key windows (the bitmap was built with atomics: read through L2)
  int* runA = run_smem;
  int* runL = run_smem + (a.NT + 1);
  const int per = (a.Nw + 511) / 512;
  const int w0 = min(tid * per, a.Nw), w1 = min(w0 + per, a.Nw);
  // the last selected offset in this thread's words, then before them (max-scan)
  int last = -1;
  for (int w = w1 - 1; w >= w0; --w) {
    const uint32_t m = __ldcg(off + w);
    if (m) {
      last = 32 * w + 31 - __clz(m);
      break;
    }
  }
  scan[tid] = last;
  __syncthreads();
  for (int o = 1; o < 512; o <<= 1) {
    const int y = (tid >= o) ? scan[tid - o] : -1;
    __syncthreads();
    scan[tid] = max(scan[tid], y);
    __syncthreads();
  }
  const int prev0 = (tid > 0) ? scan[tid - 1] : -1;
  const int last_all = scan[511];
  __syncthreads();
  // runs: a run starts at a selected offset more than 128 past the previous one
  int starts = 0;
  {
    int prev = prev0;
    for (int w = w0; w < w1; ++w)
      for (uint32_t m = __ldcg(off + w); m; m &= m - 1) {
        const int o = 32 * w + __ffs(m) - 1;
        starts += (prev < 0 || o - prev > 128) ? 1 : 0;
        prev = o;
      }
  }
  int R;
  int k = scan512(starts, scan, &R);
  R = min(R, a.NT + 1);  // at most NT runs of offsets below N (runs are more than 128 apart)
  {
    int prev = prev0;
    for (int w = w0; w < w1; ++w)
      for (uint32_t m = __ldcg(off + w); m; m &= m - 1) {
        const int o = 32 * w + __ffs(m) - 1;
        if ((prev < 0 || o - prev > 128) && k < R) {
          runA[k] = o;
          if (k > 0) runL[k - 1] = prev;
          ++k;
        }
        prev = o;
      }
  }
  if (tid == 0 && R > 0) runL[R - 1] = last_all;
  __syncthreads();
  // one chain per thread and group of runs (a group starts more than 255 past the
  // previous run's last offset): count the windows, place the chains, write them
  const int pr = (R + 511) / 512;
  const int k0 = min(tid * pr, R), k1 = min(k0 + pr, R);
  int nw = 0;
  for (int kk = k0; kk < k1; ++kk)
    if (kk == 0 || runA[kk] - runL[kk - 1] > 255) nw += vs_window_chain(runA, runL, R, kk, a.N, nullptr);
  int W;
  int base = scan512(nw, scan, &W);
  int* dl = a.dlist + (size_t)n * a.NT;
  for (int kk = k0; kk < k1; ++kk)
    if (kk == 0 || runA[kk] - runL[kk - 1] > 255) base += vs_window_chain(runA, runL, R, kk, a.N, dl + base);
  __syncthreads();
  // whole windows, and the key distances the windows cover
  __shared__ uint32_t dfw[512];
  dfw[tid] = 0u;
  __syncthreads();
  for (int i = tid; i < W; i += 512) {
    const int p = __ldcg(dl + i);
    bool all = p >= 128;
    const int lo = p - 127, hi = min(p + 127, a.N - 1);  // inclusive
    for (int w = lo >> 5; w <= (hi >> 5) && all; ++w) {
      uint32_t need = 0xFFFFFFFFu;
      if (w == (lo >> 5)) need &= 0xFFFFFFFFu << (lo & 31);
      if (w == (hi >> 5)) need &= 0xFFFFFFFFu >> (31 - (hi & 31));
      all = (__ldcg(off + w) & need) == need;
    }
    if (all) atomicOr(&dfw[i >> 5], 1u << (i & 31));
    for (int b = p + 1; b <= p + 128;) {  // bits x + 128, x = p - 127 .. p
      const int w = b >> 5, e = min(p + 128, 32 * w + 31);
      const uint32_t m = (0xFFFFFFFFu >> (31 - (e & 31))) & (0xFFFFFFFFu << (b & 31));
      atomicOr(dbh + w, m);
      b = e + 1;
    }
  }
  __syncthreads();
  if (tid < a.NTw) a.dfull[(size_t)n * a.NTw + tid] = dfw[tid];
  if (tid == 0) a.dcount[n] = W;
}

// Dynamic shared memory of vs_index_kernel: the runs of the exact mode.
inline size_t vs_index_smem(int NT) { return sizeof(int) * 2 * (size_t)(NT + 1); }

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
