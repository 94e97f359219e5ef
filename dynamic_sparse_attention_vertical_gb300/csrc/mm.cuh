// mm.cuh - the multi-modal heads' index steps: the grid lattice fit, the grid's
// column lattice, and the modality bookkeeping of Q-boundary heads.
//
// MMInference (MInference README mirror, gittoolsai.com, "TL;DR"; talk slides,
// boteman.cn, "MMInference: Grid Head in Multi-Modality" and "MMInference:
// Q-Boundary pattern").  Readings:
//   grid: one lattice j = phi (mod sigma) gives the vertical lines (key
//     columns) and the horizontal lines (query rows that keep their whole
//     causal row); (sigma, phi) maximises E(sigma, phi) = sum of the vertical
//     scores v over the lattice - lattice size * last_q / N over
//     sigma_min..sigma_max, ties to the smaller sigma, then phi;
//   Q-boundary: a query row follows the vertical-slash pattern of its own
//     modality, estimated from the 64 rows ending at that modality's last token;
//   2D-boundary (two modalities, given as runs): each modality's tokens, in
//     order, are a sub-sequence in which the modality is a vertical-slash head
//     (the tokens are permuted so that each sub-sequence is contiguous); keys of
//     the other modality before a query are all kept (the cross-modality pass),
//     and the two partial softmaxes are merged by their log-sum-exps.
#pragma once

#include "common.cuh"

namespace mi {

constexpr int kFitThreads = 1024;

// E(sigma, phi) for every phi of one sigma (blockIdx.x = sigma - sigma_min) of one
// listed head (blockIdx.y), and the best phi: best[head][sigma - sigma_min] =
// (E, phi).  Sums run in a fixed order (parts of each residue class in order),
// so the result is deterministic.
__global__ void __launch_bounds__(kFitThreads)
grid_fit_kernel(const float* vsc, int N, int sigma_min, int n_sigma, float mass, float2* best) {
  __shared__ float part[kFitThreads];
  __shared__ float be[32];
  __shared__ int bp[32];
  const int sigma = sigma_min + blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
  const float* v = vsc + (size_t)n * N;
  const float avg = mass / static_cast<float>(N);
  float e_best = -INFINITY;
  int p_best = 0x7FFFFFFF;
  if (sigma <= kFitThreads) {
    // P parts per residue class: thread t sums v[phi + sigma (part + P m)]
    const int P = kFitThreads / sigma;
    const int phi = tid % sigma, pt = tid / sigma;
    float acc = 0.f;
    if (pt < P)
      for (int j = phi + sigma * pt; j < N; j += sigma * P) acc += v[j];
    part[tid] = acc;
    __syncthreads();
    if (tid < sigma) {
      float sum = 0.f;
      for (int u = 0; u < P; ++u) sum += part[u * sigma + tid];
      const int cnt = (tid < N) ? (N - 1 - tid) / sigma + 1 : 0;
      e_best = sum - static_cast<float>(cnt) * avg;
      p_best = tid;
    }
  } else {
    for (int phi = tid; phi < sigma; phi += kFitThreads) {
      float sum = 0.f;
      for (int j = phi; j < N; j += sigma) sum += v[j];
      const int cnt = (phi < N) ? (N - 1 - phi) / sigma + 1 : 0;
      const float e = sum - static_cast<float>(cnt) * avg;
      if (e > e_best) {  // phi ascending: the first maximum stays
        e_best = e;
        p_best = phi;
      }
    }
  }
  // the largest E, then the smaller phi
  for (int off = 16; off > 0; off >>= 1) {
    const float e2 = __shfl_xor_sync(0xffffffffu, e_best, off);
    const int p2 = __shfl_xor_sync(0xffffffffu, p_best, off);
    if (e2 > e_best || (e2 == e_best && p2 < p_best)) {
      e_best = e2;
      p_best = p2;
    }
  }
  if ((tid & 31) == 0) {
    be[tid >> 5] = e_best;
    bp[tid >> 5] = p_best;
  }
  __syncthreads();
  if (tid < 32) {
    e_best = be[tid];
    p_best = bp[tid];
    for (int off = 16; off > 0; off >>= 1) {
      const float e2 = __shfl_xor_sync(0xffffffffu, e_best, off);
      const int p2 = __shfl_xor_sync(0xffffffffu, p_best, off);
      if (e2 > e_best || (e2 == e_best && p2 < p_best)) {
        e_best = e2;
        p_best = p2;
      }
    }
    if (tid == 0) best[(size_t)n * n_sigma + blockIdx.x] = make_float2(e_best, __int_as_float(p_best));
  }
}

// Per listed head: the sigma with the largest E (ties: the smaller sigma) -> grid[n] = (sigma, phi).
__global__ void grid_pick_kernel(const float2* best, int n_heads, int sigma_min, int n_sigma, int32_t* grid) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= n_heads) return;
  float e_best = -INFINITY;
  int s_best = 0, p_best = 0;
  for (int u = 0; u < n_sigma; ++u) {
    const float2 b = best[(size_t)n * n_sigma + u];
    if (u == 0 || b.x > e_best) {
      e_best = b.x;
      s_best = sigma_min + u;
      p_best = __float_as_int(b.y);
    }
  }
  grid[2 * n] = s_best;
  grid[2 * n + 1] = p_best;
}

// The grid heads' vertical lines as column lists: v_idx[n][i] = phi + i sigma
// (ascending, -1 after the last one below N).  A (sigma, phi) below sigma_min,
// with phi outside [0, sigma), or with more columns than ld raises MI_ERR_INDEX
// and gets an empty list.
__global__ void grid_lattice_kernel(const int32_t* grid, int N, int sigma_min, int ld, int32_t* v_idx,
                                    int* status) {
  const int n = blockIdx.x;
  const int sigma = grid[2 * n], phi = grid[2 * n + 1];
  bool ok = sigma >= sigma_min && phi >= 0 && phi < sigma;
  const int cnt = (ok && phi < N) ? (N - 1 - phi) / sigma + 1 : 0;
  if (cnt > ld) ok = false;
  if (!ok && threadIdx.x == 0) set_status(status, MI_ERR_INDEX);
  for (int i = threadIdx.x; i < ld; i += blockDim.x)
    v_idx[(size_t)n * ld + i] = (ok && i < cnt) ? phi + i * sigma : -1;
}

// Q-boundary bookkeeping from the modality ids: ends[m] = one past the last
// token of modality m (the estimation window of m ends there), and per 128-row
// block a bit per modality present (row blocks without the modality of an
// attention pass are skipped).  ends and blk_mods must be zero on entry.  An id
// outside [0, n_mod) raises MI_ERR_INDEX.
__global__ void modality_scan_kernel(const int32_t* modality, int N, int n_mod, int* ends, uint32_t* blk_mods,
                                     int* status) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  const int m = modality[j];
  if (m < 0 || m >= n_mod) {
    set_status(status, MI_ERR_INDEX);
    return;
  }
  atomicMax(&ends[m], j + 1);
  atomicOr(&blk_mods[j / kBM], 1u << m);
}

// The token runs of a 2D-boundary call: run u covers original tokens
// start[u] .. start[u] + len[u] - 1, all of modality mod[u] (0 or 1), which sit
// at permuted positions pstart[u] .. (modality 0's tokens first, in order).
constexpr int kMaxRuns = MI_MAX_RUNS;
struct RunTable {
  int n;
  int start[kMaxRuns], pstart[kMaxRuns], len[kMaxRuns], mod[kMaxRuns];
};

__device__ __forceinline__ int run_of(const RunTable& rt, int j) {
  int lo = 0, hi = rt.n - 1;  // the last run starting at or before j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rt.start[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Rows of q (heads 0..hq-1), k and v (heads 0..hkv-1), all [heads, N, 128] bf16,
// copied to their permuted positions; one warp per (tensor, head, token) row.
__global__ void boundary_gather_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                                       int hq, int hkv, int N, const __grid_constant__ RunTable rt,
                                       __nv_bfloat16* qp, __nv_bfloat16* kp, __nv_bfloat16* vp) {
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t rows_q = (int64_t)hq * N, rows_kv = (int64_t)hkv * N;
  if (w >= rows_q + 2 * rows_kv) return;
  const __nv_bfloat16* src;
  __nv_bfloat16* dst;
  int64_t r;
  if (w < rows_q) {
    src = q; dst = qp; r = w;
  } else if (w < rows_q + rows_kv) {
    src = k; dst = kp; r = w - rows_q;
  } else {
    src = v; dst = vp; r = w - rows_q - rows_kv;
  }
  const int h = static_cast<int>(r / N), j = static_cast<int>(r - (int64_t)h * N);
  const int u = run_of(rt, j);
  const int p = rt.pstart[u] + (j - rt.start[u]);
  const uint2* s2 = reinterpret_cast<const uint2*>(src + ((size_t)h * N + j) * kD);
  uint2* d2 = reinterpret_cast<uint2*>(dst + ((size_t)h * N + p) * kD);
  d2[lane] = s2[lane];
}

// Bit j of modbits: token j is of modality 1; mods128[t]: bit m set when the
// 128-token block t holds a token of modality m.  modbits and mods128 must be
// zero on entry.
__global__ void boundary_bits_kernel(int N, const __grid_constant__ RunTable rt, uint32_t* modbits,
                                     uint32_t* mods128) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  const int m = rt.mod[run_of(rt, j)];
  if (m) atomicOr(&modbits[j >> 5], 1u << (j & 31));
  atomicOr(&mods128[j >> 7], 1u << m);
}

// out[h][j] (and lse) = the merge of the within-modality result (op / lse_in at the
// permuted position of j) and the cross-modality result already in out / lse_x:
// O = (e^{L1} O1 + e^{L2} O2) / (e^{L1} + e^{L2}).  One warp per (listed head, token).
__global__ void boundary_merge_kernel(int N, const __grid_constant__ RunTable rt, HeadList heads,
                                      const __nv_bfloat16* op, const float* lse_in, const float* lse_x,
                                      __nv_bfloat16* out, float* lse) {
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= (int64_t)heads.n * N) return;
  const int n = static_cast<int>(w / N), j = static_cast<int>(w - (int64_t)n * N);
  const int h = heads.h[n];
  const int u = run_of(rt, j);
  const int p = rt.pstart[u] + (j - rt.start[u]);
  const float l1 = lse_in[(size_t)h * N + p], l2 = lse_x[(size_t)h * N + j];
  const float m = fmaxf(l1, l2);
  const float w1 = (l1 == -INFINITY) ? 0.f : __expf(l1 - m), w2 = (l2 == -INFINITY) ? 0.f : __expf(l2 - m);
  const float inv = 1.f / (w1 + w2);
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(op + ((size_t)h * N + p) * kD) + 2 * lane;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(out + ((size_t)h * N + j) * kD) + 2 * lane;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float2 x1 = __bfloat1622float2(a[e]), x2 = __bfloat1622float2(b[e]);
    // a side with weight 0 (no key) takes no part, whatever its output holds
    const float2 y1 = (w1 > 0.f) ? make_float2(w1 * x1.x, w1 * x1.y) : make_float2(0.f, 0.f);
    const float2 y2 = (w2 > 0.f) ? make_float2(w2 * x2.x, w2 * x2.y) : make_float2(0.f, 0.f);
    b[e] = __floats2bfloat162_rn((y1.x + y2.x) * inv, (y1.y + y2.y) * inv);
  }
  if (lse && lane == 0) lse[(size_t)h * N + j] = m + logf(w1 + w2);
}

}  // namespace mi
