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
//     modality, estimated from the 64 rows ending at that modality's last token.
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

}  // namespace mi
