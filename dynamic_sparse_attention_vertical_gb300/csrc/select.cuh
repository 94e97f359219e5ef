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
#include "pdl.cuh"

namespace mi {

// Lanes of the warp whose 8-bit value equals this lane's, among the lanes with
// act set (meaningful for active lanes only): one ballot per bit, cheaper than a
// warp match over 32-bit values (measured: the radix passes of the top-k
// 20-25 % faster, the block selection 3 %).
__device__ __forceinline__ unsigned match8(uint32_t bin, bool act) {
  unsigned m = __ballot_sync(0xffffffffu, act);
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const unsigned bb = __ballot_sync(0xffffffffu, (bin >> b) & 1u);
    m &= ((bin >> b) & 1u) ? bb : ~bb;
  }
  return m;
}

// The bin holding the rem-th largest key of a 256-bin histogram (bins in
// ascending key order) and the rank of that key inside the bin, found by one
// warp: lane L covers bins 255-8L .. 248-8L (descending).  Requires
// 1 <= rem <= the histogram's total; every lane returns the same values.
__device__ __forceinline__ void hist_pick(const int* hist, int rem, int* bin_out, int* rem_out) {
  const int lane = threadIdx.x & 31;
  const int4 lo = *reinterpret_cast<const int4*>(hist + 248 - 8 * lane);
  const int4 hi = *reinterpret_cast<const int4*>(hist + 252 - 8 * lane);
  const int c[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};  // bins 255-8L down
  int tot = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) tot += c[e];
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  const int excl = incl - tot;
  const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
  const int leader = __ffs(hit) - 1;
  int bin = 0, r = 0, cum = excl;
  bool found = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (!found && cum + c[e] >= rem) {
      found = true;
      bin = 255 - (lane * 8 + e);
      r = rem - cum;
    }
    cum += c[e];
  }
  *bin_out = __shfl_sync(0xffffffffu, bin, leader);
  *rem_out = __shfl_sync(0xffffffffu, r, leader);
}

struct SelectSmem {
  alignas(16) int hist[3][256];  // one per radix pass, rotating
  int wgt[32];
  int weq[32];
};

// The key of the k-th largest of n keys (1 <= k <= n) by a 4-pass 8-bit radix
// select; *rem_out receives how many elements equal to that key are among the
// top k.  All NT threads of the block must call it; no early exit.  One block
// barrier per pass: every warp scans the pass's histogram itself, and the
// histograms rotate over three buffers, so that a buffer is cleared (after the
// barrier of the pass that follows its last reading) one barrier before it is
// filled again.
template <int NT, class F>
__device__ uint32_t radix_kth_key(F key_at, int n, int k, SelectSmem& sm, int* rem_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  __syncthreads();  // earlier readers of the buffers are done
  for (int i = tid; i < 512; i += NT) (&sm.hist[0][0])[i] = 0;
  __syncthreads();
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int* h = sm.hist[pass % 3];
    for (int base = warp * 32; base < n; base += NT) {
      const int i = base + lane;
      bool act = false;
      uint32_t bin = 0;
      if (i < n) {
        const uint32_t u = key_at(i);
        act = (u & pmask) == prefix;
        bin = (u >> shift) & 255u;
      }
      const unsigned peers = match8(bin, act);
      if (act && lane == __ffs(peers) - 1) atomicAdd(&h[bin], __popc(peers));
    }
    __syncthreads();
    if (pass == 0 || pass == 1) {  // the buffer of pass + 2, last read in pass - 1
      int* z = sm.hist[(pass + 2) % 3];
      for (int i = tid; i < 256; i += NT) z[i] = 0;
    }
    int bin, r;
    hist_pick(h, rem, &bin, &r);
    prefix |= static_cast<uint32_t>(bin) << shift;
    pmask |= 0xFFu << shift;
    rem = r;
  }
  *rem_out = rem;
  return prefix;
}

// Ordered take: out receives, ascending, every i with key > kth plus the first
// `rem` i with key == kth (warp w sweeps its own contiguous segment).
template <int NT, class F>
__device__ void take_sorted(F key_at, int n, uint32_t kth, int rem, int* out, SelectSmem& sm) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = cdiv(cdiv(n, NW), 32) * 32;
  const int beg = min(warp * seg, n), end = min(beg + seg, n);
  int gt = 0, eq = 0;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const uint32_t u = (i < end) ? key_at(i) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, i < end && u > kth));
    eq += __popc(__ballot_sync(0xffffffffu, i < end && u == kth));
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
    const bool isg = i < end && u > kth;
    const bool ise = i < end && u == kth;
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

// key_at(i) -> order-preserving uint32 key of element i (see float_key).
// Requires 1 <= k <= n.  Writes the k selected indices ascending to out[0..k).
// All NT threads of the block must call it.  The function has no early exit:
// every thread runs every block barrier in it.
template <int NT, class F>
__device__ void topk_select_sorted(F key_at, int n, int k, int* out, SelectSmem& sm) {
  int rem;
  const uint32_t kth = radix_kth_key<NT>(key_at, n, k, sm, &rem);
  take_sorted<NT>(key_at, n, kth, rem, out, sm);
}

// The same selection by one warp (for small n: the block selection of 64x64
// blocks, n <= N / 64), so that the warps of a CTA select for different rows at
// once.  hist: 256 ints of shared memory owned by the warp, 16-byte aligned.
// The same 4-pass 8-bit radix select for the k-th key, then one ordered sweep;
// ties to the lower index, output ascending.  Requires 1 <= k <= n; every lane
// must call it.
template <class F>
__device__ void warp_topk_sorted(F key_at, int n, int k, int* out, int* hist) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int base = 0; base < n; base += 128) {  // four keys per lane read ahead
      uint32_t u[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = base + 32 * q + lane;
        u[q] = (i < n) ? key_at(i) : 0u;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool act = base + 32 * q + lane < n && (u[q] & pmask) == prefix;
        const uint32_t bin = (u[q] >> shift) & 255u;
        const unsigned peers = match8(bin, act);
        if (act && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
    }
    __syncwarp();
    int bin_sel, rem_new;
    hist_pick(hist, rem, &bin_sel, &rem_new);
    rem = rem_new;
    prefix |= static_cast<uint32_t>(bin_sel) << shift;
    pmask |= 0xFFu << shift;
    __syncwarp();
  }
  const uint32_t kth = prefix;
  const unsigned lt = (1u << lane) - 1u;
  int gb = 0, eb = 0;
  for (int base = 0; base < n; base += 128) {
    uint32_t u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = base + 32 * q + lane;
      u[q] = (i < n) ? key_at(i) : 0u;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // in index order
      const int i = base + 32 * q + lane;
      const bool isg = i < n && u[q] > kth;
      const bool ise = i < n && u[q] == kth;
      const unsigned bg = __ballot_sync(0xffffffffu, isg);
      const unsigned be = __ballot_sync(0xffffffffu, ise);
      const int G = gb + __popc(bg & lt), E = eb + __popc(be & lt);
      if (isg) out[G + min(E, rem)] = i;
      else if (ise && E < rem) out[G + E] = i;
      gb += __popc(bg);
      eb += __popc(be);
    }
  }
}

// T1: top-k of the vertical (y = 0) or slash (y = 1) scores of every listed head;
// k > N keeps all N indices, and the row is padded with -1 up to the row stride.
//
// For k much smaller than N a threshold filter does most of the work in two
// passes over the scores: the key at rank about 1.25 k S / N (+ 16) of a strided
// sample of S scores (one in 64, 2048 to 8192 of them) is a threshold that about
// 1.25 k scores reach (measured: the radix select over an 8192-score sample took a
// third of the kernel at 128K); the scores at or above it are compacted, in index
// order, into shared memory, and the exact selection runs on them.  If at least k scores reach the threshold, every
// element of the top k (ties at the k-th key included) is among them, so the
// result is the same as selecting over all N; otherwise, or if they do not fit,
// the selection runs over all N.
constexpr int kTopkU = 4;  // float4 quads per lane in flight in the threshold sweeps

// Quads base + 128 u + 4 lane (u < U) of x, each read whole when it starts before
// end (end and base multiples of 4, x 16-byte aligned); the others are zero.
template <int U>
__device__ __forceinline__ void load_quads(const float* x, int base, int end, int lane, float4* q) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = base + u * 128 + lane * 4;
    q[u] = (i < end) ? __ldg(reinterpret_cast<const float4*>(x + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

constexpr int kTopkSample = 8192;
constexpr int kTopkSampleMin = 2048;
constexpr int kTopkCand = 20480;
struct TopkSmem {
  SelectSmem sel;
  uint32_t samp[kTopkSample];
  uint32_t ckey[kTopkCand];
  int cidx[kTopkCand];
  int wcnt[32];
};
constexpr size_t kTopkSmemBytes = sizeof(TopkSmem);

__global__ void __launch_bounds__(1024, 1)
vs_topk_kernel(const float* vsc, const float* ssc, int N, int k_v, int k_s, int32_t* v_idx,
               int32_t* s_idx, int ld_v, int ld_s) {
  extern __shared__ uint8_t topk_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_raw);
  pdl_wait();  // launched as the dependent of estimation pass 2: its scores
  constexpr int NT = 1024, NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = blockIdx.x;
  const bool vert = blockIdx.y == 0;
  const float* x = (vert ? vsc : ssc) + (size_t)slot * N;
  const int k = vert ? k_v : k_s;
  const int ld = vert ? ld_v : ld_s;  // row stride >= k; the rest of a row is padding
  const int kk = min(k, N);
  int32_t* out = (vert ? v_idx : s_idx) + (size_t)slot * ld;
  auto gkey = [x](int i) { return float_key(__ldg(x + i)); };
  bool done = kk == 0;
  // the sample: one score in 64, between 2048 and kTopkSample of them
  const int S = min(kTopkSample, max(kTopkSampleMin, N >> 6));
  if (!done && N >= 4 * S && 4 * kk <= 3 * kTopkCand) {
    for (int j = tid; j < S; j += NT)
      sm.samp[j] = gkey(static_cast<int>((static_cast<int64_t>(j) * N) / S));
    __syncthreads();
    const int rs = min(S, static_cast<int>((5ll * kk * S) / (4ll * N)) + 16);
    int rem_s;
    const uint32_t* sp = sm.samp;
    const uint32_t tau = radix_kth_key<NT>([sp](int j) { return sp[j]; }, S, rs, sm.sel, &rem_s);
    // count the scores at or above the threshold, warp by warp over contiguous
    // segments; with N a multiple of 4 each lane reads float4 quads, kTopkU of them
    // in flight (the sweeps are bound by load latency), else one score at a time
    const bool vec = (N & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    constexpr int kSpan = 128 * kTopkU;  // scores per warp and vector step
    const int seg = cdiv(cdiv(N, NW), kSpan) * kSpan;
    const int beg = min(warp * seg, N), end = min(beg + seg, N);
    int c = 0;
    if (vec) {
      for (int base = beg; base < end; base += kSpan) {
        float4 q[kTopkU];
        load_quads<kTopkU>(x, base, end, lane, q);
#pragma unroll
        for (int u = 0; u < kTopkU; ++u) {
          if (base + u * 128 + lane * 4 < end)  // then all four are (end is a multiple of 4)
            c += (float_key(q[u].x) >= tau) + (float_key(q[u].y) >= tau) + (float_key(q[u].z) >= tau) +
                 (float_key(q[u].w) >= tau);
        }
      }
      c = __reduce_add_sync(0xffffffffu, c);
    } else {
      for (int base = beg; base < end; base += 32) {
        const int i = base + lane;
        c += __popc(__ballot_sync(0xffffffffu, i < end && gkey(i) >= tau));
      }
    }
    if (lane == 0) sm.wcnt[warp] = c;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < NW; ++w) {
      total += sm.wcnt[w];
      if (w < warp) before += sm.wcnt[w];
    }
    if (total >= kk && total <= kTopkCand) {  // the same for every thread
      const unsigned lt = (1u << lane) - 1u;
      if (vec) {
        for (int base = beg; base < end; base += kSpan) {
          float4 q[kTopkU];
          load_quads<kTopkU>(x, base, end, lane, q);
#pragma unroll
          for (int u = 0; u < kTopkU; ++u) {
            const int i0 = base + u * 128 + lane * 4;
            const uint32_t kq[4] = {float_key(q[u].x), float_key(q[u].y), float_key(q[u].z), float_key(q[u].w)};
            bool in[4];
            unsigned b[4];
            int below = 0, all = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              in[e] = i0 < end && kq[e] >= tau;
              b[e] = __ballot_sync(0xffffffffu, in[e]);
              below += __popc(b[e] & lt);
              all += __popc(b[e]);
            }
            // lane order, then the quad's own order: the list stays in index order
            int p = before + below;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (in[e]) {
                sm.ckey[p] = kq[e];
                sm.cidx[p] = i0 + e;
                ++p;
              }
            }
            before += all;
          }
        }
      } else {
        for (int base = beg; base < end; base += 32) {
          const int i = base + lane;
          const uint32_t u = (i < end) ? gkey(i) : 0u;
          const bool in = i < end && u >= tau;
          const unsigned b = __ballot_sync(0xffffffffu, in);
          if (in) {
            const int p = before + __popc(b & lt);
            sm.ckey[p] = u;
            sm.cidx[p] = i;
          }
          before += __popc(b);
        }
      }
      __syncthreads();
      const uint32_t* ck = sm.ckey;
      topk_select_sorted<NT>([ck](int j) { return ck[j]; }, total, kk, out, sm.sel);
      // candidate positions -> score indices (each thread its own entries)
      for (int j = tid; j < kk; j += NT) out[j] = sm.cidx[out[j]];
      done = true;
    }
    __syncthreads();
  }
  if (!done) topk_select_sorted<NT>(gkey, N, kk, out, sm.sel);
  for (int i = kk + tid; i < ld; i += NT) out[i] = -1;
}

}  // namespace mi
