// select.cuh - top-k selection by a block, a warp or a pair of CTAs (a
// thread-block cluster), returned in ascending index order.
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
// warp match over 32-bit values (measured: the top-k's two radix selects 13 and
// 25 % faster, the block selection 3 %).
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
// warp from the counts of bins 255-8L .. 248-8L (descending) in lane L's c[8].
// Requires 1 <= rem <= the histogram's total; every lane returns the same values.
__device__ __forceinline__ void pick_bin(const int (&c)[8], int rem, int* bin_out, int* rem_out) {
  const int lane = threadIdx.x & 31;
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

// Lane L's counts c[8] of bins 255-8L .. 248-8L of a 16-byte aligned histogram.
__device__ __forceinline__ void hist_counts(const int* hist, int (&c)[8]) {
  const int lane = threadIdx.x & 31;
  const int4 lo = *reinterpret_cast<const int4*>(hist + 248 - 8 * lane);
  const int4 hi = *reinterpret_cast<const int4*>(hist + 252 - 8 * lane);
  c[0] = hi.w;
  c[1] = hi.z;
  c[2] = hi.y;
  c[3] = hi.x;
  c[4] = lo.w;
  c[5] = lo.z;
  c[6] = lo.y;
  c[7] = lo.x;
}

__device__ __forceinline__ void hist_pick(const int* hist, int rem, int* bin_out, int* rem_out) {
  int c[8];
  hist_counts(hist, c);
  pick_bin(c, rem, bin_out, rem_out);
}

struct SelectSmem {
  alignas(16) int hist[3][256];  // one per radix pass, rotating
  int wgt[32];
  int weq[32];
  int pick[2];  // the pass's bin and rank, from warp 0
};

// The key of the k-th largest of n keys (1 <= k <= n) by a 4-pass 8-bit radix
// select; *rem_out receives how many elements equal to that key are among the
// top k.  All NT threads of the block must call it; no early exit.  Per pass:
// the count, a barrier, warp 0 finds the bin while the other warps clear the
// histogram of two passes later (three rotating buffers: it was last read one
// pass earlier), and a barrier before every thread reads the bin.  (Every warp
// scanning the histogram itself, with one barrier per pass, was slower: 32
// warps reading and scanning the same 256 bins.)
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
    if (warp == 0) {
      int bin, r;
      hist_pick(h, rem, &bin, &r);
      if (lane == 0) {
        sm.pick[0] = bin;
        sm.pick[1] = r;
      }
    } else if (pass == 0 || pass == 1) {
      int* z = sm.hist[(pass + 2) % 3];
      for (int i = tid - 32; i < 256; i += NT - 32) z[i] = 0;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sm.pick[0]) << shift;
    pmask |= 0xFFu << shift;
    rem = sm.pick[1];
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

// ---- the two CTAs of a thread-block cluster (the pair of one score row)

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs: shared-memory writes of either CTA before it are
// visible to both after it (release / acquire); also a barrier of each CTA.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared-memory address of the same object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_st(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int4 cluster_ld4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// The radix select of radix_kth_key over the keys of both CTAs of a pair: n is
// this CTA's count of keys, k the rank among both CTAs' keys (1 <= k <= both
// counts).  Each CTA counts its own keys; after a cluster barrier warp 0 of
// each adds the other CTA's histogram (read through distributed shared memory)
// to its own and picks the bin, so both pick the same.  The histogram cleared
// in a pass was last read, by both warps 0, before that pass's cluster barrier.
// Both CTAs must call it; every thread of them runs every barrier.
template <int NT, class F>
__device__ uint32_t radix_kth_pair(F key_at, int n, int k, SelectSmem& sm, uint32_t peer, int* rem_out) {
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
    cluster_barrier();  // both CTAs' counts of this pass are in
    if (warp == 0) {
      int c[8];
      hist_counts(h, c);
      const uint32_t ra = cluster_addr(h + 248 - 8 * lane, peer);
      const int4 lo = cluster_ld4(ra), hi = cluster_ld4(ra + 16);
      c[0] += hi.w;
      c[1] += hi.z;
      c[2] += hi.y;
      c[3] += hi.x;
      c[4] += lo.w;
      c[5] += lo.z;
      c[6] += lo.y;
      c[7] += lo.x;
      int bin, r;
      pick_bin(c, rem, &bin, &r);
      if (lane == 0) {
        sm.pick[0] = bin;
        sm.pick[1] = r;
      }
    } else if (pass == 0 || pass == 1) {
      int* z = sm.hist[(pass + 2) % 3];
      for (int i = tid - 32; i < 256; i += NT - 32) z[i] = 0;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sm.pick[0]) << shift;
    pmask |= 0xFFu << shift;
    rem = sm.pick[1];
  }
  *rem_out = rem;
  return prefix;
}

// T1: top-k of the vertical (y = 0) or slash (y = 1) scores of every listed head;
// k > N keeps all N indices, and the row is padded with -1 up to the row stride.
// Each row is selected by a cluster of two CTAs (x = 2 slot + CTA rank).
//
// For k much smaller than N a threshold filter does most of the work in two
// passes over the scores: the key at rank about 1.25 k S / N (+ 16) of a strided
// sample of S scores (one in 64, 2048 to 8192 of them; both CTAs find the same)
// is a threshold that about 1.25 k scores reach.  Each CTA counts, then compacts
// in index order into its shared memory, the scores of its half of the row at or
// above it; the exact selection runs on both halves' candidates (the radix
// histograms summed over the pair, CTA 1's output placed after CTA 0's).  If at
// least k scores reach the threshold every element of the top k (ties at the
// k-th key included) is a candidate, so the result is the same as selecting over
// all N; otherwise, or if a half's candidates do not fit, CTA 0 alone selects
// over all N.  (One CTA per row took about 60 us at 128K, most of it in the two
// sweeps and the candidates' radix, which the pair halves.)
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
  uint32_t ckey[kTopkCand];  // this CTA's candidates, in index order
  int cidx[kTopkCand];
  int wcnt[32];
  int peer_cnt;  // written by the other CTA of the pair
  int peer_gt, peer_eq;
};
constexpr size_t kTopkSmemBytes = sizeof(TopkSmem);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(1024, 1)
vs_topk_kernel(const float* vsc, const float* ssc, int N, int k_v, int k_s, int32_t* v_idx,
               int32_t* s_idx, int ld_v, int ld_s) {
  extern __shared__ uint8_t topk_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_raw);
  pdl_wait();  // launched as the dependent of estimation pass 2: its scores
  constexpr int NT = 1024, NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_cta_rank(), peer = rank ^ 1u;
  const int slot = blockIdx.x >> 1;
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
  // every decision below is the same in both CTAs (the same inputs, or values
  // both read after a cluster barrier), so both run the same cluster barriers
  if (!done && N >= 4 * S && 4 * kk <= 3 * kTopkCand) {
    for (int j = tid; j < S; j += NT)
      sm.samp[j] = gkey(static_cast<int>((static_cast<int64_t>(j) * N) / S));
    __syncthreads();
    const int rs = min(S, static_cast<int>((5ll * kk * S) / (4ll * N)) + 16);
    int rem_s;
    const uint32_t* sp = sm.samp;
    const uint32_t tau = radix_kth_key<NT>([sp](int j) { return sp[j]; }, S, rs, sm.sel, &rem_s);
    // count the scores at or above the threshold, warp by warp over contiguous
    // segments (CTA 0 the first 32, CTA 1 the next 32); with N a multiple of 4
    // each lane reads float4 quads, kTopkU of them in flight (the sweeps are
    // bound by load latency), else one score at a time
    const bool vec = (N & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    constexpr int kSpan = 128 * kTopkU;  // scores per warp and vector step
    const int seg = cdiv(cdiv(N, 2 * NW), kSpan) * kSpan;
    const int gw = static_cast<int>(rank) * NW + warp;
    const int beg = min(gw * seg, N), end = min(beg + seg, N);
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
    int before = 0, mine = 0;
    for (int w = 0; w < NW; ++w) {
      mine += sm.wcnt[w];
      if (w < warp) before += sm.wcnt[w];
    }
    if (tid == 0) cluster_st(cluster_addr(&sm.peer_cnt, peer), mine);
    cluster_barrier();
    const int other = sm.peer_cnt;
    const int total = mine + other;
    if (total >= kk && mine <= kTopkCand && other <= kTopkCand) {
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
      const uint32_t* ck = sm.ckey;
      int rem;  // radix_kth_pair starts with a block barrier: the candidates are in
      const uint32_t kth = radix_kth_pair<NT>([ck](int j) { return ck[j]; }, mine, kk, sm.sel, peer, &rem);
      // ordered take over this CTA's candidates, CTA 1's placed after CTA 0's:
      // each warp counts its segment's keys above and equal to the k-th ...
      const int tseg = cdiv(cdiv(mine, NW), 32) * 32;
      const int tb = min(warp * tseg, mine), te = min(tb + tseg, mine);
      int gt = 0, eq = 0;
      for (int base = tb; base < te; base += 32) {
        const int i = base + lane;
        const uint32_t u = (i < te) ? ck[i] : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, i < te && u > kth));
        eq += __popc(__ballot_sync(0xffffffffu, i < te && u == kth));
      }
      if (lane == 0) {
        sm.sel.wgt[warp] = gt;
        sm.sel.weq[warp] = eq;
      }
      __syncthreads();
      int gb = 0, eb = 0, cgt = 0, ceq = 0;
      for (int w = 0; w < NW; ++w) {
        if (w < warp) {
          gb += sm.sel.wgt[w];
          eb += sm.sel.weq[w];
        }
        cgt += sm.sel.wgt[w];
        ceq += sm.sel.weq[w];
      }
      // ... CTA 0 hands its totals to CTA 1 (the last access of the other CTA's
      // shared memory: after this barrier either CTA may finish)
      if (rank == 0 && tid == 0) {
        cluster_st(cluster_addr(&sm.peer_gt, peer), cgt);
        cluster_st(cluster_addr(&sm.peer_eq, peer), ceq);
      }
      cluster_barrier();
      if (rank == 1) {
        gb += sm.peer_gt;
        eb += sm.peer_eq;
      }
      // ... and writes, ascending, every score index above it plus the first
      // `rem` equal to it
      for (int base = tb; base < te; base += 32) {
        const int i = base + lane;
        const uint32_t u = (i < te) ? ck[i] : 0u;
        const bool isg = i < te && u > kth;
        const bool ise = i < te && u == kth;
        const unsigned bg = __ballot_sync(0xffffffffu, isg);
        const unsigned be = __ballot_sync(0xffffffffu, ise);
        const int G = gb + __popc(bg & lt), E = eb + __popc(be & lt);
        // the places are below kk by construction; the bound keeps a wrong
        // k-th key from writing past the row
        const int at = isg ? G + min(E, rem) : ((ise && E < rem) ? G + E : kk);
        if (at < kk) out[at] = sm.cidx[i];
        gb += __popc(bg);
        eb += __popc(be);
      }
      done = true;
    }
  }
  if (rank != 0) return;  // the rest is CTA 0's: no cluster barrier follows
  if (!done) topk_select_sorted<NT>(gkey, N, kk, out, sm.sel);
  for (int i = kk + tid; i < ld; i += NT) out[i] = -1;
}

}  // namespace mi
