// estimate.cuh - online estimation of vertical-slash indices.
//
// Method (MInference talk slides, boteman.cn, "Step 2: Online Estimation of
// Sparsity Indices"; README mirror, gittoolsai.com, "TL;DR"): the last 64
// queries of each head are scored against every key with a causal softmax;
// the probabilities are summed per key column (vertical score v) and per
// diagonal offset o = q - j (slash score s).
//
// Layout of the work: one CTA takes a pair of q-heads that share a KV head
// (128 query rows = 2 x 64, one UMMA M) and a chunk of keys (1024 in pass 1,
// 1024-4096 in pass 2), and runs
// S = Q K^T per 128-key tile on the tensor cores (TMEM accumulator), so each
// K tile is read once for both heads.  Eight warps do the arithmetic, two
// threads per row (64 keys of each tile each).
//   pass 1  per row: running max m and sum z = sum exp2(x - m) over the chunk
//   combine per row: merge the chunk partials (a warp per row) -> (m, 1/z)
//   pass 2  per 64-key half tile: four producer warps (a thread per row) write
//           a = exp2(x - m) / z into one of two shared-memory slots, skewed so
//           that every diagonal is a column; four consumer warps meanwhile sum
//           the other slot: column sums give v[j] for the half tile's keys,
//           sums down the skewed columns give s[o].
// A diagonal d (the key its row 63 meets) spans keys d-63..d, so it may start
// in the previous half tile: each consumer thread owns one diagonal position e
// and carries the partial sum of diagonal e + 64 to the next half tile, and
// each pass-2 CTA also scores the 64 keys before its chunk (a halo whose own
// outputs are discarded) so that every diagonal it writes is complete.  Every
// output element is written by exactly one thread with a fixed summation
// order: the scores are deterministic.
#pragma once

#include "common.cuh"
#include "pdl.cuh"
#include "ptx.cuh"

namespace mi {

struct EstArgs {
  int N, group, n_pairs, NC;
  int chunk2;    // pass-2 keys per CTA (a multiple of 128)
  float scale_log2;
  float* part;   // [n_heads, 64, NC, 2]  pass-1 partials (m, z)
  float* stats;  // [n_heads, 64, 2]      (m, 1/z)
  float* vsc;    // [n_heads, N]          vertical scores
  float* ssc;    // [n_heads, N]          slash scores, indexed by offset
  int* status;
  uint64_t wait_limit_ns;
  // nullptr: the query rows are the last 64 (p_i = N - 64 + i); otherwise the
  // rows end at *row_end (device int): p_i = R - 64 + i, R = min(max(*row_end, 64), N)
  const int* row_end;
  HeadList heads;
  int16_t pair_a[MI_MAX_HEADS];  // list slots; pair_b = -1: single head
  int16_t pair_b[MI_MAX_HEADS];
};

struct EstSmem {
  alignas(1024) uint8_t q[2][16384];
  alignas(1024) uint8_t k[2][2][16384];
  uint64_t q_full, k_full[2], k_empty[2], s_full[2], s_empty[2], mma_done;
  uint64_t sk_full[2], sk_empty[2];  // pass 2: the probability slots
  uint32_t tmem;
  int abort;
};
// Pass 2 keeps each half tile's probabilities in a skewed layout, per head of
// the pair 64 rows x 128 fp32: row i's key c (0..63) sits at column c + 63 - i,
// so that diagonal e (the diagonal that meets key j0 + e at row 63) is column e,
// and key column c runs along i -> c + 63 - i.  Positions outside a row's 64
// keys stay zero (written once).  Two slots: one is written while the other is
// summed.  Pass 1 uses the same space for the two column halves' (m, z).
// Pass 2 takes chunks of EstArgs::chunk2 keys, the largest of 4096, 2048 and 1024
// that still gives every SM a CTA (longer chunks make the halo tile a smaller
// share: 1/33 of a CTA's tiles at 4096 keys, 1/9 at 1024); pass 1 keeps 1024 (its
// partials are per 1024-key chunk).
inline int est_chunk2(int n_pairs, int N, int n_sms) {
  for (int c = 4096; c > 1024; c >>= 1)
    if (n_pairs * cdiv(N, c) >= n_sms) return c;
  return 1024;
}
constexpr int kSkPitch = 128;
constexpr int kSkHead = 64 * kSkPitch;
constexpr int kSkSlot = 2 * kSkHead;
constexpr int kEstThreads = 384;  // warp 0 MMA, warp 1 TMA, warps 4-11 the rows' arithmetic
constexpr int kEstMath = 256;     // threads of warps 4-11
constexpr int kEstHalf = 128;     // pass 2: producer threads (warps 4-7) = consumer threads (8-11)
constexpr size_t kEstSmem1 = sizeof(EstSmem) + 1024 + sizeof(float) * 2 * 128 * 2;
constexpr size_t kEstSmem2 = sizeof(EstSmem) + 1024 + sizeof(float) * 2 * kSkSlot;

template <int PASS>
__global__ void __launch_bounds__(kEstThreads, PASS == 1 ? 2 : 1)
est_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ EstArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  EstSmem& s = *reinterpret_cast<EstSmem*>(base);
  float* Sk = reinterpret_cast<float*>(base + sizeof(EstSmem));  // pass 2: [slot][head][64][kSkPitch]

  const int tid = threadIdx.x, warp = tid >> 5;
  const int pr = blockIdx.x, chunk = blockIdx.y;
  const int slot_a = a.pair_a[pr], slot_b = a.pair_b[pr];
  const int ha = a.heads.h[slot_a];
  const int hb = slot_b >= 0 ? a.heads.h[slot_b] : ha;
  const int g = ha / a.group;
  const int N = a.N;
  const int R = a.row_end ? min(max(__ldg(a.row_end), kLastQ), N) : N;  // one past the last query row
  const int CK = (PASS == 1) ? kChunkKeys : a.chunk2;  // keys of this CTA's chunk
  const int k_lo = chunk * CK - ((PASS == 2 && chunk > 0) ? kBN : 0);
  const int k_hi = min(N, (chunk + 1) * CK);
  const int T = cdiv(k_hi - k_lo, kBN);
  const bool has_halo = (PASS == 2 && chunk > 0);
  // the next kernel of the chain (combine after pass 1, top-k after pass 2) may
  // be scheduled now; it waits for this one to complete before reading its output
  pdl_trigger();

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.k_full[b], 1);
      mbar_init(&s.k_empty[b], 1);
      mbar_init(&s.s_full[b], 1);
      mbar_init(&s.s_empty[b], PASS == 1 ? kEstMath : kEstHalf);
    }
    mbar_init(&s.mma_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.sk_full[b], kEstHalf);
      mbar_init(&s.sk_empty[b], kEstHalf);
    }
    s.abort = 0;
    fence_mbar_init();
  }
  if (PASS == 2) {
    float4* z4 = reinterpret_cast<float4*>(Sk);
    for (int e = tid; e < 2 * kSkSlot / 4; e += kEstThreads) z4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (warp == 0) {
    tmem_alloc(&s.tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  volatile int* abort = &s.abort;
  const uint64_t lim = a.wait_limit_ns;

  if (warp == 0) {
    if (lane_id() == 0) {
      const uint32_t id = idesc_bf16(128, kBN, 0);
      bool ok = mbar_wait(&s.q_full, 0, abort, lim);
      for (int t = 0; t < T && ok; ++t) {
        const int b = t & 1;
        ok = mbar_wait(&s.k_full[b], (t >> 1) & 1, abort, lim);
        if (ok && t >= 2) ok = mbar_wait(&s.s_empty[b], ((t - 2) >> 1) & 1, abort, lim);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sdesc_sw128(smem_u32(s.q[kk >> 2]) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(s.k[b][kk >> 2]) + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + b * 128, ad, bd, id, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s.s_full[b]);
        umma_commit(&s.k_empty[b]);
      }
      umma_commit(&s.mma_done);
      mbar_wait_drain(&s.mma_done, 0, lim);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane_id() == 0) {
      mbar_arrive_expect_tx(&s.q_full, 4 * 8192);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(s.q[c], &map_q, &s.q_full, 64 * c, R - kLastQ, ha);
        tma_load_3d(s.q[c] + 8192, &map_q, &s.q_full, 64 * c, R - kLastQ, hb);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int b = t & 1;
        if (t >= 2 && !mbar_wait(&s.k_empty[b], ((t - 2) >> 1) & 1, abort, lim)) break;
        mbar_arrive_expect_tx(&s.k_full[b], 2 * 16384);
        tma_load_3d(s.k[b][0], &map_k, &s.k_full[b], 0, k_lo + t * kBN, g);
        tma_load_3d(s.k[b][1], &map_k, &s.k_full[b], 64, k_lo + t * kBN, g);
        issued = t + 1;
      }
      mbar_wait_drain(&s.q_full, 0, lim);
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait_drain(&s.k_full[t & 1], (t >> 1) & 1, lim);
    }
    __syncwarp();
  } else if (warp >= 4 && PASS == 1) {
    // two threads per row: warp w reads TMEM lanes 32 (w % 4) .. + 31 (the rows)
    // and the columns 64 ch .. 64 ch + 63 of each tile, ch = (w - 4) / 4
    const int row = ((warp & 3) << 5) | static_cast<int>(lane_id());  // rows 0-63 head a, 64-127 head b
    const int ch = (warp - 4) >> 2;
    const int hs = row >> 6, i = row & 63;
    const int slot = hs ? slot_b : slot_a;
    const int p_i = R - kLastQ + i;  // position of this query row
    const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 64 * ch;
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
    float m = -INFINITY, z = 0.f;
    for (int t = 0; t < T; ++t) {
      const int b = t & 1;
      // On a failed (timed-out) wait the loop still runs to the end with zeros, so
      // that the math warps keep meeting at the named barrier below.
      const bool ok = mbar_wait_warp(&s.s_full[b], (t >> 1) & 1, abort, lim);
      const int j0 = k_lo + t * kBN;
      // the thread's 64 columns in two halves of 32 (a running max and sum over
      // them), which keeps the registers within two CTAs per SM
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float x[32];
        if (ok) {
          tc_fence_after();
          tmem_ld32(taddr + b * 128 + 32 * hf, x);
          if (hf == 1) {
            tc_fence_before();
            mbar_arrive(&s.s_empty[b]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] = 0.f;
        }
        // keys j0 + 64 ch + 32 hf + c with c <= lim_c are causal; rows of an absent
        // second head are dropped
        const int lim_c = (slot >= 0) ? p_i - j0 - 64 * ch - 32 * hf : -1;
        if (lim_c < 31) {  // all 32 keys causal (every tile but the last ones): no per-key select
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] = (c <= lim_c) ? x[c] : -INFINITY;
        }
        // the scale is positive, so the maximum of the scaled scores is the scaled
        // maximum (rounding is monotone)
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = fmaxf(mx, x[c]);
        const float mn = fmaxf(m, mx * a.scale_log2);
        const float mb = (mn == -INFINITY) ? 0.f : mn;
        const float2 nmb2 = make_float2(-mb, -mb);
        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float2 y = fma2(make_float2(x[c], x[c + 1]), sc2, nmb2);
          acc2 = add2(acc2, make_float2(fast_exp2(y.x), fast_exp2(y.y)));
        }
        z = z * fast_exp2(m - mb) + (acc2.x + acc2.y);
        m = mn;
      }
    }
    // merge the two column halves of each row, in a fixed order
    float(*mz)[128][2] = reinterpret_cast<float(*)[128][2]>(Sk);
    mz[ch][row][0] = m;
    mz[ch][row][1] = z;
    named_bar_sync(1, kEstMath);
    if (ch == 0 && slot >= 0) {
      const float m1 = mz[1][row][0], z1 = mz[1][row][1];
      const float mn = fmaxf(m, m1);
      const float mb = (mn == -INFINITY) ? 0.f : mn;
      const float zz = z * fast_exp2(m - mb) + z1 * fast_exp2(m1 - mb);
      float* pp = a.part + (((size_t)slot * kLastQ + i) * a.NC + chunk) * 2;
      pp[0] = mn;
      pp[1] = zz;
    }
  } else if (warp >= 4) {
    const int mt = tid - 128;  // 0..255
    if (R < N) {
      // offsets R .. N-1 meet no query row: zero, this chunk's share of them
      for (int o = R + chunk * CK + mt; o < min(N, R + (chunk + 1) * CK); o += kEstMath) {
        a.ssc[(size_t)slot_a * N + o] = 0.f;
        if (slot_b >= 0) a.ssc[(size_t)slot_b * N + o] = 0.f;
      }
    }
    // the half tiles of this CTA: u = 2 t + h, from h = 1 of tile 0 when that tile
    // is the halo (only its second half reaches into the chunk's diagonals)
    const int u0 = has_halo ? 1 : 0, U = 2 * T;
    if (warp < 8) {
      // producers: thread = row (TMEM lane), 64 keys of each half tile
      const int row = ((warp & 3) << 5) | static_cast<int>(lane_id());
      const int hs = row >> 6, i = row & 63;
      const int slot = hs ? slot_b : slot_a;
      const int p_i = R - kLastQ + i;
      const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      // without a second head: m = 0, 1/z = 0 gives zeros (no inf - inf).  The
      // row statistics come from the combine kernel: wait for it (the MMA and
      // load warps, which touch only Q, K and this CTA's memory, run ahead)
      float m = 0.f, invz = 0.f;
      pdl_wait();
      if (slot >= 0) {
        m = a.stats[((size_t)slot * kLastQ + i) * 2 + 0];
        invz = a.stats[((size_t)slot * kLastQ + i) * 2 + 1];
      }
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
      const float2 nm2 = make_float2(-m, -m), iz2 = make_float2(invz, invz);
      float* sk_row = Sk + hs * kSkHead + i * (kSkPitch - 1) + 63;  // + c: key c of the half tile
      for (int u = u0; u < U; ++u) {
        const int t = u >> 1, h = u & 1, b = t & 1, sl = (u - u0) & 1;
        if ((h == 0 || u == u0) && !mbar_wait_warp(&s.s_full[b], (t >> 1) & 1, abort, lim)) break;
        float x[64];
        tc_fence_after();
        tmem_ld64(taddr + b * 128 + 64 * h, x);
        if (h == 1) {  // the TMEM buffer is free for the MMA of tile t + 2
          tc_fence_before();
          mbar_arrive(&s.s_empty[b]);
        }
        if (u - u0 >= 2 && !mbar_wait_warp(&s.sk_empty[sl], ((u - u0 - 2) >> 1) & 1, abort, lim)) break;
        const int lim_c = (slot >= 0) ? p_i - (k_lo + t * kBN + 64 * h) : -1;
        if (lim_c < 63) {  // all 64 keys causal (every half tile but the last ones): no per-key select
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = (c <= lim_c) ? x[c] : -INFINITY;
        }
        float* dst = sk_row + sl * kSkSlot;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 y = fma2(make_float2(x[c], x[c + 1]), sc2, nm2);
          const float2 pv = mul2(make_float2(fast_exp2(y.x), fast_exp2(y.y)), iz2);
          dst[c] = pv.x;
          dst[c + 1] = pv.y;
        }
        mbar_arrive(&s.sk_full[sl]);
      }
    } else {
      // consumers: thread = (head hh, position e < 64) of the half tile; sums
      // column e (diagonal j0 + e, completed with the carry), column e + 64 (the
      // part of diagonal j0 + 64 + e in this half tile: the next carry) and the
      // skewed key column e
      const int ct = tid - 256;  // 0..127
      const int hh = ct >> 6, e = ct & 63;
      const int sl_h = hh ? slot_b : slot_a;
      float carry = 0.f;
      for (int u = u0; u < U; ++u) {
        const int t = u >> 1, h = u & 1, sl = (u - u0) & 1;
        if (!mbar_wait_warp(&s.sk_full[sl], ((u - u0) >> 1) & 1, abort, lim)) break;
        const float* src = Sk + sl * kSkSlot + hh * kSkHead;
        float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
        // row r of skewed column e holds key r + e - 63 of the half tile, and of
        // column e + 64 key r + e + 1: only rows with that key in 0..63 hold a
        // probability, the rest are zeros.  The warp's positions e are 0-31 or
        // 32-63, so the rows 32-63 (lower half) and 0-62 / 0-30 cover it: the
        // skipped terms are zeros, and the sums keep their order (bit-identical)
        const bool e_lo = e < 32;  // warp-uniform
#pragma unroll
        for (int r = 0; r < 64; ++r) {
          if (r >= 32 || !e_lo) lo[r & 3] += src[r * kSkPitch + e];
          if (r <= (e_lo ? 62 : 30)) hi[r & 3] += src[r * kSkPitch + e + 64];
          cs[r & 3] += src[r * (kSkPitch - 1) + e + 63];
        }
        mbar_arrive(&s.sk_empty[sl]);
        const float dlo = (lo[0] + lo[1]) + (lo[2] + lo[3]);
        const float dhi = (hi[0] + hi[1]) + (hi[2] + hi[3]);
        const float col = (cs[0] + cs[1]) + (cs[2] + cs[3]);
        const int j0 = k_lo + t * kBN + 64 * h;
        if (!(has_halo && t == 0) && sl_h >= 0) {
          const int d = j0 + e;  // offset R - 1 - d (a key past R - 1 has no row: o < 0)
          if (d < R) a.ssc[(size_t)sl_h * N + (R - 1 - d)] = dlo + carry;
          if (d < N) a.vsc[(size_t)sl_h * N + d] = col;
        }
        carry = dhi;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s.abort && tid == 0) set_status(a.status, MI_ERR_TIMEOUT);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Merge the per-chunk (m, z) partials of every estimation row: one warp per row,
// lane l takes chunks l, l + 32, ... (coalesced), then the maximum and the
// rescaled sum are reduced over the warp in a fixed order.
// Launched as the dependent of pass 1 and followed by pass 2 (pdl.cuh).
__global__ void est_combine(const float* part, float* stats, int NC, int n_rows) {
  pdl_trigger();
  pdl_wait();  // the partials of pass 1
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  const float2* pp = reinterpret_cast<const float2*>(part + (size_t)row * NC * 2);
  float m = -INFINITY;
  for (int c = lane; c < NC; c += 32) m = fmaxf(m, pp[c].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
  for (int c = lane; c < NC; c += 32) {
    const float2 t = pp[c];
    if (t.x != -INFINITY) z += t.y * fast_exp2(t.x - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) {
    stats[(size_t)row * 2 + 0] = m;
    stats[(size_t)row * 2 + 1] = 1.f / z;
  }
}

}  // namespace mi
