// attention.cuh - the tcgen05 sparse/dense causal attention engine.
//
// One CTA computes 128 query rows (one row block r) of one head.  Its key
// range is a list of 128-key tiles chosen by the head's pattern:
//   - contiguous tiles, TMA-loaded from K/V ([Hkv, N, 128] bf16, 128-byte
//     swizzle, 64-key boxes), masked element-wise by the pattern's rule; for
//     exact vertical-slash heads these are 128-key windows at any key offset
//     (the greedy cover of the selected diagonals built by vs_index_kernel);
//   - for block-sparse heads and block-expanded vertical-slash heads, tiles
//     made of two 64-key blocks from anywhere below the diagonal (two boxes
//     each): the two 64-row halves' selections, or the blocks the row block's
//     kept 64-block distances reach, paired two per tile;
//   - for vertical-slash heads, "gathered" column tiles: the head's selected
//     key columns are copied side by side once per call (their K and V rows,
//     vs_colgather_kernel), and a tile is 128 consecutive entries of that
//     compacted list, TMA-loaded like a contiguous tile and masked to the
//     columns no contiguous tile of the row block covers (the
//     permutation-invariant gathering idea of PIT, which the MInference pages
//     name as the basis of their kernels: README mirror, gittoolsai.com,
//     "TL;DR" and the PIT note; talk slides, boteman.cn, "Dynamic Sparse
//     Attention Calculation with PIT, FlashAttention").
//
// Warp roles (192 threads, two CTAs per SM, up to 168 registers per thread):
//   warps 0-3   softmax: thread t owns query row t (TMEM lane t)
//   warp 4      TMEM allocation and the single-thread tcgen05.mma issuer
//   warp 5      Q (once), then K and V tiles (TMA boxes of 64 keys);
//               for vertical-slash heads also the rows' keep-masks
//
// Tensor memory (256 columns): S = Q K^T (fp32, columns 0-127) and O (fp32,
// columns 128-255).  Per tile: the MMA warp issues S = Q K_i^T; the softmax
// warps read their S row into registers once (mask, row maximum, exp2, pack)
// and write P_i = exp2(x - m) as bf16 pairs over the S columns they have
// consumed; the MMA warp issues O += P_i V_i with P read from tensor memory,
// chunk of keys by chunk as soon as each chunk of P is stored (unless O is
// being rescaled in this tile).  The running maximum moves (and O is rescaled
// in tensor memory) only when a tile's maximum exceeds it by more than 8 (log2
// units), so P stays below 2^8.  Shared memory holds one Q tile and one K and
// one V stage (about 112 KB), so two CTAs share an SM and one CTA's softmax
// overlaps the other's MMAs.
// Every mbarrier wait is bounded; on a timeout the CTA stops issuing work,
// waits for what it already issued, frees TMEM and records MI_ERR_TIMEOUT.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace mi {

enum Pattern : int {
  kPatDense = 0, kPatVS = 1, kPatBlock = 2, kPatAShape = 3, kPatVSExp = 4, kPatRows = 5, kPatCross = 6
};
// kPatCross: the cross-modality pairs of 2D-boundary heads (two modalities):
// row q keeps key j <= q of the other modality; only the key tiles holding the
// other modality of some row of the block are visited.
// kPatRows: the horizontal lines of grid heads (MMInference, "Grid Head in
// Multi-Modality"): the rows q = phi (mod sigma) gathered 128 at a time (CTA
// "row block" r holds rows phi + sigma (128 r + i)), each attending densely to
// its causal prefix: the permuted form of the grid's horizontal lines.
// kPatVSExp is the vertical-slash engine with block-expanded slashes: a
// compile-time variant of kPatVS (its heads use the kPatVS slots and arrays).
__host__ __device__ constexpr bool is_vs(int p) { return p == kPatVS || p == kPatVSExp; }

struct AttnArgs {
  const __nv_bfloat16* q;  // grid rows: the query rows are gathered from here
  int N;
  int ld;            // rows between consecutive heads of q, k, v, out and lse (N, or a
                     // packed batch's token count)
  int group;         // Hq / Hkv
  float scale_log2;  // log2(e) / sqrt(d)
  __nv_bfloat16* out;
  float* lse;
  int* status;
  uint64_t wait_limit_ns;
  int skip_q_load;  // fault injection (tests): Q is never loaded, waits expire
  // vertical-slash index structures (per listed head)
  const uint32_t* offbits;  // [n_heads, Nw]   bit o: offset o selected (block-expanded
                            //                 mode: bit e: 64-block distance e kept)
  const uint32_t* colbits;  // [n_heads, Nw]   bit j: column j selected
  // exact slashes: key windows p (row block r reads keys 128 r - p .. + 127 for
  // every p < 128 r, besides tile 0); block-expanded slashes need offbits alone
  const uint32_t* dbits;    // [n_heads, Dw]   bit x + 128 when a window covers key
                            //                 distance x = 128 r - j
  const uint32_t* dfull;    // [n_heads, NTw]  bit i when window i is kept whole
  const int* dlist;         // [n_heads, NT]   the windows, ascending
  const int* dcount;        // [n_heads]
  const int* clist;         // [n_heads, MI_MAX_KV]  the selected columns, ascending
  const int* ccount;        // [n_heads]
  int expand;               // block-expanded slashes: the host launches the kPatVSExp engine
  int Nw, NT, NTw, Dw;
  // block-sparse
  const int* blk_idx;  // [n_heads, ceil(N/64), topk]
  int topk;
  // A-shape
  int n_init, window;
  // grid rows (kPatRows): (sigma, phi) per listed head; a head whose sigma is below
  // grid_sigma_min (rejected by the lattice step) has no rows here either
  const int* grid;
  int grid_sigma_min;
  // Q-boundary passes: write only the rows of modality row_mod, skip the row
  // blocks without it (modality == nullptr: every row)
  const int32_t* modality;  // [N]
  const uint32_t* blk_mods;  // [ceil(N / 128)] bit m: modality m present
  int row_mod;
  // 2D-boundary cross pass (kPatCross): bit j of modbits = token j is of
  // modality 1; mods128[t] bit m = 128-token block t holds modality m
  const uint32_t* modbits;
  const uint32_t* mods128;
  int ash_n;              // layer launches: A-shape heads with their own sizes in ash_pairs
  int ash_pairs[2 * MI_MAX_HEADS];  // [A-shape slot][2] = n_init, window
  HeadList heads;
  // layer launches: the listed heads are ordered dense, vertical-slash,
  // block-sparse, A-shape; layer_base[p] is the first listed head of pattern p
  // (layer_base[4] = heads.n), so a head's slot in its pattern's arrays is its
  // listed index minus its pattern's base
  int layer_base[5];
};

struct AttnSmem {
  alignas(1024) uint8_t q[2][16384];
  alignas(1024) uint8_t k[2][16384];
  alignas(1024) uint8_t v[2][16384];
  // VS: [0, 16) the column chunks with a residual column, [16, 80) the residual
  // bits of the chunks' entries; block: per tile (block A << 4) | sub-block mask, block B
  int list[MI_MAX_KV];
  int scan[192];
  uint32_t dfull[512];  // VS: the head's whole-window bits (N <= 2^21)
  // VS: keep-masks of two tiles in flight (row i: bit c of word c / 32 keeps
  // key c of the tile), built by the loader warp; tile t uses stage t & 1
  uint32_t vmask[2][kBM][4];
  uint64_t q_full, k_full, k_empty, v_full, v_empty, s_full, p_full, pv_done, mma_done;
  // P of the first (i + 1) / NQ of the keys stored (128 softmax threads arrive);
  // the last chunk is p_full.  NQ = kPChunks<PAT>.
  uint64_t p_part[3];
  uint64_t m_full[2];  // VS: mask stage written (the 32 loader lanes arrive)
  uint32_t tmem;
  int abort;
  int n_list;    // entries in list
  int col_lo;    // VS: first entry of the compacted column list past tile 0
  int n_tiles;   // tiles this CTA processes
  int n_contig;  // leading contiguous tiles (VS)
  int has_t0;    // VS (exact): tile 0 is prepended
  int d_cnt;     // VS: windows p < 128 r; block-expanded: needed 64-key blocks
  int ash_init;  // A-shape: sink tokens of this head
  int ash_window;  // A-shape: window of this head
  int g_sigma, g_phi, g_lines;  // grid rows: stride, phase, rows on the lattice
};

constexpr int kAttnThreads = 192;
constexpr size_t kAttnSmemBytes = sizeof(AttnSmem) + 1024;
static_assert(sizeof(AttnArgs) + 5 * sizeof(CUtensorMap) <= 4096, "attention kernel parameters exceed 4 KB");
// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(2 * (kAttnSmemBytes + 1024) <= 228 * 1024, "two attention CTAs must fit on one SM");
constexpr uint32_t kTmemCols = 256;  // S (and P over it) at 0, O at 128
constexpr uint32_t kTmemO = 128;
// P is stored in NQ chunks of keys and P.V of a chunk starts as soon as it is
// stored: four for the sparse patterns (measured: vertical-slash 5 %, A-shape
// 5 %, block-sparse 2 % faster than two; eight were slower), two for dense
// (four cost it 2.6 %)
template <int PAT>
constexpr int kPChunks = PAT == kPatDense ? 2 : 4;

// ------------------------------------------------------------ tile list ----

struct TileRef {
  int kind;  // 0 contiguous, 1 gathered
  int t;     // contiguous: key tile index (exact vertical-slash windows: their
             // first key / 128); gathered: chunk of the residual list;
             // block pattern: the 64-key block in keys 0-63 of the tile
  int sub;   // block pattern: 4-bit mask (bit = rowhalf*2 + keyhalf)
  int t2;    // block pattern: the 64-key block in keys 64-127 of the tile;
             // exact vertical-slash windows: the window's list index (-1: tile 0)
  int j0;    // vertical-slash contiguous tiles: the first key
};

// Block-expanded slashes: row block r needs key block kb = 2 r + 1 - x for the set
// bits x of a bitmap over x in [0, 2 r + 1] (a kept 64-block distance x or x - 1,
// and x = 2 r + 1: block 0), held in list[kVsxBits ..]; the tiles pair them in
// order of x.  The loader walks the bitmap once with this cursor (the tiles are
// taken in order), so each tile costs a few bit operations.
constexpr int kVsxBits = 128;  // up to 1024 words (2 r + 2 <= 32768)
struct VsxCursor {
  int w;       // current word
  uint32_t m;  // its bits not yet taken
  __device__ __forceinline__ int next(const AttnSmem& s) {  // the next set bit (one exists)
    const uint32_t* fb = reinterpret_cast<const uint32_t*>(&s.list[kVsxBits]);
    while (m == 0u && w < 1023) m = fb[++w];  // (bounded by the bitmap's 1024 words)
    const int x = 32 * w + __ffs(m) - 1;
    m &= m - 1;
    return x;
  }
  __device__ __forceinline__ TileRef tile(const AttnSmem& s, int r, int i) {  // tile i < n_contig
    TileRef ref{0, 0, 0xF, -1, 0};
    ref.t = 2 * r + 1 - next(s);
    if (2 * i + 1 < s.d_cnt) ref.t2 = 2 * r + 1 - next(s);
    ref.j0 = ref.t * kBlk;
    return ref;
  }
};

template <int PAT>
__device__ __forceinline__ TileRef tile_at(const AttnSmem& s, const AttnArgs& a, int n, int r,
                                           int i) {
  TileRef ref{0, 0, 0xF, 0};
  if (PAT == kPatDense || PAT == kPatRows) {
    ref.t = i;
  } else if (PAT == kPatVSExp) {  // the block pairs come from a VsxCursor (loader)
    ref.kind = 1;
    ref.t = s.list[i - s.n_contig];  // chunk of the compacted column list
  } else if (is_vs(PAT)) {
    if (i < s.n_contig) {
      if (s.has_t0 && i == 0) {
        ref.t = 0;
        ref.t2 = -1;
        ref.j0 = 0;
      } else {  // window p: keys 128 r - p ..
        const int idx = s.d_cnt - 1 - (i - s.has_t0);  // keys ascending
        const int p = ldg_ahead(a.dlist + (size_t)n * a.NT + idx);
        ref.j0 = r * kBN - p;
        ref.t = ref.j0 >> 7;
        ref.t2 = idx;
      }
    } else {
      ref.kind = 1;
      ref.t = s.list[i - s.n_contig];  // chunk of the compacted column list
    }
  } else if (PAT == kPatCross) {
    // intervals of consecutive tiles: list[2 k] first tile, list[2 k + 1] count,
    // list[128 + k] tiles before interval k (binary search for the one holding i)
    int lo = 0, hi = s.n_list - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.list[128 + mid] <= i) lo = mid; else hi = mid - 1;
    }
    ref.t = s.list[2 * lo] + (i - s.list[128 + lo]);
  } else if (PAT == kPatBlock) {
    const int e = s.list[2 * i];
    ref.t = e >> 4;
    ref.sub = e & 0xF;
    ref.t2 = s.list[2 * i + 1];
  } else {  // A-shape: sink tiles then the window tiles
    const int t_lo = max(0, r * kBM - s.ash_window + 1) / kBN;
    const int n_sink = min(cdiv(s.ash_init, kBN), t_lo);
    ref.t = (i < n_sink) ? i : t_lo + (i - n_sink);
  }
  return ref;
}

// Bits [lo, hi) of a 32-bit word whose bit 0 is position `base`.
__device__ __forceinline__ uint32_t range_bits(int base, int lo, int hi) {
  lo = max(lo - base, 0);
  hi = min(hi - base, 32);
  if (hi <= lo) return 0u;
  const uint32_t up = (hi >= 32) ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  return up & ~((1u << lo) - 1u);
}

// The words a row's keep-mask is built from.  Vertical-slash rows get theirs
// from the loader warp's four-row fetch (vs_fetch4 / vs_row_raw); the other
// patterns' masks depend on the tile reference alone.
struct MaskRaw {
  TileRef ref;
  bool whole;        // VS: the tile is kept whole (no mask words needed)
  int base;          // VS: first offset bit of the window (q - j0 - 127)
  uint32_t off[5];   // VS: offset-bitmap words covering [base, base + 128)
  uint32_t col[4];   // VS: column-bitmap words of the tile's keys
};

// Dense, block-sparse and A-shape tiles: the reference is all a mask needs.
template <int PAT>
__device__ __forceinline__ MaskRaw mask_fetch(const AttnArgs& a, const TileRef& ref) {
  static_assert(!is_vs(PAT), "vertical-slash masks are built by the loader warp");
  MaskRaw m;
  m.ref = ref;
  m.base = 0;
  m.whole = false;
  if (PAT == kPatCross) {  // the modality bits of the tile's keys (read a tile ahead)
#pragma unroll
    for (int w = 0; w < 4; ++w) m.col[w] = ldg_ahead(a.modbits + ref.t * 4 + w);
  }
  return m;
}

// A loader lane's raw words for the four rows q0 + 32 i (i = 0..3) of a
// vertical-slash tile.  Exact slashes: the rows' offset windows start 32 bits
// apart, so eight offset-bitmap words cover all four (row i uses off[i..i+4]).
// Block-expanded slashes: the words depend on the tile alone.
struct VsRaw4 {
  TileRef ref;
  bool whole;
  int base;         // exact: first offset bit of row q0's window; expanded: bit h + 2 k when
                    // 64-row half h keeps block k (0: t, 1: t2)
  uint32_t off[8];
  uint32_t col[4];
};

template <int PAT>
__device__ __forceinline__ VsRaw4 vs_fetch4(const AttnSmem& s, const AttnArgs& a, int n, int r,
                                            const TileRef& ref, int q0) {
  VsRaw4 m;
  m.ref = ref;
  m.base = 0;
  m.whole = false;
  const uint32_t* off = a.offbits + (size_t)n * a.Nw;
  const uint32_t* col = a.colbits + (size_t)n * a.Nw;
  if (PAT == kPatVSExp) {
    if (ref.kind != 0) return m;
    // the tile is 64-key blocks A (keys 0-63) and B (keys 64-127, none when
    // t2 < 0); bit h + 2 k of base: 64-row half h keeps block k (0: A, 1: B),
    // i.e. block 0, or 64-block distance 2 r + h - block kept
    const int blk[2] = {ref.t, ref.t2};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = 2 * r + h - blk[k];
        const uint32_t w = ldg_ahead(off + min(max(e, 0) >> 5, a.Nw - 1));
        const bool kept = blk[k] == 0 || (blk[k] > 0 && e >= 0 && ((w >> (e & 31)) & 1u));
        if (blk[k] >= 0 && kept) m.base |= 1 << (h + 2 * k);
      }
#pragma unroll
      for (int w = 0; w < 2; ++w)
        m.col[2 * k + w] = (blk[k] >= 0) ? ldg_ahead(col + min(2 * blk[k] + w, a.Nw - 1)) : 0u;
    }
    // kept whole: both blocks, both halves, neither a causal block of the row block
    m.whole = m.base == 0xF && ref.t < 2 * r && ref.t2 < 2 * r;
    return m;
  }
  if (ref.kind == 0) {  // a window whose keys all lie past tile 0
    const int i = ref.t2;
    m.whole = i >= 0 && ref.j0 >= kBN && ((s.dfull[i >> 5] >> (i & 31)) & 1u);
  }
  if (ref.kind != 0 || m.whole) return m;
  const int j0 = ref.j0;
  {
    m.base = q0 - j0 - 127;
    const int w0 = m.base >> 5;  // floor; >= -4
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // the words of rows q0 .. q0 + 96; the bits the rows need are below 128 r + 127
      // (< 32 Nw), a word past the bitmap only rounds out the last one
      const int wi = w0 + i;
      m.off[i] = ldg_ahead(off + min(max(wi, 0), a.Nw - 1));
      if (wi < 0 || wi >= a.Nw) m.off[i] = 0u;
    }
  }
  // the column bits of keys j0 .. j0 + 127: five words shifted by j0 % 32 (a window
  // may start anywhere; the fifth word is past the bitmap only when j0 % 32 = 0)
  const int cw = j0 >> 5, csh = j0 & 31;
  uint32_t c5[5];
#pragma unroll
  for (int w = 0; w < 5; ++w) c5[w] = ldg_ahead(col + min(cw + w, a.Nw - 1));
#pragma unroll
  for (int w = 0; w < 4; ++w) m.col[w] = __funnelshift_r(c5[w], c5[w + 1], csh);
  return m;
}

// The raw words of row q0 + 32 i out of a lane's four-row fetch.
__device__ __forceinline__ MaskRaw vs_row_raw(const VsRaw4& m, int i, bool expanded) {
  MaskRaw r;
  r.ref = m.ref;
  r.whole = m.whole;
  r.base = expanded ? m.base : m.base + 32 * i;
#pragma unroll
  for (int k = 0; k < 5; ++k) r.off[k] = expanded ? m.off[k] : m.off[i + k];
#pragma unroll
  for (int w = 0; w < 4; ++w) r.col[w] = m.col[w];
  return r;
}

// Keep-mask of query row q over the 128 keys of tile m.ref (bit c of out[c/32]).
template <int PAT>
__device__ __forceinline__ void mask_finish(const AttnSmem& s, const AttnArgs& a, int r,
                                            const MaskRaw& m, int q, uint32_t out[4]) {
  const TileRef& ref = m.ref;
  const int j0 = is_vs(PAT) ? ref.j0 : ref.t * kBN;
  if (PAT == kPatCross) {  // keys of the other modality, j <= q
    const uint32_t rowm = (q < a.N) ? ((__ldg(a.modbits + (q >> 5)) >> (q & 31)) & 1u) : 0u;
#pragma unroll
    for (int w = 0; w < 4; ++w)
      out[w] = (q < a.N) ? ((rowm ? ~m.col[w] : m.col[w]) & range_bits(j0 + 32 * w, 0, q + 1)) : 0u;
    return;
  }
  if (PAT == kPatRows) {  // q is this row's position: keys j <= q
#pragma unroll
    for (int w = 0; w < 4; ++w) out[w] = range_bits(j0 + 32 * w, 0, q + 1);
    return;
  }
  if (PAT == kPatDense) {
#pragma unroll
    for (int w = 0; w < 4; ++w) out[w] = 0xFFFFFFFFu;
  } else if (is_vs(PAT)) {
    if (m.whole) {
#pragma unroll
      for (int w = 0; w < 4; ++w) out[w] = 0xFFFFFFFFu;
      return;  // never the diagonal tile (distance > 0)
    }
    // offsets q - j0 - c for c = 0..127 are the 128 bits starting at base, reversed
    const int sh = m.base & 31;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int k = 3 - w;
      const uint32_t win = __funnelshift_r(m.off[k], m.off[k + 1], sh);
      out[w] = __brev(win) | m.col[w];
    }
    if (j0 == 0) {  // the first 64 keys
      out[0] = 0xFFFFFFFFu;
      out[1] = 0xFFFFFFFFu;
    } else if (j0 < kBN) {  // a window reaching into tile 0 leaves those keys to it
#pragma unroll
      for (int w = 0; w < 4; ++w) out[w] &= range_bits(j0 + 32 * w, kBN, 1 << 30);
    }
    if (ref.t == r) {  // the query's own 64-block
      const int lb = (q >> 6) << 6;
#pragma unroll
      for (int w = 0; w < 4; ++w) out[w] |= range_bits(j0 + 32 * w, lb, lb + kBlk);
    }
  } else if (PAT == kPatBlock) {
    // keys 0-63 are block ref.t, keys 64-127 block ref.t2; a row keeps a block
    // its half selected, causally inside its own block
    const int half = (q >> 6) & 1, own = q >> 6;
    const uint32_t lo = ((ref.sub >> (half * 2)) & 1) ? 0xFFFFFFFFu : 0u;
    const uint32_t hi = ((ref.sub >> (half * 2 + 1)) & 1) ? 0xFFFFFFFFu : 0u;
    out[0] = lo;
    out[1] = lo;
    out[2] = hi;
    out[3] = hi;
    if (ref.t == own) {
      out[0] &= range_bits(ref.t * kBlk, 0, q + 1);
      out[1] &= range_bits(ref.t * kBlk + 32, 0, q + 1);
    }
    if (ref.t2 == own) {
      out[2] &= range_bits(ref.t2 * kBlk, 0, q + 1);
      out[3] &= range_bits(ref.t2 * kBlk + 32, 0, q + 1);
    }
    return;
  } else {  // A-shape
#pragma unroll
    for (int w = 0; w < 4; ++w)
      out[w] = range_bits(j0 + 32 * w, 0, s.ash_init) |
               range_bits(j0 + 32 * w, q - s.ash_window + 1, q + 1);
  }
  if (ref.t == r) {  // the diagonal tile: causal
#pragma unroll
    for (int w = 0; w < 4; ++w) out[w] &= range_bits(j0 + 32 * w, 0, q + 1);
  }
}

// Keep-masks of a loader lane's four rows q0 + 32 i of a vertical-slash tile.
// Off the diagonal tile the rows share their words: with exact slashes row i's
// word w is the reversed offset window E[i + 3 - w] (windows 32 bits apart), with
// block-expanded slashes rows 0-1 and 2-3 fall in the same 64-row half.  Whole,
// gathered and diagonal tiles take the per-row path.
template <int PAT>
__device__ __forceinline__ void vs_masks4(const AttnSmem& s, const AttnArgs& a, int r, const VsRaw4& m,
                                          int q0, uint32_t out[4][4]) {
  const TileRef& ref = m.ref;
  if (ref.kind == 1) {  // a column tile: the same residual bits for every row
    const uint4 w = *reinterpret_cast<const uint4*>(&s.list[16 + 4 * ref.t]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[i][0] = w.x;
      out[i][1] = w.y;
      out[i][2] = w.z;
      out[i][3] = w.w;
    }
    return;
  }
  if (PAT == kPatVSExp) {
    // row i (q0 + 32 i) lies in 64-row half i / 2; a block of the row block's own
    // two (>= 2 r) is causal
    const int A = ref.t, Bb = ref.t2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int h = i >> 1, q = q0 + 32 * i;
      const uint32_t lo = (m.whole || ((m.base >> h) & 1)) ? 0xFFFFFFFFu : 0u;
      const uint32_t hi = (m.whole || ((m.base >> (2 + h)) & 1)) ? 0xFFFFFFFFu : 0u;
      out[i][0] = lo | m.col[0];
      out[i][1] = lo | m.col[1];
      out[i][2] = (Bb >= 0) ? (hi | m.col[2]) : 0u;
      out[i][3] = (Bb >= 0) ? (hi | m.col[3]) : 0u;
      if (A >= 2 * r) {
        out[i][0] &= range_bits(A * kBlk, 0, q + 1);
        out[i][1] &= range_bits(A * kBlk + 32, 0, q + 1);
      }
      if (Bb >= 2 * r) {
        out[i][2] &= range_bits(Bb * kBlk, 0, q + 1);
        out[i][3] &= range_bits(Bb * kBlk + 32, 0, q + 1);
      }
    }
    return;
  }
  if (ref.kind == 0 && !m.whole && ref.t != r) {
    {
      const int sh = m.base & 31;
      uint32_t e[7];
#pragma unroll
      for (int k = 0; k < 7; ++k) e[k] = __brev(__funnelshift_r(m.off[k], m.off[k + 1], sh));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int w = 0; w < 4; ++w) out[i][w] = e[i + 3 - w] | m.col[w];
      }
      if (ref.j0 > 0 && ref.j0 < kBN) {  // a window reaching into tile 0 leaves those keys to it
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t keep = range_bits(ref.j0 + 32 * w, kBN, 1 << 30);
#pragma unroll
          for (int i = 0; i < 4; ++i) out[i][w] &= keep;
        }
      }
    }
    if (ref.j0 == 0) {  // the first 64 keys
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        out[i][0] = 0xFFFFFFFFu;
        out[i][1] = 0xFFFFFFFFu;
      }
    }
    return;
  }
  if constexpr (PAT != kPatVSExp) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mask_finish<PAT>(s, a, r, vs_row_raw(m, i, false), q0 + 32 * i, out[i]);
  }
}

// ------------------------------------------------------------- prologue ----

// Block-wide exclusive scan of one int per thread (192 threads); returns the
// exclusive prefix and writes the total to *total.
__device__ __forceinline__ int block_excl_scan(int x, int* scratch, int* total) {
  const int tid = threadIdx.x;
  scratch[tid] = x;
  __syncthreads();
  for (int off = 1; off < 192; off <<= 1) {
    const int y = (tid >= off) ? scratch[tid - off] : 0;
    __syncthreads();
    scratch[tid] += y;
    __syncthreads();
  }
  const int incl = scratch[tid];
  *total = scratch[191];
  __syncthreads();
  return incl - x;
}

// A vertical column that no contiguous tile of row block r covers.
// db: exact slashes the windows' coverage bits; block-expanded the kept 64-block
// distances.
template <int PAT>
__device__ __forceinline__ bool residual_column(int j, int N, int r, const uint32_t* db) {
  if (PAT == kPatVSExp) {  // past block 0, before the row block, in a block it does not need
    if (j < kBlk || j >= N || j >= r * kBN) return false;
    const int e = 2 * r - (j >> 6);  // >= 1; the block is needed for distance e or e + 1
    const uint32_t w0 = __ldg(db + (e >> 5)), w1 = __ldg(db + ((e + 1) >> 5));
    return !(((w0 >> (e & 31)) & 1u) || ((w1 >> ((e + 1) & 31)) & 1u));
  }
  const int t = j >> 7;
  if (j < 0 || j >= N || t < 1 || t >= r) return false;
  // no window covers key distance x = 128 r - j (bit x + 128)
  const int x = r * kBN - j + kBN;
  return !((__ldg(db + (x >> 5)) >> (x & 31)) & 1u);
}

template <int PAT>
__device__ __forceinline__ void attn_prologue(AttnSmem& s, const AttnArgs& a, int n, int r) {
  const int tid = threadIdx.x;
  if (PAT == kPatDense) {
    if (tid == 0) s.n_tiles = r + 1;
  } else if (PAT == kPatCross) {
    // key tiles t <= r holding the other modality of some row of the block:
    // (mods128[t] | mods128[r]) == both modalities; as intervals of consecutive
    // tiles (each holds a run of a modality, so there are at most MI_MAX_RUNS)
    const uint32_t mr = __ldg(a.mods128 + r);
    auto need = [&](int t) { return t >= 0 && t <= r && ((__ldg(a.mods128 + t) | mr) == 3u); };
    const int per = cdiv(r + 1, kAttnThreads);
    const int t0 = min(tid * per, r + 1), t1 = min(t0 + per, r + 1);
    int ns = 0;
    for (int t = t0; t < t1; ++t) ns += (need(t) && !need(t - 1)) ? 1 : 0;
    int total;
    int pos = block_excl_scan(ns, s.scan, &total);
    for (int t = t0; t < t1; ++t) {
      if (!(need(t) && !need(t - 1)) || pos >= 64) continue;
      int e = t;
      while (need(e + 1)) ++e;
      s.list[2 * pos] = t;
      s.list[2 * pos + 1] = e - t + 1;
      ++pos;
    }
    __syncthreads();
    if (tid == 0) {
      const int ni = min(total, 64);
      int acc = 0;
      for (int k = 0; k < ni; ++k) {
        s.list[128 + k] = acc;
        acc += s.list[2 * k + 1];
      }
      s.n_list = ni;
      s.n_tiles = acc;
    }
  } else if (PAT == kPatRows) {
    if (tid == 0) {  // key tiles up to the block's last row
      const int last = s.g_phi + s.g_sigma * min(r * kBM + kBM - 1, s.g_lines - 1);
      s.n_tiles = last / kBN + 1;
    }
  } else if (PAT == kPatAShape) {
    if (tid == 0) {
      const int t_lo = max(0, r * kBM - s.ash_window + 1) / kBN;
      const int n_sink = min(cdiv(s.ash_init, kBN), t_lo);
      s.n_tiles = n_sink + (r - t_lo + 1);
    }
  } else if (is_vs(PAT)) {
    if (PAT == kPatVSExp) {
      // the key blocks this row block needs: x = 2 r + 1 - kb for x in [0, 2 r + 1]
      // with 64-block distance x or x - 1 kept, and x = 2 r + 1 (block 0), as a
      // bitmap over x in list[kVsxBits ..]
      const uint32_t* eb = a.offbits + (size_t)n * a.Nw;
      const int X = 2 * r + 2, nfw = cdiv(X, 32);
      uint32_t* fb = reinterpret_cast<uint32_t*>(&s.list[kVsxBits]);
      int mine = 0;
      for (int w = tid; w < nfw; w += 192) {
        const uint32_t ew = __ldg(eb + w), ep = (w > 0) ? __ldg(eb + w - 1) : 0u;
        uint32_t f = ew | (ew << 1) | (ep >> 31);
        if (w == nfw - 1) {
          f |= 1u << ((X - 1) & 31);                   // x = 2 r + 1: block 0
          if (X & 31) f &= (1u << (X & 31)) - 1u;     // nothing past x = 2 r + 1
        }
        fb[w] = f;
        mine += __popc(f);
      }
      int total;
      block_excl_scan(mine, s.scan, &total);  // (its barriers also publish the bitmap)
      if (tid == 0) {
        s.d_cnt = total;                // needed blocks, paired two per tile
        s.n_contig = (total + 1) >> 1;
      }
    } else {
      // contiguous tiles: tile 0, then the windows p < 128 r (keys 128 r - p ..).
      // All threads count in parallel (independent loads).
      const int* dl = a.dlist + (size_t)n * a.NT;
      const int dc = __ldg(a.dcount + n);
      int below = 0;  // s.has_t0 was set to 1 before the barrier-init sync
      for (int e = tid; e < dc; e += 192) below += (__ldg(dl + e) < r * kBN) ? 1 : 0;
      int n_below;
      block_excl_scan(below, s.scan, &n_below);
      if (tid == 0) {
        s.d_cnt = n_below;
        s.n_contig = n_below + s.has_t0;
      }
      for (int w = tid; w < a.NTw; w += 192) s.dfull[w] = __ldg(a.dfull + (size_t)n * a.NTw + w);
    }
    // column tiles: chunks of 128 entries of the head's compacted column list,
    // from the first column past tile 0 (entry lo) to the last before this row
    // block (entry hi); an entry is kept when its column is residual (no
    // contiguous tile of this row block covers it), a chunk when it keeps one
    const int* cl = a.clist + (size_t)n * MI_MAX_KV;
    const uint32_t* db = (PAT == kPatVSExp) ? a.offbits + (size_t)n * a.Nw : a.dbits + (size_t)n * a.Dw;
    const int cnt = __ldg(a.ccount + n);
    const int j_first = (PAT == kPatVSExp) ? kBlk : kBN;  // past block 0, or past tile 0
    uint32_t* resbits = reinterpret_cast<uint32_t*>(&s.list[16]);  // 64 words: entries lo .. lo + 2047
    if (tid < 64) resbits[tid] = 0u;
    int c_lo = 0, c_hi = 0;
    for (int e = tid; e < cnt; e += 192) {
      const int j = __ldg(cl + e);
      c_lo += (j < j_first) ? 1 : 0;
      c_hi += (j < r * kBN) ? 1 : 0;
    }
    int lo, hi;
    block_excl_scan(c_lo, s.scan, &lo);  // (its barriers also order the resbits clear)
    block_excl_scan(c_hi, s.scan, &hi);
    for (int e = lo + tid; e < hi; e += 192) {
      if (residual_column<PAT>(__ldg(cl + e), a.N, r, db))
        atomicOr(&resbits[(e - lo) >> 5], 1u << ((e - lo) & 31));
    }
    __syncthreads();
    if (tid == 0) {
      int nc = 0;
      for (int c = 0; c < cdiv(hi - lo, kBN); ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(&resbits[4 * c]);
        if (w.x | w.y | w.z | w.w) s.list[nc++] = c;
      }
      s.n_list = nc;
      s.col_lo = lo;
      s.n_tiles = s.n_contig + nc;
    }
  } else {  // block-sparse: the two 64-row halves' selected 64-key blocks, paired into 128-key tiles
    // A tile holds any two blocks A (keys 0-63) and B (keys 64-127).  Blocks
    // selected by both halves pair with each other (tiles kept whole); the
    // blocks only one half selected pair with the other half's (each half keeps
    // its own block of the tile).  The bitmaps and lists live in the V buffer,
    // which the loads only fill after this prologue.
    const int NB = cdiv(a.N, kBlk);
    const int nblk = min(2 * r + 2, NB);  // blocks this CTA's rows can select
    const int nwb = cdiv(nblk, 32);
    uint32_t* bm0 = reinterpret_cast<uint32_t*>(&s.v[0][0]);  // <= 1024 words each (N <= 2^21)
    uint32_t* bm1 = bm0 + nwb;
    int* lc = reinterpret_cast<int*>(bm1 + nwb);  // selected by both halves
    int* l0 = lc + a.topk;                        // by the first half only
    int* l1 = l0 + a.topk;                        // by the second half only (3 x topk <= 3 K ints)
    for (int w = tid; w < 2 * nwb; w += kAttnThreads) bm0[w] = 0u;
    __syncthreads();
    const int* b0 = a.blk_idx + ((size_t)n * NB + 2 * r) * a.topk;  // row half 1 follows at + topk
    const int nsel = ((2 * r + 1) < NB) ? 2 * a.topk : a.topk;
    for (int i = tid; i < nsel; i += kAttnThreads) {
      const int hf = (i >= a.topk) ? 1 : 0;
      const int c = __ldg(b0 + i);
      if (c >= 0 && c <= 2 * r + hf) atomicOr(&(hf ? bm1 : bm0)[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
    const int per = cdiv(nwb, kAttnThreads);
    const int w0 = min(tid * per, nwb), w1 = min(w0 + per, nwb);
    int nc = 0, n0 = 0, n1 = 0;
    for (int w = w0; w < w1; ++w) {
      const uint32_t x0 = bm0[w], x1 = bm1[w];
      nc += __popc(x0 & x1);
      n0 += __popc(x0 & ~x1);
      n1 += __popc(x1 & ~x0);
    }
    int tc, t0, t1;
    int pc = block_excl_scan(nc, s.scan, &tc);
    int p0 = block_excl_scan(n0, s.scan, &t0);
    int p1 = block_excl_scan(n1, s.scan, &t1);
    for (int w = w0; w < w1; ++w) {
      const uint32_t x0 = bm0[w], x1 = bm1[w];
      for (uint32_t m = x0 & x1; m; m &= m - 1) lc[pc++] = 32 * w + __ffs(m) - 1;
      for (uint32_t m = x0 & ~x1; m; m &= m - 1) l0[p0++] = 32 * w + __ffs(m) - 1;
      for (uint32_t m = x1 & ~x0; m; m &= m - 1) l1[p1++] = 32 * w + __ffs(m) - 1;
    }
    __syncthreads();
    const int ncp = (tc + 1) / 2;
    const int ntile = ncp + max(t0, t1);  // <= topk <= MI_MAX_KV / 2
    for (int t = tid; t < ntile; t += kAttnThreads) {
      int A, Bb, sub;
      if (t < ncp) {
        A = lc[2 * t];
        Bb = (2 * t + 1 < tc) ? lc[2 * t + 1] : -1;
        sub = (Bb >= 0) ? 0xF : 0x5;
      } else {
        const int j = t - ncp;
        A = (j < t0) ? l0[j] : -1;
        Bb = (j < t1) ? l1[j] : -1;
        sub = (A >= 0 ? 0x1 : 0) | (Bb >= 0 ? 0x8 : 0);
      }
      // an empty half of a tile loads the other block again (finite data, masked)
      if (A < 0) A = Bb;
      if (Bb < 0) Bb = A;
      s.list[2 * t] = (A << 4) | sub;
      s.list[2 * t + 1] = Bb;
    }
    if (tid == 0) {
      s.n_list = ntile;
      s.n_tiles = ntile;
    }
    __syncthreads();  // the lists in the V buffer are read before any V load is issued
    fence_proxy_async_smem();  // generic writes to the V buffer before its TMA loads
  }
  __syncthreads();
}

// ---------------------------------------------------------------- kernel ----

// The engine for one CTA: row block r of head h, whose pattern arrays sit at
// slot n.  Called by the per-pattern kernels and by the layer kernel.
template <int PAT>
__device__ __forceinline__ void attn_body(uint8_t* smem_raw, const CUtensorMap& map_q,
                                          const CUtensorMap& map_k, const CUtensorMap& map_v,
                                          const CUtensorMap& map_kr, const CUtensorMap& map_vr,
                                          const AttnArgs& a, int r, int n, int h) {
  AttnSmem& s = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const int g = h / a.group;
  // Work-free CTAs leave before any set-up (the same decision in every thread):
  // a Q-boundary pass's row block without its modality, a grid-rows block past
  // the head's lattice rows.
  if (a.modality && !((__ldg(a.blk_mods + r) >> a.row_mod) & 1u)) return;
  int g_sigma = 1, g_phi = 0, g_lines = 0;
  if (PAT == kPatRows) {
    g_sigma = __ldg(a.grid + 2 * n);
    g_phi = __ldg(a.grid + 2 * n + 1);
    if (g_sigma >= max(a.grid_sigma_min, 1) && g_phi >= 0 && g_phi < g_sigma && g_phi < a.N)
      g_lines = (a.N - 1 - g_phi) / g_sigma + 1;
    if (r * kBM >= g_lines) return;
  }

  if (tid == 0) {
    s.g_sigma = g_sigma;
    s.g_phi = g_phi;
    s.g_lines = g_lines;
    mbar_init(&s.q_full, 1);
    mbar_init(&s.k_full, 1);
    mbar_init(&s.k_empty, 1);
    mbar_init(&s.v_full, 1);
    mbar_init(&s.v_empty, 1);
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_full, 128);
    mbar_init(&s.p_part[0], 128);
    mbar_init(&s.p_part[1], 128);
    mbar_init(&s.p_part[2], 128);
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.mma_done, 1);
    mbar_init(&s.m_full[0], 32);
    mbar_init(&s.m_full[1], 32);
    s.abort = 0;
    s.has_t0 = 1;
    s.ash_init = a.ash_n ? a.ash_pairs[2 * n] : a.n_init;
    s.ash_window = a.ash_n ? a.ash_pairs[2 * n + 1] : a.window;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&s.tmem, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 160) {
    tma_prefetch_map(&map_k);
    tma_prefetch_map(&map_v);
    if (is_vs(PAT)) {
      tma_prefetch_map(&map_kr);
      tma_prefetch_map(&map_vr);
    }
  }
  __syncthreads();  // barriers initialised
  if (PAT == kPatRows) {
    // the lattice rows phi + sigma (128 r + i), copied by the loader warp into the
    // 128-byte-swizzled Q tile (rows past the lattice are zero), then made
    // visible to the tensor core's proxy
    if (warp == 5 && !a.skip_q_load) {
      const int l = lane_id();
#pragma unroll 1
      for (int i = l; i < kBM; i += 32) {
        const bool live = r * kBM + i < g_lines;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + ((size_t)h * a.ld + (live ? g_phi + g_sigma * (r * kBM + i) : 0)) * kD);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint4 val = live ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(s.q[u >> 3] + sw128_offset(i, u & 7)) = val;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (l == 0) mbar_arrive(&s.q_full);
    }
  } else if (tid == 160 && !a.skip_q_load) {  // Q does not depend on the tile list: load it first
    mbar_arrive_expect_tx(&s.q_full, 2 * 16384);
    tma_load_3d(s.q[0], &map_q, &s.q_full, 0, r * kBM, h);
    tma_load_3d(s.q[1], &map_q, &s.q_full, 64, r * kBM, h);
  }
  tc_fence_before();
  attn_prologue<PAT>(s, a, n, r);  // ends with __syncthreads
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  const int T = s.n_tiles;
  volatile int* abort = &s.abort;
  const uint64_t lim = a.wait_limit_ns;

  if (warp == 4) {
    // ------------------------------------------------------------ MMA ----
    if (lane_id() == 0) {
      const uint32_t id_qk = idesc_bf16(kBM, kBN, 0);
      const uint32_t id_pv = idesc_bf16(kBM, kD, 1);
      bool ok = mbar_wait(&s.q_full, 0, abort, lim);
      for (int t = 0; t < T && ok; ++t) {
        ok = mbar_wait(&s.k_full, t & 1, abort, lim);
        // S is overwritten: P of the previous tile must have been consumed
        if (ok && t >= 1) ok = mbar_wait(&s.pv_done, (t - 1) & 1, abort, lim);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sdesc_sw128(smem_u32(s.q[kk >> 2]) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(s.k[kk >> 2]) + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem, ad, bd, id_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s.s_full);
        umma_commit(&s.k_empty);
        constexpr int NQ = kPChunks<PAT>;
        ok = mbar_wait(&s.v_full, t & 1, abort, lim);
#pragma unroll
        for (int qq = 0; qq < NQ && ok; ++qq) {
          ok = mbar_wait(qq < NQ - 1 ? &s.p_part[qq] : &s.p_full, t & 1, abort, lim);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = qq * (8 / NQ); kk < (qq + 1) * (8 / NQ); ++kk) {
            const uint64_t bd = sdesc_sw128(smem_u32(s.v[0]) + kk * 2048, 16384, 1024);
            umma_bf16_ts(tmem + kTmemO, tmem + kk * 8, bd, id_pv, (t > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        umma_commit(&s.pv_done);
        umma_commit(&s.v_empty);
      }
      umma_commit(&s.mma_done);  // completes when everything issued above is done
      mbar_wait_drain(&s.mma_done, 0, lim);
    }
    __syncwarp();
  } else if (warp == 5) {
    // -------------------------------------------------------------- loader ----
    int issued = 0;
    // the next tile's reference (a global load for vertical-slash heads) is read
    // before waiting for the buffers, so its latency overlaps those waits
    VsxCursor cur{0, (PAT == kPatVSExp) ? reinterpret_cast<const uint32_t*>(&s.list[kVsxBits])[0] : 0u};
    auto next_ref = [&](int i) -> TileRef {
      if (PAT == kPatVSExp && i < s.n_contig) return cur.tile(s, r, i);
      return tile_at<PAT>(s, a, n, r, i);
    };
    TileRef ref_next = (T > 0) ? next_ref(0) : TileRef{0, 0, 0, 0};
    auto load = [&](const TileRef& ref, const CUtensorMap* map, const CUtensorMap* rows_map,
                    uint64_t* full, uint8_t (*buf)[16384]) {
      if (ref.kind == 0) {
        // two 64-key boxes per 64-column half: keys 0-63 and 64-127 of the
        // tile (for block-sparse tiles, blocks ref.t and ref.t2)
        if (lane_id() == 0) {
          // block pattern: blocks t and t2; block-expanded slashes: blocks t and t2 (t
          // again when there is no second block: loaded, masked out)
          const int ka = (PAT == kPatBlock || PAT == kPatVSExp) ? ref.t * kBlk : is_vs(PAT) ? ref.j0 : ref.t * kBN;
          const int kb = (PAT == kPatBlock) ? ref.t2 * kBlk
                         : (PAT == kPatVSExp) ? (ref.t2 >= 0 ? ref.t2 : ref.t) * kBlk
                         : is_vs(PAT) ? ref.j0 + kBlk : ref.t * kBN + kBlk;
          mbar_arrive_expect_tx(full, 2 * 16384);
          tma_load_3d(buf[0], map, full, 0, ka, g);
          tma_load_3d(buf[0] + 8192, map, full, 0, kb, g);
          tma_load_3d(buf[1], map, full, 64, ka, g);
          tma_load_3d(buf[1] + 8192, map, full, 64, kb, g);
        }
      } else {
        // a column tile: 128 consecutive rows of the head's compacted K or V
        // columns (rows_map: [listed heads, MI_MAX_KV, 128]), two 64-row boxes
        // per 64-column half
        if (lane_id() == 0) {
          const int row0 = s.col_lo + ref.t * kBN;
          mbar_arrive_expect_tx(full, 2 * 16384);
          tma_load_3d(buf[0], rows_map, full, 0, row0, n);
          tma_load_3d(buf[0] + 8192, rows_map, full, 0, row0 + kBlk, n);
          tma_load_3d(buf[1], rows_map, full, 64, row0, n);
          tma_load_3d(buf[1] + 8192, rows_map, full, 64, row0 + kBlk, n);
        }
      }
    };
    // vertical-slash: this warp also builds the keep-masks, lane l for rows
    // l + 32 i; their raw words are loaded a tile ahead of their use
    const int q0 = r * kBM + static_cast<int>(lane_id());
    VsRaw4 raw_next;
    if (is_vs(PAT) && T > 0) raw_next = vs_fetch4<PAT>(s, a, n, r, ref_next, q0);
    for (int t = 0; t < T; ++t) {
      const TileRef ref = ref_next;
      VsRaw4 raw;
      if (is_vs(PAT)) raw = raw_next;
      if (t + 1 < T) ref_next = next_ref(t + 1);
      if (t >= 1 && !mbar_wait_warp(&s.k_empty, (t - 1) & 1, abort, lim)) break;
      load(ref, &map_k, &map_kr, &s.k_full, s.k);
      if (is_vs(PAT)) {
        // stage t & 1 was last read by the softmax of tile t - 2, which ended
        // before P.V of t - 2 and hence before S of t - 1 (waited for above)
        uint32_t mk[4][4];
        vs_masks4<PAT>(s, a, r, raw, q0, mk);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(&s.vmask[t & 1][lane_id() + 32 * i][0]) =
              make_uint4(mk[i][0], mk[i][1], mk[i][2], mk[i][3]);
        mbar_arrive(&s.m_full[t & 1]);
        if (t + 1 < T) raw_next = vs_fetch4<PAT>(s, a, n, r, ref_next, q0);
      }
      if (t >= 1 && !mbar_wait_warp(&s.v_empty, (t - 1) & 1, abort, lim)) {
        issued = -(t + 1);  // K of tile t issued, V not
        break;
      }
      load(ref, &map_v, &map_vr, &s.v_full, s.v);
      issued = t + 1;
      __syncwarp();
    }
    // drain: the last loads must land before the CTA can exit
    if (lane_id() == 0) {
      mbar_wait_drain(&s.q_full, 0, lim);
      const int nk = issued < 0 ? -issued : issued, nv = issued < 0 ? -issued - 1 : issued;
      if (nk > 0) mbar_wait_drain(&s.k_full, (nk - 1) & 1, lim);
      if (nv > 0) mbar_wait_drain(&s.v_full, (nv - 1) & 1, lim);
    }
    __syncwarp();
  } else if (warp < 4) {
    // --------------------------------------------------------- softmax ----
    const int row = tid;  // TMEM lane and row within the block
    // the row's position: the block's row, or for grid rows the lattice row
    const int q = (PAT == kPatRows) ? g_phi + g_sigma * (r * kBM + row) : r * kBM + row;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t s_addr = tmem + lane_base, o_addr = tmem + lane_base + kTmemO;
    const float sl = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // other patterns: tile references are read one and two tiles ahead;
    // vertical-slash masks come ready-made from the loader warp
    TileRef ref_next2{0, 0, 0};
    MaskRaw raw_next{};
    if constexpr (!is_vs(PAT)) {
      ref_next2 = (T > 1) ? tile_at<PAT>(s, a, n, r, 1) : TileRef{0, 0, 0, 0};
      raw_next = mask_fetch<PAT>(a, (T > 0) ? tile_at<PAT>(s, a, n, r, 0) : TileRef{0, 0, 0, 0});
    }
    for (int t = 0; t < T; ++t) {
      uint32_t mk[4];
      if constexpr (is_vs(PAT)) {
        ok = mbar_wait_warp(&s.m_full[t & 1], (t >> 1) & 1, abort, lim);
        if (!ok) break;
        const uint4 m4 = *reinterpret_cast<const uint4*>(&s.vmask[t & 1][row][0]);
        mk[0] = m4.x;
        mk[1] = m4.y;
        mk[2] = m4.z;
        mk[3] = m4.w;
        ok = mbar_wait_warp(&s.s_full, t & 1, abort, lim);
        if (!ok) break;
        tc_fence_after();
      } else {
        const MaskRaw raw = raw_next;
        if (t + 1 < T) raw_next = mask_fetch<PAT>(a, ref_next2);
        if (t + 2 < T) ref_next2 = tile_at<PAT>(s, a, n, r, t + 2);
        ok = mbar_wait_warp(&s.s_full, t & 1, abort, lim);
        if (!ok) break;
        tc_fence_after();
        mask_finish<PAT>(s, a, r, raw, q, mk);
      }
      // the row of S in registers: one tensor-memory read per tile
      float x[128];
      tmem_ld128(s_addr, x);  // one x128 load (measured 2-6 % faster than two x64)
      // masked keys read as -inf.  A row of an exact vertical-slash tile is
      // almost never kept whole, so those tiles select without a per-row branch
      // (measured: the branch cost more than it saved); the other patterns and
      // the block-expanded slashes skip the rows whose mask is all ones.
      if (PAT == kPatVS || (mk[0] & mk[1] & mk[2] & mk[3]) != 0xFFFFFFFFu) {
#pragma unroll
        for (int e = 0; e < 128; ++e) x[e] = ((mk[e >> 5] >> (e & 31)) & 1u) ? x[e] : -INFINITY;
      }
      // row maximum as a tree: eight independent chains of three-input max
      float m8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m8[j] = fmaxf(x[j], x[8 + j]);
#pragma unroll
      for (int e = 16; e < 128; e += 16) {
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = fmax3(m8[j], x[e + j], x[e + 8 + j]);
      }
      const float mraw = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
      const float mx = mraw * sl;  // sl > 0: the maximum commutes with the scale
      const bool upd = mx > m_ref + 8.0f;
      const bool rescale_o = upd && (m_ref != -INFINITY);
      float alpha = 1.f;
      if (rescale_o) alpha = fast_exp2(m_ref - mx);
      if (upd) {
        l *= alpha;
        m_ref = mx;
      }
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
      // P = exp2(x * sl - m) as bf16 pairs over the consumed S columns; the
      // scale-and-shift and the row sum take two keys per instruction (f32x2)
      float2 rs4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // independent partial sums
      const float2 sl2 = make_float2(sl, sl), nmb2 = make_float2(-mb, -mb);
      const bool resc = __any_sync(0xffffffffu, rescale_o);
      constexpr int NQ = kPChunks<PAT>, CP = 64 / NQ;  // chunks, bf16 pairs per chunk
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) {
        uint32_t pk[CP];
#pragma unroll
        for (int e = 0; e < CP; ++e) {
          const float2 y = fma2(make_float2(x[qq * 2 * CP + 2 * e], x[qq * 2 * CP + 2 * e + 1]), sl2, nmb2);
          const float2 p = make_float2(fast_exp2(y.x), fast_exp2(y.y));
          rs4[e & 3] = add2(rs4[e & 3], p);
          __nv_bfloat162 bb = __floats2bfloat162_rn(p.x, p.y);
          pk[e] = *reinterpret_cast<uint32_t*>(&bb);
        }
        if constexpr (CP == 32) {
          tmem_st32u(s_addr + qq * CP, pk);
        } else {
          tmem_st16(s_addr + qq * CP, pk);
        }
        if (qq < NQ - 1 && !resc) {  // P.V of these keys can start now
          tc_fence_before();
          mbar_arrive(&s.p_part[qq]);
        }
      }
      // O holds P.V of tiles < t (that P.V completed before S of tile t was
      // written); it is rescaled after P is stored, when the row is dead
      // and its registers are free
      if (resc) {  // tcgen05.ld/st are warp-collective
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(o_addr + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(o_addr + c * 32, o);
        }
      }
      const float2 rs = add2(add2(rs4[0], rs4[1]), add2(rs4[2], rs4[3]));
      l += rs.x + rs.y;
      tc_fence_before();
      if (resc) {
#pragma unroll
        for (int qq = 0; qq < NQ - 1; ++qq) mbar_arrive(&s.p_part[qq]);
      }
      mbar_arrive(&s.p_full);
    }
    // epilogue: O / l
    if (ok && T > 0) ok = mbar_wait_warp(&s.pv_done, (T - 1) & 1, abort, lim);
    if (ok) {
      tc_fence_after();
      const bool in_range = ((PAT == kPatRows) ? (r * kBM + row < g_lines) : (q < a.N)) &&
                            (!a.modality || __ldg(a.modality + q) == a.row_mod);
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow = a.out + ((size_t)h * a.ld + q) * kD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(o_addr + c * 32, o);
        if (in_range) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              // a row that kept no key (possible in the cross-modality pass, whose
              // O may never have been written) is written as zeros
              __nv_bfloat162 bb = (l > 0.f) ? __floats2bfloat162_rn(o[u * 8 + 2 * e] * inv,
                                                                    o[u * 8 + 2 * e + 1] * inv)
                                            : __floats2bfloat162_rn(0.f, 0.f);
              pk[e] = *reinterpret_cast<uint32_t*>(&bb);
            }
            *reinterpret_cast<uint4*>(orow + c * 32 + u * 8) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      if (in_range && a.lse)
        a.lse[(size_t)h * a.ld + q] =
            (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s.abort && tid == 0) set_status(a.status, MI_ERR_TIMEOUT);
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One pattern for all listed heads: blockIdx.y is the listed head, blockIdx.x
// the row block counted from the last (the heaviest first).
template <int PAT>
__global__ void __launch_bounds__(kAttnThreads, 2)
attn_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_kr,
            const __grid_constant__ CUtensorMap map_vr, const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int n = blockIdx.y;
  attn_body<PAT>(smem_raw, map_q, map_k, map_v, map_kr, map_vr, a,
                 static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x), n, a.heads.h[n]);
}

}  // namespace mi

namespace mi {

// Host launcher, explicitly instantiated in attn_kernels_*.cu so that the
// pattern variants compile in parallel.
template <int PAT>
cudaError_t launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mkr, const CUtensorMap& mvr, const AttnArgs& a,
                        int n_row_blocks, cudaStream_t st);

// Layer launcher (all patterns of a layer's heads in one launch).
cudaError_t launch_attn_layer(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                              const CUtensorMap& mkr, const CUtensorMap& mvr, const AttnArgs& a,
                              int n_row_blocks, cudaStream_t st);

}  // namespace mi
