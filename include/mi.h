/*
 * mi.h - C ABI of libmi.so: dynamic sparse prefill attention on one GB300 (sm_103a).
 *
 * The method (MInference): every attention head follows one of three sparse
 * patterns, fixed per head offline; for vertical-slash heads the concrete
 * indices are estimated online from the input, and sparse kernels then compute
 * only the kept part of causal attention.
 *   - MInference README mirror, gittoolsai.com, "TL;DR" (offline pattern per
 *     head, online approximation of the sparse indices, custom kernels) and
 *     "Kernel-only usage" (vertical_slash_sparse_attention(q, k, v,
 *     vertical_topk, slash), block_sparse_attention(q, k, v, topk),
 *     streaming_forward(q, k, v, init_num, local_window_num)).
 *   - MInference talk slides, boteman.cn (H. Jiang, "System-Algorithm
 *     Co-design"): the A-shape, Vertical-Slash and block-sparse patterns;
 *     "Step 2: Online Estimation of Sparsity Indices"; "Dynamic Sparse
 *     Attention Calculation with PIT, FlashAttention".
 *
 * Conventions shared by every call
 * --------------------------------
 *  Tensors.  q: [Hq, N, d], k and v: [Hkv, N, d], out: [Hq, N, d]; all bf16
 *    (mi_bf16 = raw bf16 bits), row-major and contiguous, DEVICE pointers owned
 *    by the caller.  d must be 128 and 1 <= N <= 2^21 (the estimation, which
 *    scores the last 64 queries, needs N >= 64).  A last, partial 64-block of
 *    rows or keys is a block of its own (block-sparse pooling takes the mean
 *    of its rows).
 *    Grouped-query attention: q-head h reads KV head h / (Hq / Hkv);
 *    Hq % Hkv == 0.  q, k, v, out must be 16-byte aligned.
 *  Heads.  `heads` is a HOST array of n_heads distinct q-head indices in
 *    [0, Hq) (at most MI_MAX_HEADS); NULL means all heads 0..Hq-1 and then
 *    n_heads must equal Hq.  Per-head index arrays (v_idx, s_idx, blk_idx) are
 *    laid out in the order of this list.  Only the listed heads' rows of
 *    `out` (and `lse`) are written, so three pattern calls with disjoint head
 *    lists fill one layer's output.
 *  lse.  Optional DEVICE float [Hq, N]: natural-log sum of exp(q.k/sqrt(d))
 *    over the kept keys of each row (NULL = not written).
 *  Softmax scale is 1/sqrt(d) everywhere.
 *  Workspace.  Every call takes caller-owned DEVICE scratch of at least
 *    mi_workspace_bytes(op, ...) bytes, 256-byte aligned; its first word is the
 *    call's device status.  The library allocates no device memory, keeps no
 *    state between calls and never synchronizes inside a compute call: all
 *    work is queued on `stream` (0 = legacy default stream).  Calls that share
 *    a workspace must not overlap on the GPU.
 *  Errors.  A call returns MI_OK or a negative MI_ERR_* at launch time
 *    (argument, shape, workspace, CUDA launch errors); nothing crosses the ABI
 *    as an exception.  Errors that depend on data (an index out of range or
 *    unsorted, a pipeline wait that timed out) are written to the workspace
 *    status word; mi_read_status() reads it.  mi_strerror() describes a code.
 */
#ifndef MI_H
#define MI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mi_bf16;
typedef struct CUstream_st* mi_stream_t; /* a cudaStream_t */

#define MI_OK 0
#define MI_ERR_ARG (-1)           /* NULL/misaligned pointer, bad head list, k < 0, ... */
#define MI_ERR_SHAPE (-2)         /* d != 128, N out of range, Hq % Hkv != 0, last_q != 64, ... */
#define MI_ERR_WORKSPACE (-3)     /* workspace NULL, misaligned or smaller than required */
#define MI_ERR_CUDA (-4)          /* a CUDA call or kernel launch failed */
#define MI_ERR_INDEX (-5)         /* device status: index out of range or not strictly ascending */
#define MI_ERR_TIMEOUT (-6)       /* device status: a bounded pipeline wait expired */
#define MI_ERR_UNIMPLEMENTED (-7) /* option not supported by this build */
#define MI_ERR_DEVICE (-8)        /* current device is not an sm_103 GPU */

#define MI_MAX_HEADS 256
#define MI_HEAD_DIM 128
#define MI_LAST_Q 64
#define MI_BLOCK 64
#define MI_MAX_KV 2048 /* largest vertical budget the sparse attention kernel accepts */
#define MI_MAX_MODALITIES 8    /* modalities a Q-boundary call accepts */
#define MI_GRID_MAX_SIGMA 4096 /* largest stride range a grid estimation scans */
#define MI_MAX_RUNS 64         /* modality runs a 2D-boundary call accepts */

/* ops for mi_workspace_bytes */
#define MI_OP_VS_ESTIMATE 1
#define MI_OP_VS_SPARSE_ATTN 2
#define MI_OP_BLOCK_SPARSE_ATTN 3
#define MI_OP_ASHAPE_ATTN 4
#define MI_OP_DENSE_CAUSAL_ATTN 5
#define MI_OP_GRID_ESTIMATE 6
#define MI_OP_GRID_ATTN 7
#define MI_OP_QBOUNDARY_ESTIMATE 8
#define MI_OP_QBOUNDARY_ATTN 9
#define MI_OP_BOUNDARY2D_ATTN 10

/* flags for mi_block_sparse_attn */
#define MI_IDX_GIVEN 1

/*
 * Bytes of workspace `op` needs.  Unused arguments may be 0.  Returns 0 for an
 * unknown op or impossible sizes.
 */
size_t mi_workspace_bytes(int op, int n_heads, int Hkv, int N, int k_v, int k_s, int topk);

/*
 * Online estimation of vertical-slash indices for the listed heads.
 * Slides: "Step 2: Online Estimation of Sparsity Indices"; README mirror,
 * "Kernel-only usage" (vertical_topk, slash).
 *
 * For each listed q-head h with KV head g and the query rows
 * p_i = N - last_q + i (i < last_q):
 *   l_ij = q[h,p_i].k[g,j] / sqrt(d) for j <= p_i, a_ij = softmax_j(l_ij),
 *   vertical score  v[j] = sum_i a_ij,
 *   slash score     s[o] = sum_i a_{i, p_i - o}   (diagonal offset o = q - j).
 * v_idx[n, 0..k_v') receives the k_v' = min(k_v, N) columns with the largest
 * v and s_idx[n, 0..k_s') the k_s' = min(k_s, N) offsets with the largest s
 * (ties: lower index first), each sorted ascending.  v_idx is [n_heads, k_v]
 * and s_idx [n_heads, k_s] int32 DEVICE arrays; entries beyond k_v' / k_s'
 * are set to -1.  last_q must be 64; k_v, k_s >= 0 (0 is legal).
 * Scores are accumulated in fp32 from bf16 tensor-core products.
 */
int mi_vs_estimate(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                   const int32_t* heads, int n_heads, int last_q, int k_v, int k_s,
                   int32_t* v_idx, int32_t* s_idx, void* workspace, size_t ws_bytes,
                   mi_stream_t stream);

/*
 * Vertical-slash sparse attention with given indices.
 * Slides: "Vertical-Slash" pattern and "Dynamic Sparse Attention Calculation
 * with PIT, FlashAttention"; README mirror: vertical_slash_sparse_attention.
 *
 * flags = 0 (exact diagonals): row q of head h keeps key j iff j <= q and
 * (j < 64 or j/64 == q/64 or j in v_idx[n] or q - j in s_idx[n]); a key kept
 * by several rules counts once.
 * flags = MI_VS_BLOCK_EXPANDED (the 64x64 block cover of the diagonals used by
 * the pages' block kernels): with D = {0} and, for each o in s_idx[n], o/64 and
 * (if o % 64 != 0) o/64 + 1 -- the 64-block distances a diagonal o crosses --
 * row q keeps key j iff j <= q and (j < 64 or j in v_idx[n] or
 * q/64 - j/64 in D): every 64x64 block a selected diagonal passes through is
 * kept whole.
 * out[h, q] = softmax over kept keys of q.k/sqrt(d), times V.
 * v_idx: [n_heads, k_v] and s_idx: [n_heads, k_s] int32 DEVICE arrays, each row
 * strictly ascending, values in [0, N); a trailing run of -1 is allowed and
 * ignored (the layout mi_vs_estimate writes).  An entry out of range or out of
 * order sets MI_ERR_INDEX in the status word and is skipped.  k_v <= MI_MAX_KV.
 * Unknown flag bits: MI_ERR_UNIMPLEMENTED.
 */
#define MI_VS_BLOCK_EXPANDED 1
int mi_vs_sparse_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                      int N, int d, const int32_t* heads, int n_heads, const int32_t* v_idx,
                      int k_v, const int32_t* s_idx, int k_s, int flags, mi_bf16* out, float* lse,
                      void* workspace, size_t ws_bytes, mi_stream_t stream);

/*
 * Block-sparse attention over 64x64 blocks.
 * Slides: "block-sparse" pattern; README mirror: block_sparse_attention(q, k, v, topk).
 *
 * Query block r (rows 64r..64r+63) keeps key blocks c <= r.  Unless
 * (flags & MI_IDX_GIVEN), the blocks are chosen here: the top-min(topk, r+1)
 * blocks by sigma[r, c] = mean(q rows of block r) . mean(k rows of block c)
 * (ties: lower c), and written to blk_idx.  With MI_IDX_GIVEN, blk_idx is read
 * (a row that is not ascending, exceeds r or has a value after -1 padding
 * sets MI_ERR_INDEX).  blk_idx: [n_heads, ceil(N/64), topk] int32 DEVICE array; each
 * row ascending, padded with -1 after the last selected block.  Row q keeps j
 * iff j <= q and j/64 is selected for q/64.  block must be 64,
 * 1 <= topk <= MI_MAX_KV / 2.
 */
int mi_block_sparse_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                         int N, int d, const int32_t* heads, int n_heads, int block, int topk,
                         int32_t* blk_idx, int flags, mi_bf16* out, float* lse, void* workspace,
                         size_t ws_bytes, mi_stream_t stream);

/*
 * A-shape attention: attention sinks plus a local window.
 * Slides: "A-shape" pattern; README mirror: streaming_forward(q, k, v,
 * init_num, local_window_num).
 *
 * Row q keeps j iff j <= q and (j < n_init or q - j < window); both sizes in
 * tokens, n_init >= 0, window >= 1.
 */
int mi_ashape_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N,
                   int d, const int32_t* heads, int n_heads, int n_init, int window, mi_bf16* out,
                   float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream);

/*
 * Dense causal attention (row q keeps every j <= q): the FlashAttention
 * baseline the pages measure the sparse kernels against (slides: "Latency at
 * 1M tokens on a single A100: FlashAttn 30 mins vs MInference 3 mins").
 */
int mi_dense_causal_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                         int N, int d, const int32_t* heads, int n_heads, mi_bf16* out,
                         float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream);

/*
 * A whole layer in one call: every q-head with its own pattern and budgets.
 * Slides: "Step 1: Kernel-Aware Sparse Pattern Search" (each head's pattern is
 * fixed offline) and "Step 2: Online Estimation of Sparsity Indices" (the indices
 * of the dynamic patterns are found online); README mirror, "TL;DR".
 *
 * cfg: HOST array of Hq entries.  Head h gets the result of the per-pattern call
 * its cfg[h].pattern names, with that entry's budgets:
 *   MI_PAT_VS      mi_vs_estimate (k_v, k_s) + mi_vs_sparse_attn (vs_flags);
 *   MI_PAT_BLOCK   mi_block_sparse_attn with its own selection (topk);
 *   MI_PAT_ASHAPE  mi_ashape_attn (n_init, window);
 *   MI_PAT_DENSE   mi_dense_causal_attn;
 *   MI_PAT_SKIP    nothing (out rows of the head are left untouched).
 * Budgets may differ between heads; vs_flags must be the same for every
 * vertical-slash head.  Fields a pattern does not use are ignored.
 * The estimation and block selection run per group of heads with equal
 * budgets; the attention of every head of every pattern is ONE kernel launch,
 * ordered dense, vertical-slash, block-sparse, A-shape with the heaviest row
 * blocks first, so that lighter work fills the end of heavier work.
 * workspace: mi_layer_workspace_bytes(Hq, Hkv, N, cfg) bytes of device memory.
 * Errors: an invalid cfg entry returns MI_ERR_ARG (MI_ERR_SHAPE for shapes), as
 * the per-pattern calls do; data errors land in the status word
 * (mi_read_status on the workspace).
 */
#define MI_PAT_SKIP (-1)
#define MI_PAT_DENSE 0
#define MI_PAT_VS 1
#define MI_PAT_BLOCK 2
#define MI_PAT_ASHAPE 3
typedef struct {
  int32_t pattern;   /* MI_PAT_* */
  int32_t k_v, k_s;  /* vertical-slash budgets (0 <= k_v <= MI_MAX_KV, k_s >= 0) */
  int32_t vs_flags;  /* 0 or MI_VS_BLOCK_EXPANDED */
  int32_t topk;      /* block-sparse: 1 <= topk <= MI_MAX_KV / 2 */
  int32_t n_init, window; /* A-shape: n_init >= 0, window >= 1 */
} mi_head_cfg;

size_t mi_layer_workspace_bytes(int Hq, int Hkv, int N, const mi_head_cfg* cfg);

int mi_layer_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N,
                  int d, const mi_head_cfg* cfg, mi_bf16* out, float* lse, void* workspace,
                  size_t ws_bytes, mi_stream_t stream);

/*
 * A packed batch of sequences of any lengths (varlen), each through the layer
 * call above with the same cfg.  q: [Hq, total, d], k and v: [Hkv, total, d],
 * out: [Hq, total, d], lse (optional): [Hq, total]; sequence b holds tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 of every head and attends only to itself
 * (its own causal prefix).  cu_seqlens: HOST array of n_seqs + 1 non-decreasing
 * int32 with cu_seqlens[0] = 0 and cu_seqlens[n_seqs] = total; an empty
 * sequence is skipped.  A sequence shorter than 64 tokens (too short for the
 * estimation, which scores the last 64 queries) runs its vertical-slash heads
 * dense.  The sequences run one after another on the stream, sharing one
 * workspace of mi_layer_workspace_bytes_varlen(...) bytes and its status word.
 * Errors: a malformed cu_seqlens or a sequence longer than 2^21 returns
 * MI_ERR_ARG; otherwise as mi_layer_attn.
 */
size_t mi_layer_workspace_bytes_varlen(int Hq, int Hkv, const int32_t* cu_seqlens, int n_seqs,
                                       const mi_head_cfg* cfg);

int mi_layer_attn_varlen(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                         int total, int d, const int32_t* cu_seqlens, int n_seqs,
                         const mi_head_cfg* cfg, mi_bf16* out, float* lse, void* workspace,
                         size_t ws_bytes, mi_stream_t stream);

/*
 * Multi-modal heads (MMInference).  README mirror, "TL;DR": modality-aware,
 * permutation-based sparse attention for the grid pattern of visual inputs and
 * for the modality boundaries of mixed inputs.  Slides: "MMInference: Grid Head
 * in Multi-Modality" (horizontal and vertical lines, evenly spaced, often
 * symmetrical; stride and starting position vary with the context) and
 * "MMInference: Q-Boundary pattern" (intra-modality consistency).
 *
 * Grid head: one lattice L = {j : j = phi (mod sigma)} gives both the vertical
 * lines and the horizontal lines.  Row q keeps key j iff j <= q and (j < 64 or
 * j/64 == q/64 or j in L or q in L): a row on the lattice keeps its whole
 * causal row.
 *
 * mi_grid_estimate: (sigma, phi) per listed head from the vertical scores v of
 * the last 64 queries (as in mi_vs_estimate): the lattice with the largest
 * E(sigma, phi) = sum over j in L of v[j] - |L| * 64 / N over
 * sigma_min <= sigma <= sigma_max and 0 <= phi < sigma; ties go to the smaller
 * sigma, then the smaller phi (fp32 scores).  grid: DEVICE int32 [n_heads, 2]
 * = (sigma, phi).  1 <= sigma_min <= sigma_max <= N and
 * sigma_max - sigma_min < MI_GRID_MAX_SIGMA, else MI_ERR_ARG; last_q must be 64.
 * Workspace: mi_workspace_bytes(MI_OP_GRID_ESTIMATE, n_heads, Hkv, N, 0, 0, 0).
 */
int mi_grid_estimate(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                     const int32_t* heads, int n_heads, int last_q, int sigma_min, int sigma_max,
                     int32_t* grid, void* workspace, size_t ws_bytes, mi_stream_t stream);

/*
 * mi_grid_attn: grid attention with given (sigma, phi) (DEVICE int32 [n_heads, 2],
 * e.g. from mi_grid_estimate).  The vertical lines run as vertical-slash columns;
 * the horizontal lines are gathered 128 rows at a time (the "permuted grid")
 * and attend densely to their causal prefix.  sigma_min is a lower bound on
 * every head's sigma, at least ceil(N / MI_MAX_KV) (at most MI_MAX_KV lattice
 * columns), else MI_ERR_ARG; a (sigma, phi) below it or with phi outside
 * [0, sigma) sets MI_ERR_INDEX in the status word and that head's lattice (its
 * columns and its rows) is left out: its rows keep the first and own block only.  Workspace: mi_workspace_bytes(MI_OP_GRID_ATTN, n_heads, Hkv, N, 0, 0, 0).
 */
int mi_grid_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N, int d,
                 const int32_t* heads, int n_heads, const int32_t* grid, int sigma_min, mi_bf16* out,
                 float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream);

/*
 * Q-Boundary head: every token j carries a modality id modality[j] in
 * [0, n_mod) (DEVICE int32 [N], n_mod <= MI_MAX_MODALITIES), and a query row
 * follows the vertical-slash pattern of its own modality.
 *
 * mi_qboundary_estimate: for each modality m, the vertical-slash estimation of
 * mi_vs_estimate with the 64 query rows that end at the last token of m (rows
 * R - 64 .. R - 1, R = max(one past that token, 64)); v_idx [n_mod, n_heads, k_v]
 * and s_idx [n_mod, n_heads, k_s] DEVICE int32, each row as mi_vs_estimate
 * writes it.  An id outside [0, n_mod) sets MI_ERR_INDEX in the status word.
 * Workspace: mi_workspace_bytes(MI_OP_QBOUNDARY_ESTIMATE, n_heads, Hkv, N, 0, 0, 0).
 */
int mi_qboundary_estimate(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                          const int32_t* heads, int n_heads, const int32_t* modality, int n_mod,
                          int last_q, int k_v, int k_s, int32_t* v_idx, int32_t* s_idx, void* workspace,
                          size_t ws_bytes, mi_stream_t stream);

/*
 * mi_qboundary_attn: row q of modality m keeps what mi_vs_sparse_attn (exact
 * diagonals) keeps with v_idx[m] / s_idx[m] (layouts as above, original token
 * positions).  One vertical-slash pass per modality writes that modality's rows;
 * row blocks without it are skipped.  Index errors as mi_vs_sparse_attn.
 * Workspace: mi_workspace_bytes(MI_OP_QBOUNDARY_ATTN, n_heads, Hkv, N, 0, 0, 0).
 */
int mi_qboundary_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N, int d,
                      const int32_t* heads, int n_heads, const int32_t* modality, int n_mod,
                      const int32_t* v_idx, int k_v, const int32_t* s_idx, int k_s, mi_bf16* out,
                      float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream);

/*
 * 2D-Boundary head (slides, "MMInference: 2D-Boundary pattern": the modality
 * boundary splits both axes; "modality-separated continuity").  Two modalities,
 * given as runs: runs is a HOST int32 array [n_runs][2] of (modality 0 or 1,
 * length >= 1) in token order, the lengths summing to N, n_runs <= MI_MAX_RUNS.
 * Each modality's tokens, in order, form a sub-sequence in which the modality is
 * a vertical-slash head: its index sets are estimated from the sub-sequence's
 * last 64 tokens (as mi_vs_estimate on the sub-sequence alone) and its columns,
 * offsets, first block and own block count sub-sequence positions, so that a
 * diagonal continues across the other modality's tokens.  A sub-sequence of
 * fewer than 64 tokens is dense within itself.  Row q keeps, in addition, every
 * key j <= q of the other modality.
 * v_idx [2, Hq, k_v] and s_idx [2, Hq, k_s] (DEVICE int32, per modality, in
 * sub-sequence positions) receive the estimated sets, or with flags =
 * MI_IDX_GIVEN are read instead.  Every q-head is computed (no head list).
 * The tokens are permuted so that each sub-sequence is contiguous (the
 * "permutation-based" kernels of the README mirror's TL;DR), the within-modality
 * and cross-modality passes run separately and are merged by their log-sum-exps.
 * Workspace: mi_workspace_bytes(MI_OP_BOUNDARY2D_ATTN, Hq, Hkv, N, 0, 0, 0)
 * (holds permuted copies of q, k, v and o).  Malformed runs: MI_ERR_ARG.
 */
int mi_boundary2d_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N, int d,
                       const int32_t* runs, int n_runs, int k_v, int k_s, int32_t* v_idx, int32_t* s_idx,
                       int flags, mi_bf16* out, float* lse, void* workspace, size_t ws_bytes,
                       mi_stream_t stream);

/*
 * mi_vs_estimate_noalloc: mi_vs_estimate for callers that cannot allocate device
 * memory (for instance an engine whose memory pool owns the whole device, or a
 * plugin running where cudaMalloc is not allowed).  The pages have no
 * counterpart; this is a packaging variant of the call above.
 *
 * Same arguments, results and errors as mi_vs_estimate, minus the workspace: the
 * scratch is a fixed array of MI_NOALLOC_SCRATCH_BYTES (36 MiB) in device memory
 * owned by libmi.so, present on every GPU that loads the library until the
 * process exits.  The call allocates nothing.
 *  - Size limit: the job must fit the array, i.e.
 *    mi_workspace_bytes(MI_OP_VS_ESTIMATE, n_heads, Hkv, N, 0, 0, 0)
 *    <= MI_NOALLOC_SCRATCH_BYTES.  That size is 256 + 512 * n_heads * ceil(N / 1024)
 *    + 512 * n_heads + 8 * n_heads * N bytes, each of the five terms rounded up to
 *    a multiple of 256.  A whole 32-head layer fits up to N = 138686 tokens (so at
 *    128K tokens); 32 heads at N = 138687 do not.  A job that does not fit
 *    returns MI_ERR_WORKSPACE before any work is queued, after the argument and
 *    shape checks of mi_vs_estimate (which come first, as in that call).
 *  - Set-up: the first call on a device, with that device current, looks up the
 *    array's device address (once per device).  Make that first call before any
 *    stream capture begins.  The address belongs to the context of that first
 *    call: after a cudaDeviceReset the library must not be used again in the
 *    process.
 *  - Sharing: every call uses the same array and leaves its contents behind; the
 *    call clears what has to start at zero.  Calls that overlap on the GPU (on
 *    different streams or from different threads) race on the array and must be
 *    serialised by the caller.
 *  - The device status word lives in the shared array and cannot be read back
 *    with mi_read_status; use mi_vs_estimate with a workspace when it matters.
 */
#define MI_NOALLOC_SCRATCH_BYTES (36u << 20)
int mi_vs_estimate_noalloc(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                           const int32_t* heads, int n_heads, int last_q, int k_v, int k_s,
                           int32_t* v_idx, int32_t* s_idx, mi_stream_t stream);

/*
 * Test-only fault injection for the bounded-wait path.  mode 1 makes the
 * attention kernels skip their Q load, so the first pipeline wait of every CTA
 * expires after `wait_limit_ns`; the CTA then stops, drains what it issued,
 * frees its tensor memory and the call reports MI_ERR_TIMEOUT through the
 * status word.  No fault, trap or unbounded wait is involved.  mode 0 (the
 * default) restores normal operation and the 4 s limit (wait_limit_ns is
 * ignored).  Process-wide setting: not for concurrent use with real work.
 * Returns MI_OK, or MI_ERR_ARG for an unknown mode or a limit of 0 or above
 * 10 s.
 */
#define MI_FAULT_NONE 0
#define MI_FAULT_SKIP_Q_LOAD 1
int mi_debug_inject(int mode, uint64_t wait_limit_ns);

/*
 * Synchronizes `stream`, then returns the status word of the last call that
 * used `workspace` (MI_OK, MI_ERR_INDEX or MI_ERR_TIMEOUT), or MI_ERR_CUDA if
 * the synchronization or the read failed.
 */
int mi_read_status(const void* workspace, mi_stream_t stream);

/* Static description of an MI_* code; for MI_ERR_CUDA the text of the last
 * CUDA error seen by this thread is returned (thread-local buffer). */
const char* mi_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MI_H */
