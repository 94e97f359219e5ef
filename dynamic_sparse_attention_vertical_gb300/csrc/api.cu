// api.cu - the C ABI declared in include/mi.h.
//
// Host side: argument and shape checks, carving of the caller's workspace,
// TMA descriptor encoding and kernel launches on the caller's stream.  No
// device allocation, no synchronization (except mi_read_status), no state kept
// between calls.  The attention variants are compiled in attn_kernels_*.cu.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <utility>

#include "attention.cuh"
#include "block.cuh"
#include "estimate.cuh"
#include "mm.cuh"
#include "select.cuh"
#include "vs_index.cuh"

using namespace mi;

namespace {

thread_local char g_msg[512];

int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_msg, sizeof(g_msg), "CUDA error in %s: %s", where, cudaGetErrorString(e));
  return MI_ERR_CUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [heads, N, 128] bf16 as a 3-D tensor (d, N, heads), consecutive heads `ld` rows
// apart (ld = N for a contiguous tensor; a sequence of a packed batch keeps the
// batch's row count); box = 64 columns x box_rows rows, 128-byte swizzle (one box
// row = 128 bytes).  Rows past N read as zero.
int make_map(CUtensorMap* m, const void* base, int heads, int N, int box_rows, int64_t ld) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    snprintf(g_msg, sizeof(g_msg), "cuTensorMapEncodeTiled is not available from the driver");
    return MI_ERR_CUDA;
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(ld) * kD * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_msg, sizeof(g_msg), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MI_ERR_CUDA;
  }
  return MI_OK;
}

int check_device() {
  static int verdict[64];  // 0 unknown, 1 sm_103, -1 other (benign race: same value)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return MI_ERR_DEVICE;
  if (verdict[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    verdict[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (verdict[dev] < 0) {
    snprintf(g_msg, sizeof(g_msg), "libmi.so is built for sm_103a only");
    return MI_ERR_DEVICE;
  }
  return MI_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxHq = 4 * MI_MAX_HEADS;

// Shape checks shared by every call; fills the head list.
int check_common(const void* q, const void* k, int Hq, int Hkv, int N, int d,
                 const int32_t* heads, int n_heads, HeadList* hl) {
  if (!q || !k || !aligned16(q) || !aligned16(k)) return MI_ERR_ARG;
  if (d != kD) return MI_ERR_SHAPE;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq > kMaxHq) return MI_ERR_SHAPE;
  if (N < 1 || N > (1 << 21)) return MI_ERR_SHAPE;
  if (n_heads <= 0 || n_heads > MI_MAX_HEADS || n_heads > Hq) return MI_ERR_ARG;
  if (!heads && n_heads != Hq) return MI_ERR_ARG;
  bool seen[kMaxHq] = {};
  hl->n = n_heads;
  for (int i = 0; i < n_heads; ++i) {
    const int h = heads ? heads[i] : i;
    if (h < 0 || h >= Hq || seen[h]) return MI_ERR_ARG;
    seen[h] = true;
    hl->h[i] = static_cast<int16_t>(h);
  }
  return MI_OK;
}

// ---------------------------------------------------------- workspace ----

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  }
};

struct EstLayout {
  size_t status, part, stats, vsc, ssc, total;
  int NC;
};
EstLayout est_layout(int n_heads, int N) {
  EstLayout L;
  Carve c;
  L.NC = cdiv(N, kChunkKeys);
  L.status = c.take(256);
  L.part = c.take(sizeof(float) * (size_t)n_heads * kLastQ * L.NC * 2);
  L.stats = c.take(sizeof(float) * (size_t)n_heads * kLastQ * 2);
  L.vsc = c.take(sizeof(float) * (size_t)n_heads * N);
  L.ssc = c.take(sizeof(float) * (size_t)n_heads * N);
  L.total = c.off;
  return L;
}

struct VsLayout {
  size_t status, offbits, colbits, dbits, dfull, dlist, dcount, clist, ccount, kc, vc, total;
  int Nw, NT, NTw, Dw;
};
VsLayout vs_layout(int n_heads, int N) {
  VsLayout L;
  Carve c;
  L.NT = cdiv(N, kBN);
  L.Nw = 4 * L.NT;  // padded to whole 128-key tiles
  L.NTw = cdiv(L.NT, 32);
  L.Dw = L.Nw + 8;  // the windows' key-distance bits, x + 128 for x in [-127, N)
  L.status = c.take(256);
  L.offbits = c.take(sizeof(uint32_t) * (size_t)n_heads * L.Nw);
  L.colbits = c.take(sizeof(uint32_t) * (size_t)n_heads * L.Nw);
  L.dbits = c.take(sizeof(uint32_t) * (size_t)n_heads * L.Dw);
  L.dfull = c.take(sizeof(uint32_t) * (size_t)n_heads * L.NTw);
  L.dlist = c.take(sizeof(int) * (size_t)n_heads * L.NT);
  L.dcount = c.take(sizeof(int) * (size_t)n_heads);
  L.clist = c.take(sizeof(int) * (size_t)n_heads * MI_MAX_KV);
  L.ccount = c.take(sizeof(int) * (size_t)n_heads);
  L.kc = c.take(sizeof(uint16_t) * kD * (size_t)n_heads * MI_MAX_KV);
  L.vc = c.take(sizeof(uint16_t) * kD * (size_t)n_heads * MI_MAX_KV);
  L.total = c.off;
  return L;
}

struct BlockLayout {
  size_t status, qbar, kbar, total;
};
BlockLayout block_layout(int n_heads, int Hkv, int N) {
  BlockLayout L;
  Carve c;
  const int NB = cdiv(N, kBlk);
  L.status = c.take(256);
  L.qbar = c.take(sizeof(float) * (size_t)n_heads * NB * kD);
  L.kbar = c.take(sizeof(float) * (size_t)Hkv * NB * kD);
  L.total = c.off;
  return L;
}

// Multi-modal calls: grid estimation (lattice scores per sigma), grid attention
// (lattice columns, then a vertical-slash workspace), Q-boundary estimation and
// attention (modality ends and per-row-block modality bits, then the estimation
// or vertical-slash workspace).
struct MmLayout {
  size_t status, aux, ends, blk, sub, vsw, qp, kp, vp, op, lse1, lse2, total;
};
MmLayout mm_layout(int op, int n_heads, int N, int Hkv = 0) {
  MmLayout L;
  Carve c;
  L.status = c.take(256);
  L.aux = L.ends = L.blk = 0;
  if (op == MI_OP_GRID_ESTIMATE) {
    L.aux = c.take(sizeof(float) * 2 * (size_t)n_heads * MI_GRID_MAX_SIGMA);
    L.sub = c.take(est_layout(n_heads, N).total);
  } else if (op == MI_OP_GRID_ATTN) {
    L.aux = c.take(sizeof(int32_t) * (size_t)n_heads * MI_MAX_KV);
    L.sub = c.take(vs_layout(n_heads, N).total);
  } else if (op == MI_OP_BOUNDARY2D_ATTN) {
    // n_heads is Hq here: the permuted copy holds every q-head
    L.ends = 0;
    L.blk = c.take(sizeof(uint32_t) * 4 * (size_t)cdiv(N, kBM));              // modality bits (whole tiles)
    L.aux = c.take(sizeof(uint32_t) * (size_t)cdiv(N, kBM));                  // modalities per 128 tokens
    L.sub = c.take(est_layout(n_heads, N).total);                             // estimation
    L.vsw = c.take(vs_layout(n_heads, N).total);                              // vertical-slash passes
    L.qp = c.take(sizeof(uint16_t) * kD * (size_t)n_heads * N);               // permuted q, k, v, o
    L.kp = c.take(sizeof(uint16_t) * kD * (size_t)std::max(Hkv, 1) * N);
    L.vp = c.take(sizeof(uint16_t) * kD * (size_t)std::max(Hkv, 1) * N);
    L.op = c.take(sizeof(uint16_t) * kD * (size_t)n_heads * N);
    L.lse1 = c.take(sizeof(float) * (size_t)n_heads * N);                     // within-modality lse
    L.lse2 = c.take(sizeof(float) * (size_t)n_heads * N);                     // cross-modality lse
  } else {
    L.ends = c.take(sizeof(int) * MI_MAX_MODALITIES);
    L.blk = c.take(sizeof(uint32_t) * (size_t)cdiv(N, kBM));
    L.sub = c.take(op == MI_OP_QBOUNDARY_ESTIMATE ? est_layout(n_heads, N).total : vs_layout(n_heads, N).total);
  }
  L.total = c.off;
  return L;
}

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < need) return MI_ERR_WORKSPACE;
  return MI_OK;
}

int set_smem(const void* kernel, size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "cudaFuncSetAttribute");
}

// SMs of the current device, queried once per device.
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

int launched(const char* what) {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MI_OK : cuda_fail(e, what);
}

const float kScaleLog2 = 1.4426950408889634f / std::sqrt(static_cast<float>(kD));

// Launch a kernel as the programmatic dependent of the kernel before it in the
// stream (pdl.cuh): it may be scheduled while that one drains and waits for it
// on the device.
template <typename... P, typename... A>
int launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const char* what,
                     A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
  return e == cudaSuccess ? MI_OK : cuda_fail(e, what);
}

// Test-only fault injection (mi_debug_inject); normal operation: mode 0, 4 s waits.
std::atomic<int> g_fault_mode{MI_FAULT_NONE};
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

int zero_status(int* status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "cudaMemsetAsync");
}

// Shared by the four attention entry points: pattern-specific fields of `a` are set.
// Vertical-slash launches pass the listed heads' compacted column rows (kc, vc:
// [n_heads, MI_MAX_KV, 128] bf16) for the column tiles.
template <int PAT>
int run_attention(const void* q, const void* k, const void* v, int Hq, int Hkv, int N,
                  mi_bf16* out, float* lse, int* status, AttnArgs& a, cudaStream_t st,
                  const void* kc = nullptr, const void* vc = nullptr, int n_blocks = 0, int64_t ld = 0) {
  CUtensorMap mq, mk, mv, mkr, mvr;
  int rc;
  if (ld <= 0) ld = N;  // rows between heads (a sequence inside a longer buffer: that buffer's rows)
  if ((rc = make_map(&mq, q, Hq, N, kBM, ld)) || (rc = make_map(&mk, k, Hkv, N, kBlk, ld)) ||
      (rc = make_map(&mv, v, Hkv, N, kBlk, ld)))
    return rc;
  if (is_vs(PAT)) {  // column tiles
    if ((rc = make_map(&mkr, kc, a.heads.n, MI_MAX_KV, kBlk, MI_MAX_KV)) ||
        (rc = make_map(&mvr, vc, a.heads.n, MI_MAX_KV, kBlk, MI_MAX_KV)))
      return rc;
  } else {
    mkr = mk;
    mvr = mv;
  }
  a.q = reinterpret_cast<const __nv_bfloat16*>(q);
  a.N = N;
  a.ld = static_cast<int>(ld);
  a.group = Hq / Hkv;
  a.scale_log2 = kScaleLog2;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.skip_q_load = g_fault_mode.load() == MI_FAULT_SKIP_Q_LOAD ? 1 : 0;
  cudaError_t e = launch_attn<PAT>(mq, mk, mv, mkr, mvr, a, n_blocks > 0 ? n_blocks : cdiv(N, kBM), st);
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "attention kernel");
}

int attn_preamble(const void* q, const void* k, const void* v, int Hq, int Hkv, int N, int d,
                  const int32_t* heads, int n_heads, const void* out, AttnArgs* a) {
  int rc = check_device();
  if (rc) return rc;
  memset(a, 0, sizeof(*a));
  if ((rc = check_common(q, k, Hq, Hkv, N, d, heads, n_heads, &a->heads))) return rc;
  if (!v || !out || !aligned16(v) || !aligned16(out)) return MI_ERR_ARG;
  return MI_OK;
}

// Estimation of the listed heads (E1, E2, T1) into rows of ld_v / ld_s entries of
// v_idx / s_idx; ws is an est_layout(heads.n, N) workspace.
// row_end (device int, nullable): the query rows end there instead of at N.
int est_run(const void* q, const void* k, int Hq, int Hkv, int N, int64_t ld, const HeadList& heads,
            int k_v, int k_s, int32_t* v_idx, int ld_v, int32_t* s_idx, int ld_s, char* ws,
            int* status, cudaStream_t st, const int* row_end = nullptr) {
  EstArgs a;
  memset(&a, 0, sizeof(a));
  a.heads = heads;
  const int n_heads = heads.n;
  const EstLayout L = est_layout(n_heads, N);
  // pair up listed heads that share a KV head (two heads fill one 128-row UMMA)
  const int group = Hq / Hkv;
  int pending[kMaxHq];
  for (int g = 0; g < Hkv; ++g) pending[g] = -1;
  int np = 0;
  for (int i = 0; i < n_heads; ++i) {
    const int g = a.heads.h[i] / group;
    if (pending[g] < 0) {
      pending[g] = i;
    } else {
      a.pair_a[np] = static_cast<int16_t>(pending[g]);
      a.pair_b[np] = static_cast<int16_t>(i);
      ++np;
      pending[g] = -1;
    }
  }
  for (int g = 0; g < Hkv; ++g)
    if (pending[g] >= 0) {
      a.pair_a[np] = static_cast<int16_t>(pending[g]);
      a.pair_b[np] = -1;
      ++np;
    }
  a.N = N;
  a.group = group;
  a.n_pairs = np;
  a.NC = L.NC;
  a.scale_log2 = kScaleLog2;
  a.part = reinterpret_cast<float*>(ws + L.part);
  a.stats = reinterpret_cast<float*>(ws + L.stats);
  a.vsc = reinterpret_cast<float*>(ws + L.vsc);
  a.ssc = reinterpret_cast<float*>(ws + L.ssc);
  a.status = status;
  a.wait_limit_ns = kWaitLimitNs;
  a.row_end = row_end;
  a.chunk2 = est_chunk2(np, N, sm_count());

  static std::once_flag once;
  static int once_rc = MI_OK;
  std::call_once(once, [] {
    once_rc = set_smem(reinterpret_cast<const void*>(est_kernel<1>), kEstSmem1);
    if (once_rc == MI_OK) once_rc = set_smem(reinterpret_cast<const void*>(est_kernel<2>), kEstSmem2);
    if (once_rc == MI_OK) once_rc = set_smem(reinterpret_cast<const void*>(vs_topk_kernel), kTopkSmemBytes);
  });
  if (once_rc) return once_rc;

  int rc;
  CUtensorMap mq, mk;
  if ((rc = make_map(&mq, q, Hq, N, kLastQ, ld)) || (rc = make_map(&mk, k, Hkv, N, kBN, ld))) return rc;
  const dim3 grid(np, L.NC);
  est_kernel<1><<<grid, kEstThreads, kEstSmem1, st>>>(mq, mk, a);
  if ((rc = launched("estimation pass 1"))) return rc;
  // combine, pass 2 and the top-k each start while the kernel before them drains
  const float* part = a.part;
  if ((rc = launch_dependent(est_combine, dim3(cdiv(n_heads * kLastQ, 8)), dim3(256), 0, st, "estimation combine",
                             part, a.stats, L.NC, n_heads * kLastQ)))
    return rc;
  if ((rc = launch_dependent(est_kernel<2>, dim3(np, cdiv(N, a.chunk2)), dim3(kEstThreads), kEstSmem2, st,
                             "estimation pass 2", mq, mk, a)))
    return rc;
  if (ld_v > 0 || ld_s > 0) {
    const float *vsc = a.vsc, *ssc = a.ssc;
    // a cluster of two CTAs per (head, vertical | slash) row
    if ((rc = launch_dependent(vs_topk_kernel, dim3(2 * n_heads, 2), dim3(1024), kTopkSmemBytes, st, "top-k", vsc,
                               ssc, N, k_v, k_s, v_idx, s_idx, ld_v, ld_s)))
      return rc;
  }
  return MI_OK;
}

// Index build of the listed vertical-slash heads into a vs_layout workspace, and
// the structures it leaves in the attention arguments.
int vs_index_run(const VsLayout& L, char* ws, int n_heads, int N, const int32_t* v_idx, int k_v,
                 const int32_t* s_idx, int k_s, int expanded, int* status, cudaStream_t st, AttnArgs& a) {
  static std::once_flag once;
  static int once_rc = MI_OK;
  std::call_once(once, [] {
    once_rc = set_smem(reinterpret_cast<const void*>(vs_index_kernel), vs_index_smem(cdiv(1 << 21, kBN)));
  });
  if (once_rc) return once_rc;
  VsIndexArgs ia;
  ia.N = N;
  ia.k_v = k_v;
  ia.k_s = k_s;
  ia.Nw = L.Nw;
  ia.NT = L.NT;
  ia.NTw = L.NTw;
  ia.Dw = L.Dw;
  ia.expanded = expanded;
  ia.v_idx = v_idx;
  ia.s_idx = s_idx;
  ia.offbits = reinterpret_cast<uint32_t*>(ws + L.offbits);
  ia.colbits = reinterpret_cast<uint32_t*>(ws + L.colbits);
  ia.dbits = reinterpret_cast<uint32_t*>(ws + L.dbits);
  ia.dfull = reinterpret_cast<uint32_t*>(ws + L.dfull);
  ia.dlist = reinterpret_cast<int*>(ws + L.dlist);
  ia.dcount = reinterpret_cast<int*>(ws + L.dcount);
  ia.clist = reinterpret_cast<int*>(ws + L.clist);
  ia.ccount = reinterpret_cast<int*>(ws + L.ccount);
  ia.status = status;
  vs_index_kernel<<<n_heads, 512, vs_index_smem(L.NT), st>>>(ia);
  int rc;
  if ((rc = launched("vertical-slash index build"))) return rc;
  a.offbits = ia.offbits;
  a.colbits = ia.colbits;
  a.dbits = ia.dbits;
  a.dfull = ia.dfull;
  a.dlist = ia.dlist;
  a.dcount = ia.dcount;
  a.clist = ia.clist;
  a.ccount = ia.ccount;
  a.expand = expanded;
  a.Nw = L.Nw;
  a.NT = L.NT;
  a.NTw = L.NTw;
  a.Dw = L.Dw;
  return MI_OK;
}

// Vertical-slash attention of the listed heads (a.heads) with given indices: index
// build, column copy, attention.  vws is a vs_layout(a.heads.n, N) workspace; errors
// of the data go to `status`.  a's row filter (modality) and grid fields are kept.
int vs_attn_run(const void* q, const void* k, const void* v, int Hq, int Hkv, int N, AttnArgs& a,
                const int32_t* v_idx, int k_v, const int32_t* s_idx, int k_s, int expanded,
                mi_bf16* out, float* lse, char* vws, int* status, cudaStream_t st, int64_t ld = 0) {
  if (ld <= 0) ld = N;
  int rc;
  const int n_heads = a.heads.n;
  const VsLayout L = vs_layout(n_heads, N);
  char* ws = vws;
  if ((rc = vs_index_run(L, ws, n_heads, N, v_idx, k_v, s_idx, k_s, expanded, status, st, a))) return rc;
  __nv_bfloat16* kc = reinterpret_cast<__nv_bfloat16*>(ws + L.kc);
  __nv_bfloat16* vc = reinterpret_cast<__nv_bfloat16*>(ws + L.vc);
  vs_colgather_kernel<<<dim3(cdiv(std::min(k_v + kBN, MI_MAX_KV), 8), n_heads), 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(k), reinterpret_cast<const __nv_bfloat16*>(v), ld, Hq / Hkv,
      a.heads, a.clist, a.ccount, kc, vc);
  if ((rc = launched("vertical-slash column copy"))) return rc;
  return expanded ? run_attention<kPatVSExp>(q, k, v, Hq, Hkv, N, out, lse, status, a, st, kc, vc, 0, ld)
                  : run_attention<kPatVS>(q, k, v, Hq, Hkv, N, out, lse, status, a, st, kc, vc, 0, ld);
}

// ------------------------------------------------------------ layer calls ----

// The heads of a layer call grouped by pattern and budget.  Slots of one pattern
// are numbered group after group, so every group's rows are contiguous.
struct LayerPlan {
  int n_listed = 0, n_vs = 0, n_blk = 0, n_ash = 0;
  int KV = 0, KS = 0, TK = 0, vs_flags = 0;
  HeadList listed;                        // launch order: dense, VS, block, A-shape
  int n_vg = 0, vg_kv[MI_MAX_HEADS], vg_ks[MI_MAX_HEADS], vg_start[MI_MAX_HEADS + 1];
  int n_bg = 0, bg_tk[MI_MAX_HEADS], bg_start[MI_MAX_HEADS + 1];
  int16_t vs_head[MI_MAX_HEADS], blk_head[MI_MAX_HEADS];
  int ash[2 * MI_MAX_HEADS];
  int max_vg = 0;
};

// vs_as_dense: vertical-slash heads run dense (a sequence too short to estimate).
int layer_plan(const mi_head_cfg* cfg, int Hq, int N, bool vs_as_dense, LayerPlan* P) {
  if (!cfg) return MI_ERR_ARG;
  int n_dense = 0;
  int16_t dense_h[MI_MAX_HEADS];
  bool have_vs = false;
  for (int h = 0; h < Hq; ++h) {
    const mi_head_cfg& c = cfg[h];
    switch (c.pattern) {
      case MI_PAT_SKIP: continue;
      case MI_PAT_DENSE: break;
      case MI_PAT_VS:
        if (c.k_v < 0 || c.k_s < 0 || c.k_v > MI_MAX_KV) return MI_ERR_ARG;
        if (c.vs_flags & ~MI_VS_BLOCK_EXPANDED) return MI_ERR_UNIMPLEMENTED;
        if (have_vs && c.vs_flags != P->vs_flags) return MI_ERR_ARG;
        have_vs = true;
        P->vs_flags = c.vs_flags;
        break;
      case MI_PAT_BLOCK:
        if (c.topk < 1 || c.topk > MI_MAX_KV / 2) return MI_ERR_ARG;
        break;
      case MI_PAT_ASHAPE:
        if (c.n_init < 0 || c.window < 1) return MI_ERR_ARG;
        break;
      default: return MI_ERR_ARG;
    }
    if (P->n_listed == MI_MAX_HEADS) return MI_ERR_ARG;
    ++P->n_listed;
    if (c.pattern == MI_PAT_DENSE || (c.pattern == MI_PAT_VS && vs_as_dense))
      dense_h[n_dense++] = static_cast<int16_t>(h);
  }
  if (P->n_listed == 0) return MI_ERR_ARG;
  int n = 0;
  auto list = [&](int h) { P->listed.h[n++] = static_cast<int16_t>(h); };
  for (int i = 0; i < n_dense; ++i) list(dense_h[i]);
  // vertical-slash heads, grouped by (k_v, k_s) in order of first appearance
  bool done[kMaxHq] = {};
  for (int h = 0; h < Hq && !vs_as_dense; ++h) {
    if (cfg[h].pattern != MI_PAT_VS || done[h]) continue;
    const int kv = cfg[h].k_v, ks = cfg[h].k_s;
    P->vg_kv[P->n_vg] = kv;
    P->vg_ks[P->n_vg] = ks;
    P->vg_start[P->n_vg] = P->n_vs;
    for (int h2 = h; h2 < Hq; ++h2)
      if (cfg[h2].pattern == MI_PAT_VS && !done[h2] && cfg[h2].k_v == kv && cfg[h2].k_s == ks) {
        done[h2] = true;
        P->vs_head[P->n_vs] = static_cast<int16_t>(h2);
        list(h2);
        ++P->n_vs;
      }
    P->max_vg = std::max(P->max_vg, P->n_vs - P->vg_start[P->n_vg]);
    P->KV = std::max(P->KV, kv);
    P->KS = std::max(P->KS, ks);
    ++P->n_vg;
  }
  P->vg_start[P->n_vg] = P->n_vs;
  for (int h = 0; h < Hq; ++h) {
    if (cfg[h].pattern != MI_PAT_BLOCK || done[h]) continue;
    const int tk = cfg[h].topk;
    P->bg_tk[P->n_bg] = tk;
    P->bg_start[P->n_bg] = P->n_blk;
    for (int h2 = h; h2 < Hq; ++h2)
      if (cfg[h2].pattern == MI_PAT_BLOCK && !done[h2] && cfg[h2].topk == tk) {
        done[h2] = true;
        P->blk_head[P->n_blk] = static_cast<int16_t>(h2);
        list(h2);
        ++P->n_blk;
      }
    P->TK = std::max(P->TK, tk);
    ++P->n_bg;
  }
  P->bg_start[P->n_bg] = P->n_blk;
  for (int h = 0; h < Hq; ++h) {
    if (cfg[h].pattern != MI_PAT_ASHAPE) continue;
    P->ash[2 * P->n_ash] = std::min(cfg[h].n_init, N);
    P->ash[2 * P->n_ash + 1] = std::min(cfg[h].window, N);
    list(h);
    ++P->n_ash;
  }
  P->listed.n = n;
  return MI_OK;
}

struct LayerLayout {
  size_t status, est, vs, vidx, sidx, blk, blkidx, total;
};
LayerLayout layer_layout(const LayerPlan& P, int Hkv, int N) {
  LayerLayout L;
  Carve c;
  L.status = c.take(256);
  L.est = c.take(P.n_vs ? est_layout(P.max_vg, N).total : 0);
  L.vs = c.take(P.n_vs ? vs_layout(P.n_vs, N).total : 0);
  L.vidx = c.take(sizeof(int32_t) * (size_t)P.n_vs * std::max(P.KV, 1));
  L.sidx = c.take(sizeof(int32_t) * (size_t)P.n_vs * std::max(P.KS, 1));
  L.blk = c.take(P.n_blk ? block_layout(P.n_blk, Hkv, N).total : 0);
  L.blkidx = c.take(sizeof(int32_t) * (size_t)P.n_blk * cdiv(N, kBlk) * std::max(P.TK, 1));
  L.total = c.off;
  return L;
}

// One layer over one sequence: q, k, v, out (and lse) point at the sequence's first
// row, consecutive heads `ld` rows apart; ws / L / status from the caller.
int layer_run(const void* q, const void* k, const void* v, int Hq, int Hkv, int N, int64_t ld,
              const LayerPlan& P, mi_bf16* out, float* lse, char* ws, const LayerLayout& L,
              int* status, cudaStream_t st) {
  int rc;
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.heads = P.listed;
  const int group = Hq / Hkv;
  // vertical-slash heads: estimation per budget group, one index build
  __nv_bfloat16 *kc = nullptr, *vc = nullptr;  // their compacted column rows
  int32_t* vidx = reinterpret_cast<int32_t*>(ws + L.vidx);
  int32_t* sidx = reinterpret_cast<int32_t*>(ws + L.sidx);
  if (P.n_vs) {
    for (int gi = 0; gi < P.n_vg; ++gi) {
      HeadList hl;
      hl.n = P.vg_start[gi + 1] - P.vg_start[gi];
      for (int i = 0; i < hl.n; ++i) hl.h[i] = P.vs_head[P.vg_start[gi] + i];
      const size_t r0 = P.vg_start[gi];
      if ((rc = est_run(q, k, Hq, Hkv, N, ld, hl, P.vg_kv[gi], P.vg_ks[gi], vidx + r0 * P.KV, P.KV,
                        sidx + r0 * P.KS, P.KS, ws + L.est, status, st)))
        return rc;
    }
    const VsLayout V = vs_layout(P.n_vs, N);
    char* vw = ws + L.vs;
    if ((rc = vs_index_run(V, vw, P.n_vs, N, vidx, P.KV, sidx, P.KS, (P.vs_flags & MI_VS_BLOCK_EXPANDED) ? 1 : 0,
                           status, st, a)))
      return rc;
    HeadList hv;
    hv.n = P.n_vs;
    for (int i = 0; i < P.n_vs; ++i) hv.h[i] = P.vs_head[i];
    kc = reinterpret_cast<__nv_bfloat16*>(vw + V.kc);
    vc = reinterpret_cast<__nv_bfloat16*>(vw + V.vc);
    vs_colgather_kernel<<<dim3(cdiv(std::min(P.KV + kBN, MI_MAX_KV), 8), P.n_vs), 256, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(k), reinterpret_cast<const __nv_bfloat16*>(v), ld, group, hv,
        a.clist, a.ccount, kc, vc);
    if ((rc = launched("vertical-slash column copy"))) return rc;
  }
  // block-sparse heads: pooling once, selection per top-k group
  if (P.n_blk) {
    const BlockLayout BL = block_layout(P.n_blk, Hkv, N);
    char* bw = ws + L.blk;
    float* qbar = reinterpret_cast<float*>(bw + BL.qbar);
    float* kbar = reinterpret_cast<float*>(bw + BL.kbar);
    int32_t* blk = reinterpret_cast<int32_t*>(ws + L.blkidx);
    const int NB = cdiv(N, kBlk);
    HeadList hb;
    hb.n = P.n_blk;
    for (int i = 0; i < P.n_blk; ++i) hb.h[i] = P.blk_head[i];
    const int wq = P.n_blk * NB, wk = Hkv * NB;
    block_pool_kernel<<<cdiv(wq, 8), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(q), N, ld,
                                                   P.n_blk, NB, hb, 1, qbar);
    if ((rc = launched("block pooling (q)"))) return rc;
    block_pool_kernel<<<cdiv(wk, 8), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(k), N, ld,
                                                   Hkv, NB, hb, 0, kbar);
    if ((rc = launched("block pooling (k)"))) return rc;
    if ((rc = set_smem(reinterpret_cast<const void*>(block_select_kernel), 160 * 1024))) return rc;
    for (int gi = 0; gi < P.n_bg; ++gi) {
      HeadList hl;
      const int s0 = P.bg_start[gi];
      hl.n = P.bg_start[gi + 1] - s0;
      for (int i = 0; i < hl.n; ++i) hl.h[i] = P.blk_head[s0 + i];
      const int R = block_select_rows(NB, 160 * 1024);
      block_select_kernel<<<dim3(cdiv(NB, R), hl.n), 256, sizeof(float) * NB * R, st>>>(
          qbar + (size_t)s0 * NB * kD, kbar, NB, group, hl, P.bg_tk[gi], P.TK, R,
          blk + (size_t)s0 * NB * P.TK);
      if ((rc = launched("block selection"))) return rc;
    }
    a.blk_idx = blk;
    a.topk = P.TK;
  }
  // A-shape heads: per-head sizes, passed in the kernel arguments
  a.ash_n = P.n_ash;
  for (int i = 0; i < 2 * P.n_ash; ++i) a.ash_pairs[i] = P.ash[i];
  // listed order is dense, vertical-slash, block-sparse, A-shape
  {
    const int n_dense = P.listed.n - P.n_vs - P.n_blk - P.n_ash;
    a.layer_base[kPatDense] = 0;
    a.layer_base[kPatVS] = n_dense;
    a.layer_base[kPatBlock] = n_dense + P.n_vs;
    a.layer_base[kPatAShape] = n_dense + P.n_vs + P.n_blk;
    a.layer_base[4] = P.listed.n;
  }
  // the attention of every listed head in one launch
  CUtensorMap mq, mk, mv, mkr, mvr;
  if ((rc = make_map(&mq, q, Hq, N, kBM, ld)) || (rc = make_map(&mk, k, Hkv, N, kBlk, ld)) ||
      (rc = make_map(&mv, v, Hkv, N, kBlk, ld)))
    return rc;
  if (P.n_vs) {  // the vertical-slash heads' column tiles
    if ((rc = make_map(&mkr, kc, P.n_vs, MI_MAX_KV, kBlk, MI_MAX_KV)) ||
        (rc = make_map(&mvr, vc, P.n_vs, MI_MAX_KV, kBlk, MI_MAX_KV)))
      return rc;
  } else {
    mkr = mk;
    mvr = mv;
  }
  a.N = N;
  a.ld = static_cast<int>(ld);
  a.group = group;
  a.scale_log2 = kScaleLog2;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.skip_q_load = g_fault_mode.load() == MI_FAULT_SKIP_Q_LOAD ? 1 : 0;
  cudaError_t e = launch_attn_layer(mq, mk, mv, mkr, mvr, a, cdiv(N, kBM), st);
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "layer attention kernel");
}

int check_modality(const int32_t* modality, int n_mod) {
  if (!modality || n_mod < 1 || n_mod > MI_MAX_MODALITIES) return MI_ERR_ARG;
  return MI_OK;
}

// Modality ends and per-row-block modality bits into the workspace (zeroed first).
int modality_scan(const int32_t* modality, int N, int n_mod, char* ws, const MmLayout& L, int* status,
                  cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws + L.ends, 0, sizeof(int) * MI_MAX_MODALITIES, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.blk, 0, sizeof(uint32_t) * (size_t)cdiv(N, kBM), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  modality_scan_kernel<<<cdiv(N, 256), 256, 0, st>>>(modality, N, n_mod, reinterpret_cast<int*>(ws + L.ends),
                                                     reinterpret_cast<uint32_t*>(ws + L.blk), status);
  return launched("modality scan");
}

}  // namespace

// ====================================================================== ABI ==

extern "C" {

size_t mi_workspace_bytes(int op, int n_heads, int Hkv, int N, int k_v, int k_s, int topk) {
  (void)k_v;
  (void)k_s;
  (void)topk;
  if (n_heads <= 0 || N <= 0) return 0;
  switch (op) {
    case MI_OP_VS_ESTIMATE: return est_layout(n_heads, N).total;
    case MI_OP_VS_SPARSE_ATTN: return vs_layout(n_heads, N).total;
    case MI_OP_BLOCK_SPARSE_ATTN: return Hkv > 0 ? block_layout(n_heads, Hkv, N).total : 0;
    case MI_OP_ASHAPE_ATTN:
    case MI_OP_DENSE_CAUSAL_ATTN: return 256;
    case MI_OP_GRID_ESTIMATE:
    case MI_OP_GRID_ATTN:
    case MI_OP_QBOUNDARY_ESTIMATE:
    case MI_OP_QBOUNDARY_ATTN: return mm_layout(op, n_heads, N).total;
    case MI_OP_BOUNDARY2D_ATTN: return Hkv > 0 ? mm_layout(op, n_heads, N, Hkv).total : 0;
    default: return 0;
  }
}

int mi_vs_estimate(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                   const int32_t* heads, int n_heads, int last_q, int k_v, int k_s,
                   int32_t* v_idx, int32_t* s_idx, void* workspace, size_t ws_bytes,
                   mi_stream_t stream) {
  int rc = check_device();
  if (rc) return rc;
  HeadList hl;
  if ((rc = check_common(q, k, Hq, Hkv, N, d, heads, n_heads, &hl))) return rc;
  if (last_q != kLastQ || N < kLastQ) return MI_ERR_SHAPE;
  if (k_v < 0 || k_s < 0) return MI_ERR_ARG;
  if ((k_v > 0 && !v_idx) || (k_s > 0 && !s_idx)) return MI_ERR_ARG;
  const EstLayout L = est_layout(n_heads, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  return est_run(q, k, Hq, Hkv, N, N, hl, k_v, k_s, v_idx, k_v, s_idx, k_s, ws, status, st);
}

int mi_vs_sparse_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                      int N, int d, const int32_t* heads, int n_heads, const int32_t* v_idx,
                      int k_v, const int32_t* s_idx, int k_s, int flags, mi_bf16* out, float* lse,
                      void* workspace, size_t ws_bytes, mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, heads, n_heads, out, &a);
  if (rc) return rc;
  if (flags & ~MI_VS_BLOCK_EXPANDED) return MI_ERR_UNIMPLEMENTED;
  const int expanded = (flags & MI_VS_BLOCK_EXPANDED) ? 1 : 0;
  if (k_v < 0 || k_s < 0 || k_v > MI_MAX_KV) return MI_ERR_ARG;
  if ((k_v > 0 && !v_idx) || (k_s > 0 && !s_idx)) return MI_ERR_ARG;
  const VsLayout L = vs_layout(n_heads, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;

  return vs_attn_run(q, k, v, Hq, Hkv, N, a, v_idx, k_v, s_idx, k_s, expanded, out, lse, ws, status, st);
}

int mi_block_sparse_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                         int N, int d, const int32_t* heads, int n_heads, int block, int topk,
                         int32_t* blk_idx, int flags, mi_bf16* out, float* lse, void* workspace,
                         size_t ws_bytes, mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, heads, n_heads, out, &a);
  if (rc) return rc;
  if (block != kBlk) return MI_ERR_SHAPE;
  if (topk < 1 || topk > MI_MAX_KV / 2 || !blk_idx) return MI_ERR_ARG;
  if (flags & ~MI_IDX_GIVEN) return MI_ERR_UNIMPLEMENTED;
  const BlockLayout L = block_layout(n_heads, Hkv, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  const int NB = cdiv(N, kBlk);
  if (!(flags & MI_IDX_GIVEN)) {
    float* qbar = reinterpret_cast<float*>(ws + L.qbar);
    float* kbar = reinterpret_cast<float*>(ws + L.kbar);
    const int wq = n_heads * NB, wk = Hkv * NB;
    block_pool_kernel<<<cdiv(wq, 8), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(q), N, N,
                                                   n_heads, NB, a.heads, 1, qbar);
    if ((rc = launched("block pooling (q)"))) return rc;
    block_pool_kernel<<<cdiv(wk, 8), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(k), N, N,
                                                   Hkv, NB, a.heads, 0, kbar);
    if ((rc = launched("block pooling (k)"))) return rc;
    static std::once_flag once;
    static int once_rc = MI_OK;
    std::call_once(once, [] {
      once_rc = set_smem(reinterpret_cast<const void*>(block_select_kernel), 160 * 1024);
    });
    if (once_rc) return once_rc;
    const int R = block_select_rows(NB, 160 * 1024);
    block_select_kernel<<<dim3(cdiv(NB, R), n_heads), 256, sizeof(float) * NB * R, st>>>(
        qbar, kbar, NB, Hq / Hkv, a.heads, topk, topk, R, blk_idx);
    if ((rc = launched("block selection"))) return rc;
  } else {
    const int rows = n_heads * NB;
    block_validate_kernel<<<cdiv(rows, 256), 256, 0, st>>>(blk_idx, NB, topk, rows, status);
    if ((rc = launched("block index validation"))) return rc;
  }
  a.blk_idx = blk_idx;
  a.topk = topk;
  return run_attention<kPatBlock>(q, k, v, Hq, Hkv, N, out, lse, status, a, st);
}

int mi_ashape_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N,
                   int d, const int32_t* heads, int n_heads, int n_init, int window, mi_bf16* out,
                   float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, heads, n_heads, out, &a);
  if (rc) return rc;
  if (n_init < 0 || window < 1) return MI_ERR_ARG;
  if ((rc = check_ws(workspace, ws_bytes, 256))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  if ((rc = zero_status(status, st))) return rc;
  a.n_init = n_init < N ? n_init : N;
  a.window = window < N ? window : N;
  return run_attention<kPatAShape>(q, k, v, Hq, Hkv, N, out, lse, status, a, st);
}

int mi_dense_causal_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                         int N, int d, const int32_t* heads, int n_heads, mi_bf16* out,
                         float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, heads, n_heads, out, &a);
  if (rc) return rc;
  if ((rc = check_ws(workspace, ws_bytes, 256))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  if ((rc = zero_status(status, st))) return rc;
  return run_attention<kPatDense>(q, k, v, Hq, Hkv, N, out, lse, status, a, st);
}

size_t mi_layer_workspace_bytes(int Hq, int Hkv, int N, const mi_head_cfg* cfg) {
  if (Hq <= 0 || Hkv <= 0 || N <= 0 || Hq > kMaxHq || Hq % Hkv != 0) return 0;
  LayerPlan P;
  if (layer_plan(cfg, Hq, N, false, &P)) return 0;
  return layer_layout(P, Hkv, N).total;
}

int mi_layer_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N,
                  int d, const mi_head_cfg* cfg, mi_bf16* out, float* lse, void* workspace,
                  size_t ws_bytes, mi_stream_t stream) {
  int rc = check_device();
  if (rc) return rc;
  LayerPlan P;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return MI_ERR_ARG;
  if (d != kD) return MI_ERR_SHAPE;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq > kMaxHq) return MI_ERR_SHAPE;
  if (N < 1 || N > (1 << 21)) return MI_ERR_SHAPE;
  if ((rc = layer_plan(cfg, Hq, N, false, &P))) return rc;
  if (P.n_vs && N < kLastQ) return MI_ERR_SHAPE;
  const LayerLayout L = layer_layout(P, Hkv, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  return layer_run(q, k, v, Hq, Hkv, N, N, P, out, lse, ws, L, status, st);
}

// Validates cu_seqlens and returns the longest sequence (0 on error).
static int varlen_check(const int32_t* cu, int n_seqs, int total, int* n_max_long, int* n_max_short) {
  if (!cu || n_seqs < 1 || cu[0] != 0 || cu[n_seqs] != total || total < 1) return 0;
  int nmax = 0;
  *n_max_long = 0;
  *n_max_short = 0;
  for (int b = 0; b < n_seqs; ++b) {
    const int n = cu[b + 1] - cu[b];
    if (n < 0 || n > (1 << 21)) return 0;
    nmax = std::max(nmax, n);
    if (n >= kLastQ) *n_max_long = std::max(*n_max_long, n);
    else *n_max_short = std::max(*n_max_short, n);
  }
  return nmax;
}

size_t mi_layer_workspace_bytes_varlen(int Hq, int Hkv, const int32_t* cu_seqlens, int n_seqs,
                                       const mi_head_cfg* cfg) {
  if (Hq <= 0 || Hkv <= 0 || Hq > kMaxHq || Hq % Hkv != 0 || !cu_seqlens || n_seqs < 1) return 0;
  int nl, ns;
  if (!varlen_check(cu_seqlens, n_seqs, cu_seqlens[n_seqs], &nl, &ns)) return 0;
  LayerPlan Pl, Ps;
  size_t need = 0;
  if (nl) {
    if (layer_plan(cfg, Hq, nl, false, &Pl)) return 0;
    need = std::max(need, layer_layout(Pl, Hkv, nl).total);
  }
  if (ns) {
    if (layer_plan(cfg, Hq, ns, true, &Ps)) return 0;
    need = std::max(need, layer_layout(Ps, Hkv, ns).total);
  }
  return need;
}

int mi_layer_attn_varlen(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv,
                         int total, int d, const int32_t* cu_seqlens, int n_seqs,
                         const mi_head_cfg* cfg, mi_bf16* out, float* lse, void* workspace,
                         size_t ws_bytes, mi_stream_t stream) {
  int rc = check_device();
  if (rc) return rc;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return MI_ERR_ARG;
  if (d != kD) return MI_ERR_SHAPE;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq > kMaxHq) return MI_ERR_SHAPE;
  int nl, ns;
  if (!cu_seqlens || n_seqs < 1 || !varlen_check(cu_seqlens, n_seqs, total, &nl, &ns)) return MI_ERR_ARG;
  LayerPlan Pl, Ps;
  size_t need = 0;
  if (nl) {
    if ((rc = layer_plan(cfg, Hq, nl, false, &Pl))) return rc;
    need = std::max(need, layer_layout(Pl, Hkv, nl).total);
  }
  if (ns) {
    if ((rc = layer_plan(cfg, Hq, ns, true, &Ps))) return rc;
    need = std::max(need, layer_layout(Ps, Hkv, ns).total);
  }
  if ((rc = check_ws(workspace, ws_bytes, need))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);  // offset 0 of every layer layout
  if ((rc = zero_status(status, st))) return rc;
  for (int b = 0; b < n_seqs; ++b) {
    const int n = cu_seqlens[b + 1] - cu_seqlens[b];
    if (n == 0) continue;
    const LayerPlan& P = (n >= kLastQ) ? Pl : Ps;
    const LayerLayout L = layer_layout(P, Hkv, n);
    const size_t row = static_cast<size_t>(cu_seqlens[b]);
    if ((rc = layer_run(q + row * kD, k + row * kD, v + row * kD, Hq, Hkv, n, total, P,
                        out + row * kD, lse ? lse + row : nullptr, ws, L, status, st)))
      return rc;
  }
  return MI_OK;
}

int mi_debug_inject(int mode, uint64_t wait_limit_ns) {
  if (mode == MI_FAULT_NONE) {
    g_fault_mode.store(MI_FAULT_NONE);
    g_wait_limit_ns.store(kWaitLimitNs);
    return MI_OK;
  }
  if (mode != MI_FAULT_SKIP_Q_LOAD || wait_limit_ns == 0 || wait_limit_ns > 10000000000ull)
    return MI_ERR_ARG;
  g_wait_limit_ns.store(wait_limit_ns);
  g_fault_mode.store(mode);
  return MI_OK;
}

// ---------------------------------------------------- multi-modal heads ----

int mi_grid_estimate(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                     const int32_t* heads, int n_heads, int last_q, int sigma_min, int sigma_max,
                     int32_t* grid, void* workspace, size_t ws_bytes, mi_stream_t stream) {
  int rc = check_device();
  if (rc) return rc;
  HeadList hl;
  if ((rc = check_common(q, k, Hq, Hkv, N, d, heads, n_heads, &hl))) return rc;
  if (last_q != kLastQ || N < kLastQ) return MI_ERR_SHAPE;
  if (!grid || sigma_min < 1 || sigma_max < sigma_min || sigma_max > N ||
      sigma_max - sigma_min + 1 > MI_GRID_MAX_SIGMA)
    return MI_ERR_ARG;
  const MmLayout L = mm_layout(MI_OP_GRID_ESTIMATE, n_heads, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  // the vertical scores of the last 64 queries (no top-k), then the lattice fit
  if ((rc = est_run(q, k, Hq, Hkv, N, N, hl, 0, 0, nullptr, 0, nullptr, 0, ws + L.sub, status, st))) return rc;
  const EstLayout E = est_layout(n_heads, N);
  const float* vsc = reinterpret_cast<const float*>(ws + L.sub + E.vsc);
  float2* best = reinterpret_cast<float2*>(ws + L.aux);
  const int n_sigma = sigma_max - sigma_min + 1;
  grid_fit_kernel<<<dim3(n_sigma, n_heads), kFitThreads, 0, st>>>(vsc, N, sigma_min, n_sigma,
                                                                 static_cast<float>(kLastQ), best);
  if ((rc = launched("grid lattice scores"))) return rc;
  grid_pick_kernel<<<cdiv(n_heads, 128), 128, 0, st>>>(best, n_heads, sigma_min, n_sigma, grid);
  return launched("grid lattice choice");
}

int mi_grid_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N, int d,
                 const int32_t* heads, int n_heads, const int32_t* grid, int sigma_min, mi_bf16* out,
                 float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, heads, n_heads, out, &a);
  if (rc) return rc;
  if (!grid || sigma_min < 1 || sigma_min < cdiv(N, MI_MAX_KV)) return MI_ERR_ARG;
  const MmLayout L = mm_layout(MI_OP_GRID_ATTN, n_heads, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  // vertical lines: the lattice columns through the vertical-slash engine (no
  // diagonals), with the first block and the own block; every row is written
  int32_t* vidx = reinterpret_cast<int32_t*>(ws + L.aux);
  grid_lattice_kernel<<<n_heads, 256, 0, st>>>(grid, N, sigma_min, MI_MAX_KV, vidx, status);
  if ((rc = launched("grid lattice columns"))) return rc;
  AttnArgs base = a;
  if ((rc = vs_attn_run(q, k, v, Hq, Hkv, N, a, vidx, MI_MAX_KV, nullptr, 0, 0, out, lse, ws + L.sub, status, st)))
    return rc;
  // horizontal lines: the lattice rows, gathered 128 at a time, dense and causal;
  // they overwrite those rows (same stream, after the pass above)
  base.grid = grid;
  base.grid_sigma_min = sigma_min;
  return run_attention<kPatRows>(q, k, v, Hq, Hkv, N, out, lse, status, base, st, nullptr, nullptr,
                                 cdiv(cdiv(N, sigma_min), kBM));
}


int mi_qboundary_estimate(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N, int d,
                          const int32_t* heads, int n_heads, const int32_t* modality, int n_mod,
                          int last_q, int k_v, int k_s, int32_t* v_idx, int32_t* s_idx, void* workspace,
                          size_t ws_bytes, mi_stream_t stream) {
  int rc = check_device();
  if (rc) return rc;
  HeadList hl;
  if ((rc = check_common(q, k, Hq, Hkv, N, d, heads, n_heads, &hl))) return rc;
  if (last_q != kLastQ || N < kLastQ) return MI_ERR_SHAPE;
  if ((rc = check_modality(modality, n_mod))) return rc;
  if (k_v < 0 || k_s < 0) return MI_ERR_ARG;
  if ((k_v > 0 && !v_idx) || (k_s > 0 && !s_idx)) return MI_ERR_ARG;
  const MmLayout L = mm_layout(MI_OP_QBOUNDARY_ESTIMATE, n_heads, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  if ((rc = modality_scan(modality, N, n_mod, ws, L, status, st))) return rc;
  const int* ends = reinterpret_cast<const int*>(ws + L.ends);
  for (int m = 0; m < n_mod; ++m) {  // one estimation per modality, its window ending at its last token
    if ((rc = est_run(q, k, Hq, Hkv, N, N, hl, k_v, k_s, v_idx + (size_t)m * n_heads * k_v, k_v,
                      s_idx + (size_t)m * n_heads * k_s, k_s, ws + L.sub, status, st, ends + m)))
      return rc;
  }
  return MI_OK;
}

int mi_qboundary_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N, int d,
                      const int32_t* heads, int n_heads, const int32_t* modality, int n_mod,
                      const int32_t* v_idx, int k_v, const int32_t* s_idx, int k_s, mi_bf16* out,
                      float* lse, void* workspace, size_t ws_bytes, mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, heads, n_heads, out, &a);
  if (rc) return rc;
  if ((rc = check_modality(modality, n_mod))) return rc;
  if (k_v < 0 || k_s < 0 || k_v > MI_MAX_KV) return MI_ERR_ARG;
  if ((k_v > 0 && !v_idx) || (k_s > 0 && !s_idx)) return MI_ERR_ARG;
  const MmLayout L = mm_layout(MI_OP_QBOUNDARY_ATTN, n_heads, N);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  if ((rc = modality_scan(modality, N, n_mod, ws, L, status, st))) return rc;
  for (int m = 0; m < n_mod; ++m) {  // each modality's rows with its own index sets
    AttnArgs am = a;
    am.modality = modality;
    am.blk_mods = reinterpret_cast<const uint32_t*>(ws + L.blk);
    am.row_mod = m;
    if ((rc = vs_attn_run(q, k, v, Hq, Hkv, N, am, v_idx ? v_idx + (size_t)m * n_heads * k_v : nullptr, k_v,
                          s_idx ? s_idx + (size_t)m * n_heads * k_s : nullptr, k_s, 0, out, lse, ws + L.sub,
                          status, st)))
      return rc;
  }
  return MI_OK;
}

int mi_boundary2d_attn(const mi_bf16* q, const mi_bf16* k, const mi_bf16* v, int Hq, int Hkv, int N, int d,
                       const int32_t* runs, int n_runs, int k_v, int k_s, int32_t* v_idx, int32_t* s_idx,
                       int flags, mi_bf16* out, float* lse, void* workspace, size_t ws_bytes,
                       mi_stream_t stream) {
  AttnArgs a;
  int rc = attn_preamble(q, k, v, Hq, Hkv, N, d, nullptr, Hq, out, &a);
  if (rc) return rc;
  if (flags & ~MI_IDX_GIVEN) return MI_ERR_UNIMPLEMENTED;
  if (!runs || n_runs < 1 || n_runs > MI_MAX_RUNS) return MI_ERR_ARG;
  if (k_v < 0 || k_s < 0 || k_v > MI_MAX_KV) return MI_ERR_ARG;
  if ((k_v > 0 && !v_idx) || (k_s > 0 && !s_idx)) return MI_ERR_ARG;
  // the runs: original starts, and permuted starts (modality 0's tokens first)
  RunTable rt;
  rt.n = n_runs;
  int seg[2] = {0, 0};
  int64_t total = 0;
  for (int u = 0; u < n_runs; ++u) {
    const int m = runs[2 * u], len = runs[2 * u + 1];
    if ((m != 0 && m != 1) || len < 1) return MI_ERR_ARG;
    rt.start[u] = static_cast<int>(total);
    rt.len[u] = len;
    rt.mod[u] = m;
    total += len;
    if (total > N) return MI_ERR_ARG;
    seg[m] += len;
  }
  if (total != N) return MI_ERR_ARG;
  {
    int at[2] = {0, seg[0]};
    for (int u = 0; u < n_runs; ++u) {
      rt.pstart[u] = at[rt.mod[u]];
      at[rt.mod[u]] += rt.len[u];
    }
  }
  const MmLayout L = mm_layout(MI_OP_BOUNDARY2D_ATTN, Hq, N, Hkv);
  if ((rc = check_ws(workspace, ws_bytes, L.total))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  if ((rc = zero_status(status, st))) return rc;
  uint32_t* modbits = reinterpret_cast<uint32_t*>(ws + L.blk);
  uint32_t* mods128 = reinterpret_cast<uint32_t*>(ws + L.aux);
  cudaError_t e = cudaMemsetAsync(modbits, 0, sizeof(uint32_t) * 4 * (size_t)cdiv(N, kBM), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(mods128, 0, sizeof(uint32_t) * (size_t)cdiv(N, kBM), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  boundary_bits_kernel<<<cdiv(N, 256), 256, 0, st>>>(N, rt, modbits, mods128);
  if ((rc = launched("modality bits"))) return rc;
  __nv_bfloat16* qp = reinterpret_cast<__nv_bfloat16*>(ws + L.qp);
  __nv_bfloat16* kp = reinterpret_cast<__nv_bfloat16*>(ws + L.kp);
  __nv_bfloat16* vp = reinterpret_cast<__nv_bfloat16*>(ws + L.vp);
  __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(ws + L.op);
  float* lse1 = reinterpret_cast<float*>(ws + L.lse1);
  float* lse2 = reinterpret_cast<float*>(ws + L.lse2);
  const int64_t rows = (int64_t)(Hq + 2 * Hkv) * N;
  boundary_gather_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const __nv_bfloat16*>(k),
      reinterpret_cast<const __nv_bfloat16*>(v), Hq, Hkv, N, rt, qp, kp, vp);
  if ((rc = launched("modality permutation"))) return rc;
  // each modality's sub-sequence as a vertical-slash head of its own (rows N apart);
  // one too short to estimate (fewer than 64 tokens) is dense
  for (int m = 0; m < 2; ++m) {
    const int n_m = seg[m], off = m ? seg[0] : 0;
    if (n_m == 0) continue;
    const size_t eo = (size_t)off * kD;
    AttnArgs am = a;
    int32_t* vm = v_idx ? v_idx + (size_t)m * Hq * k_v : nullptr;
    int32_t* sm = s_idx ? s_idx + (size_t)m * Hq * k_s : nullptr;
    if (n_m >= kLastQ) {
      if (!(flags & MI_IDX_GIVEN) &&
          (rc = est_run(qp + eo, kp + eo, Hq, Hkv, n_m, N, a.heads, k_v, k_s, vm, k_v, sm, k_s, ws + L.sub,
                        status, st)))
        return rc;
      if ((rc = vs_attn_run(qp + eo, kp + eo, vp + eo, Hq, Hkv, n_m, am, vm, k_v, sm, k_s, 0,
                            reinterpret_cast<mi_bf16*>(op + eo), lse1 + off, ws + L.vsw, status, st, N)))
        return rc;
    } else {
      if ((rc = run_attention<kPatDense>(qp + eo, kp + eo, vp + eo, Hq, Hkv, n_m,
                                         reinterpret_cast<mi_bf16*>(op + eo), lse1 + off, status, am, st,
                                         nullptr, nullptr, 0, N)))
        return rc;
    }
  }
  // the cross-modality pairs in original positions, into out / lse2
  AttnArgs ax = a;
  ax.modbits = modbits;
  ax.mods128 = mods128;
  if ((rc = run_attention<kPatCross>(q, k, v, Hq, Hkv, N, out, lse2, status, ax, st))) return rc;
  const int64_t mrows = (int64_t)Hq * N;
  boundary_merge_kernel<<<static_cast<unsigned>((mrows + 7) / 8), 256, 0, st>>>(
      N, rt, a.heads, op, lse1, lse2, reinterpret_cast<__nv_bfloat16*>(out), lse);
  return launched("2D-boundary merge");
}

int mi_read_status(const void* workspace, mi_stream_t stream) {
  if (!workspace) return MI_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  return v;
}

const char* mi_strerror(int code) {
  switch (code) {
    case MI_OK: return "success";
    case MI_ERR_ARG: return "invalid argument (null/misaligned pointer, head list or budget)";
    case MI_ERR_SHAPE:
      return "unsupported shape (d must be 128, N a multiple of 64 in [64, 2^21], Hq % Hkv == 0, "
             "last_q 64, block 64)";
    case MI_ERR_WORKSPACE: return "workspace missing, not 256-byte aligned or too small";
    case MI_ERR_CUDA: return g_msg[0] ? g_msg : "CUDA error";
    case MI_ERR_INDEX:
      return "index out of range, not strictly ascending, or a value after -1 padding";
    case MI_ERR_TIMEOUT: return "a bounded pipeline wait in a kernel expired";
    case MI_ERR_UNIMPLEMENTED: return "option not supported by this build";
    case MI_ERR_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
    default: return "unknown error code";
  }
}

}  // extern "C"
