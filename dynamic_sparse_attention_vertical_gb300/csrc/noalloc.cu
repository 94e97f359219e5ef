// noalloc.cu - vertical-slash index estimation for callers that cannot allocate.
//
// mi_vs_estimate needs a caller workspace of mi_workspace_bytes(MI_OP_VS_ESTIMATE, ...)
// bytes.  Some callers have no way to get one: a serving engine that reserves all
// device memory for its own pool up front, a plugin that runs inside another
// framework's callbacks where calling cudaMalloc is not allowed (or would force a
// device-wide synchronisation in the middle of its work), or a small tool that
// links only this library.  mi_vs_estimate_noalloc gives them the same computation
// with scratch memory owned by the library: a fixed array in device memory,
// defined below, that exists on every GPU that loads libmi.so until the process
// exits.  The call itself allocates nothing.
#include <mutex>

#include "common.cuh"

namespace {

// Library-owned estimation scratch (status word, row statistics, scores).
// On the host, `g_est_scratch` names a host-side stand-in, not device memory:
// host code must use the address returned by cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_est_scratch[MI_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mu;
// Device address of g_est_scratch, per device ordinal, looked up once with that
// device current.  It belongs to the context that existed at the lookup: after a
// cudaDeviceReset the library must not be used again in the process.
void* g_scratch_addr[64];

// Once per device, with that device current: look up the scratch's device address.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MI_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MI_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_est_scratch) != cudaSuccess || !p) return MI_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MI_OK;
}

}  // namespace

extern "C" int mi_vs_estimate_noalloc(const mi_bf16* q, const mi_bf16* k, int Hq, int Hkv, int N,
                                      int d, const int32_t* heads, int n_heads, int last_q,
                                      int k_v, int k_s, int32_t* v_idx, int32_t* s_idx,
                                      mi_stream_t stream) {
  // Argument and shape checks in mi_vs_estimate's own order: without a workspace
  // that call queues nothing and returns the first argument, shape or device
  // error, or MI_ERR_WORKSPACE when everything else is valid.
  int rc = mi_vs_estimate(q, k, Hq, Hkv, N, d, heads, n_heads, last_q, k_v, k_s, v_idx, s_idx,
                          nullptr, 0, stream);
  if (rc != MI_ERR_WORKSPACE) return rc;
  const size_t need = mi_workspace_bytes(MI_OP_VS_ESTIMATE, n_heads, Hkv, N, k_v, k_s, 0);
  if (need > MI_NOALLOC_SCRATCH_BYTES) return MI_ERR_WORKSPACE;  // job too large for the array
  void* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch)) != MI_OK) return rc;
  // The status word at the start of the scratch is cleared by the call itself;
  // every other scratch element is written before it is read.
  return mi_vs_estimate(q, k, Hq, Hkv, N, d, heads, n_heads, last_q, k_v, k_s, v_idx, s_idx,
                        scratch, MI_NOALLOC_SCRATCH_BYTES, stream);
}
