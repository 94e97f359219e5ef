// common.cuh - definitions shared by the kernels and the C-ABI host code.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/mi.h"

namespace mi {

constexpr int kD = MI_HEAD_DIM;    // head dim handled by the kernels
constexpr int kBM = 128;           // query rows per attention CTA (one UMMA M)
constexpr int kBN = 128;           // keys per tile (one UMMA N)
constexpr int kLastQ = MI_LAST_Q;  // estimation query rows per head
constexpr int kBlk = MI_BLOCK;     // pattern block (first block, local block, 64x64 blocks)
constexpr int kChunkKeys = 1024;   // keys per estimation CTA
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // bounded pipeline waits: 4 s

// Head list passed by value as a kernel parameter (host-side list, no copy).
struct HeadList {
  int n;
  int16_t h[MI_MAX_HEADS];
};

// Record a data-dependent error in the status word (first error wins).
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace mi
