// pdl.cuh - programmatic dependent launch between the estimation kernels.
//
// A kernel launched with the programmatic stream serialization attribute may be
// scheduled while the kernel before it in the stream is still running, as soon
// as every CTA of that kernel has signalled pdl_trigger() (or exited).  Its CTAs
// can then set up (barriers, tensor memory, loads of inputs that no kernel of
// the chain writes) while the previous kernel drains, and must call pdl_wait()
// before touching anything the previous kernels write: pdl_wait() returns once
// the previous kernel has completed and its memory operations are visible, and
// since each kernel of a chain waits so before it completes, also those of every
// kernel before it.  In a kernel launched without the attribute both are no-ops.
#pragma once

namespace mi {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace mi
