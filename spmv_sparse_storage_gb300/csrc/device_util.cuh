// device_util.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace spmv {

constexpr unsigned kFullMask = 0xffffffffu;

// Matrix arrays are read exactly once per SpMV: stream them past L1 and mark
// them evict-first in L2 so that the gathered x vector stays resident.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ int4 ld_stream(const int4* p) { return __ldcs(p); }
__device__ __forceinline__ float ld_stream(const float* p) { return __ldcs(p); }
__device__ __forceinline__ int ld_stream(const int* p) { return __ldcs(p); }

// x is gathered through the read-only path (reused across rows).
__device__ __forceinline__ float ld_x(const float* p) { return __ldg(p); }

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (no-op when the kernel was
// not launched as a programmatic dependent).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next kernel in the stream (if launched as a programmatic
// dependent) to start its prologue.
__device__ __forceinline__ void grid_dependency_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(kFullMask, v, off);
  return v;
}

__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_down_sync(kFullMask, v, off));
  return v;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_down_sync(kFullMask, v, off));
  return v;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace spmv
