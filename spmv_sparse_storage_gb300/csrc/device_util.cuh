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

__device__ __forceinline__ double ld_stream(const double* p) { return __ldcs(p); }

// x is gathered through the read-only path (reused across rows).
__device__ __forceinline__ float ld_x(const float* p) { return __ldg(p); }
__device__ __forceinline__ double ld_x(const double* p) { return __ldg(p); }

// Value type of the matrix and the vectors: float (4-byte values) or double
// (8-byte values). Vec4<T> = four consecutive values read or written with
// 16-byte accesses (one for float, two for double); the address must be
// 16-byte aligned.
template <class T>
struct Vec4 {
  T x, y, z, w;
};
__device__ __forceinline__ Vec4<float> ld4_stream(const float* p) {
  const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
  return {v.x, v.y, v.z, v.w};
}
__device__ __forceinline__ Vec4<double> ld4_stream(const double* p) {
  const double2 a = __ldcs(reinterpret_cast<const double2*>(p));
  const double2 b = __ldcs(reinterpret_cast<const double2*>(p) + 1);
  return {a.x, a.y, b.x, b.y};
}
__device__ __forceinline__ Vec4<float> ld4(const float* p) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  return {v.x, v.y, v.z, v.w};
}
__device__ __forceinline__ Vec4<double> ld4(const double* p) {
  const double2 a = reinterpret_cast<const double2*>(p)[0];
  const double2 b = reinterpret_cast<const double2*>(p)[1];
  return {a.x, a.y, b.x, b.y};
}
__device__ __forceinline__ void st4(float* p, const Vec4<float>& v) {
  *reinterpret_cast<float4*>(p) = make_float4(v.x, v.y, v.z, v.w);
}
__device__ __forceinline__ void st4(double* p, const Vec4<double>& v) {
  reinterpret_cast<double2*>(p)[0] = make_double2(v.x, v.y);
  reinterpret_cast<double2*>(p)[1] = make_double2(v.z, v.w);
}
__device__ __forceinline__ float fma_t(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fma_t(double a, double b, double c) { return fma(a, b, c); }

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

