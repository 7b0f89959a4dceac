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


namespace spmv {

// 16-byte asynchronous copy from global to shared memory (the address
// pair 16-byte aligned): no register holds the data, so a lane can have all
// its copies in flight at once. cp_async_wait_all waits for the lane's own
// copies; other lanes see them after a warp synchronisation.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
// 4- or 8-byte asynchronous copy from global to shared memory (both
// addresses aligned to the size).
template <int N>
__device__ __forceinline__ void cp_async_small(void* smem, const void* gmem) {
  static_assert(N == 4 || N == 8, "4 or 8 bytes");
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(gmem), "n"(N)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Copies CSR entries [a0, a1) of colIdx/value into one warp's shared-memory
// buffers: entry k to sCol[k - base], sVal[k - base], base = a0 rounded down
// to a multiple of 4, so that 4-entry groups land on 16-byte boundaries (the
// buffers start 16-byte aligned and hold a1 - base entries). VEC: colIdx and
// value are 16-byte aligned; whole groups then move as asynchronous 16-byte
// copies, all issued before one wait, and the partial groups at the two ends
// entry by entry. Positions and counters are 64-bit (a1 may lie within one
// step of INT32_MAX). All 32 lanes call it; the caller synchronises the warp
// afterwards.
template <class T, bool VEC>
__device__ __forceinline__ void warp_stage_entries(const int* __restrict__ colIdx,
                                                   const T* __restrict__ value, int a0, int a1,
                                                   int lane, int* __restrict__ sCol,
                                                   T* __restrict__ sVal) {
  const long long base = a0 & ~3LL;
  if (VEC) {
    const long long v0 = min(((long long)a0 + 3) & ~3LL, (long long)a1);  // first whole group
    const long long v1 = max((long long)a1 & ~3LL, v0);                   // end of whole groups
    for (long long g = (v0 >> 2) + lane; g < (v1 >> 2); g += 32) {
      cp_async16(sCol + (4 * g - base), colIdx + 4 * g);
      cp_async16(sVal + (4 * g - base), value + 4 * g);
      if (sizeof(T) == 8) cp_async16(sVal + (4 * g - base) + 2, value + 4 * g + 2);
    }
    for (long long k = a0 + lane; k < v0; k += 32) {
      sCol[k - base] = ld_stream(colIdx + k);
      sVal[k - base] = ld_stream(value + k);
    }
    for (long long k = v1 + lane; k < a1; k += 32) {
      sCol[k - base] = ld_stream(colIdx + k);
      sVal[k - base] = ld_stream(value + k);
    }
    cp_async_wait_all();
  } else {
    for (long long k = a0 + lane; k < a1; k += 32) {
      sCol[k - base] = ld_stream(colIdx + k);
      sVal[k - base] = ld_stream(value + k);
    }
  }
}

// Warp-staged row scatters: for widths in [kStageMinK, kStageMaxK<T>],
// kStageWarps warps per block, each with buffers of 32 * width + 8 entries.
// Narrower rows take the direct form: measured in the bench step, the CSR ->
// ELL conversion of a 5-point Laplacian (width 5) took 72.9 us staged
// against 60.4 direct, while a 27-point stencil (width 27) took 272.8
// against 335.
constexpr int kStageMinK = 24;
template <class T>
constexpr int kStageMaxK = sizeof(T) == 4 ? 32 : 24;
constexpr int kStageWarps = 4;
template <class T>
inline size_t warp_stage_smem(int width) {
  return (size_t)kStageWarps * (32 * (size_t)width + 8) * (sizeof(int) + sizeof(T));
}

}  // namespace spmv
