// Conjugate gradient around the SpMV ("Sparse Matrices and Basic Formats (COO
// and CSR)", section "Background & SpMV": A·X + Y = 0 for positive-definite A
// is solved by iterating on a guess X, forming A·X + Y and correcting X along
// a direction built from the gradient; A·X + Y is that gradient). Textbook CG
// of Hestenes and Stiefel in the gradient form g = A·X + Y, d_0 = -g_0:
//   q = A d;  alpha = g'g / d'q;  X += alpha d;  g += alpha q;
//   stop when |g| <= tol |Y|;  beta = g'g_new / g'g;  d = -g + beta d.
//
// Vectors are fp32 in HBM. Every inner product is summed in fp32 inside a
// thread and a block (a short chain, then a 256-leaf tree); each block stores
// its partial and the last block to finish (ticket counter) adds the partials
// in fp64 and derives alpha, beta and the stop decision on the device, so an
// iteration needs no host round trip. Once stopped, every kernel returns at
// entry: the iterate is the one of an exact stop however many iterations the
// host enqueued.
//
// Two kernels per iteration (the two inner products are the two grid-wide
// dependencies): with A in ELL, k_cg_ell_q forms d_new = -g + beta d_old for
// its own rows (into the other of two d buffers) and q = A d_new, taking each
// gathered d_new_j = -g_j + beta d_old_j by the same fmaf as its owner, so the
// values agree bit for bit; k_cg_update then moves X and g.
#include "internal.h"
#include "device_util.cuh"

namespace spmv {
namespace {

constexpr int kCgThreads = 256;
constexpr int kCgMaxBlocks = 4096;  // partial-sum slots in the work buffer

__device__ __forceinline__ float block_sum(float v, float* sRed) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) sRed[w] = v;
  __syncthreads();
  float s = 0.f;
  if (w == 0) {
    s = lane < (int)(blockDim.x >> 5) ? sRed[lane] : 0.f;
    s = warp_sum(s);
  }
  __syncthreads();  // sRed is reused by the next call
  return s;         // valid in thread 0
}

// Stores this block's N partial sums (partials[i * gridDim.x + block]) and
// takes a ticket; in the last block to arrive, every thread gets the fp64
// totals in tot[] (summed by warp 0) and the function returns true.
template <int N>
__device__ __forceinline__ bool grid_sum(const float (&part)[N], float* partials,
                                         unsigned* ticket, double (&tot)[N]) {
  __shared__ float sRed[kCgThreads / 32];
  __shared__ bool sLast;
  __shared__ double sTot[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float b = block_sum(part[i], sRed);
    if (threadIdx.x == 0) partials[i * gridDim.x + blockIdx.x] = b;
  }
  if (threadIdx.x == 0) {
    __threadfence();
    sLast = atomicAdd(ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!sLast) return false;
  __threadfence();
  if (threadIdx.x < 32) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      double s = 0.0;
      for (unsigned b = threadIdx.x; b < gridDim.x; b += 32)
        s += (double)__ldcg(partials + i * gridDim.x + b);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_down_sync(kFullMask, s, off);
      if (threadIdx.x == 0) sTot[i] = s;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) tot[i] = sTot[i];
  return true;
}

__device__ __forceinline__ bool running(const CgState* st) {
  return *reinterpret_cast<const volatile int*>(&st->status) == kCgRunning;
}

// g'g and Y'Y of the start; beta = 0 so that the first direction is -g (the
// d buffers are zeroed by the host); decides whether X_0 already satisfies
// the tolerance.
__global__ void __launch_bounds__(kCgThreads) k_cg_start(int R, const float* __restrict__ g,
                                                         const float* __restrict__ Y, double tol,
                                                         float* partials, CgState* st) {
  float part[2] = {0.f, 0.f};
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R;
       i += (long long)gridDim.x * blockDim.x) {
    const float gi = g[i], yi = Y[i];
    part[0] = fmaf(gi, gi, part[0]);
    part[1] = fmaf(yi, yi, part[1]);
  }
  double tot[2];
  if (grid_sum<2>(part, partials, &st->ticket, tot) && threadIdx.x == 0) {
    const double gg = tot[0], yy = tot[1];
    st->gg = gg;
    st->beta = 0.0;
    st->gnorm = sqrt(gg);
    st->stop = tol * sqrt(yy);
    st->ynorm = sqrt(yy);
    st->iter = 0;
    st->ticket = 0;
    __threadfence();
    st->status = (sqrt(gg) <= st->stop || gg == 0.0) ? kCgConverged : kCgRunning;
  }
}

__device__ __forceinline__ void finish_alpha(double dq, CgState* st) {
  st->ticket = 0;
  if (!(dq > 0.0)) {
    __threadfence();
    st->status = kCgBreakdown;
  } else {
    st->alpha = st->gg / dq;
  }
}

// generic path: d = -g + beta d in place, before q = A d
template <bool VEC>
__global__ void __launch_bounds__(kCgThreads) k_cg_direction(int R, const float* __restrict__ g,
                                                             float* __restrict__ d,
                                                             const CgState* st) {
  if (!running(st)) return;
  const float b = (float)st->beta;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (VEC) {
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4* d4 = reinterpret_cast<float4*>(d);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (R >> 2);
         i += stride) {
      const float4 gi = g4[i];
      float4 di = d4[i];
      di.x = fmaf(b, di.x, -gi.x); di.y = fmaf(b, di.y, -gi.y);
      di.z = fmaf(b, di.z, -gi.z); di.w = fmaf(b, di.w, -gi.w);
      d4[i] = di;
    }
  } else {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R; i += stride)
      d[i] = fmaf(b, d[i], -g[i]);
  }
}

// generic path: d'q after q = A d; alpha = g'g / d'q
template <bool VEC>
__global__ void __launch_bounds__(kCgThreads) k_cg_dot(int R, const float* __restrict__ d,
                                                       const float* __restrict__ q,
                                                       float* partials, CgState* st) {
  if (!running(st)) return;
  float part[1] = {0.f};
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (VEC) {
    const float4* d4 = reinterpret_cast<const float4*>(d);
    const float4* q4 = reinterpret_cast<const float4*>(q);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (R >> 2);
         i += stride) {
      const float4 a = d4[i], b = q4[i];
      part[0] = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, part[0]))));
    }
  } else {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R; i += stride)
      part[0] = fmaf(d[i], q[i], part[0]);
  }
  double tot[1];
  if (grid_sum<1>(part, partials, &st->ticket, tot) && threadIdx.x == 0) finish_alpha(tot[0], st);
}

__device__ __forceinline__ float dir(float b, float dOld, float g) { return fmaf(b, dOld, -g); }

__device__ __forceinline__ float gather_dir(const float* __restrict__ g,
                                            const float* __restrict__ dOld, float b, int c) {
  return dir(b, ld_x(dOld + c), ld_x(g + c));
}

// Asks L2 to fetch the line holding p (no register, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ELL path: d_new = -g + beta d_old (own rows, stored), q = A d_new (stored),
// d_new'q; alpha = g'g / d_new'q. Grid-stride over groups of 4 rows when
// numRows % 4 == 0 (aligned 16-byte slot loads), else over single rows.
template <bool VEC4>
__global__ void __launch_bounds__(kCgThreads, 4) k_cg_ell_q(
    int R, int K, const int* __restrict__ ellCol, const float* __restrict__ ellVal,
    const float* __restrict__ g, const float* __restrict__ dOld, float* __restrict__ dNew,
    float* __restrict__ q, float* partials, CgState* st) {
  if (VEC4) {
    // the first four slot rows of this thread's first rows into L2 before the
    // wait (the matrix is never written during the solve; no registers held)
    const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long ld = R >> 2;
    if (first < ld) {
      for (int u = 0; u < 4 && u < K; ++u) {
        prefetch_l2(reinterpret_cast<const int4*>(ellCol) + (size_t)u * ld + first);
        prefetch_l2(reinterpret_cast<const float4*>(ellVal) + (size_t)u * ld + first);
      }
    }
  }
  grid_dependency_wait();     // the previous update's g, d and state
  grid_dependency_trigger();  // the next kernel may be scheduled as blocks exit
  if (!running(st)) return;
  const float b = (float)st->beta;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float part[1] = {0.f};
  if (VEC4) {
    const long long ld = R >> 2;
    const int4* c4 = reinterpret_cast<const int4*>(ellCol);
    const float4* v4 = reinterpret_cast<const float4*>(ellVal);
    for (long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; t0 < ld; t0 += stride) {
      const float4 gi = reinterpret_cast<const float4*>(g)[t0];
      const float4 oi = reinterpret_cast<const float4*>(dOld)[t0];
      const float4 di = make_float4(dir(b, oi.x, gi.x), dir(b, oi.y, gi.y), dir(b, oi.z, gi.z),
                                    dir(b, oi.w, gi.w));
      reinterpret_cast<float4*>(dNew)[t0] = di;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      int t = 0;
      for (; t + 4 <= K; t += 4) {
        int4 c[4];
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          c[u] = ld_stream(c4 + (size_t)(t + u) * ld + t0);
          v[u] = ld_stream(v4 + (size_t)(t + u) * ld + t0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (c[u].x >= 0) acc.x = fmaf(v[u].x, gather_dir(g, dOld, b, c[u].x), acc.x);
          if (c[u].y >= 0) acc.y = fmaf(v[u].y, gather_dir(g, dOld, b, c[u].y), acc.y);
          if (c[u].z >= 0) acc.z = fmaf(v[u].z, gather_dir(g, dOld, b, c[u].z), acc.z);
          if (c[u].w >= 0) acc.w = fmaf(v[u].w, gather_dir(g, dOld, b, c[u].w), acc.w);
        }
      }
      for (; t < K; ++t) {
        const int4 c = ld_stream(c4 + (size_t)t * ld + t0);
        const float4 v = ld_stream(v4 + (size_t)t * ld + t0);
        if (c.x >= 0) acc.x = fmaf(v.x, gather_dir(g, dOld, b, c.x), acc.x);
        if (c.y >= 0) acc.y = fmaf(v.y, gather_dir(g, dOld, b, c.y), acc.y);
        if (c.z >= 0) acc.z = fmaf(v.z, gather_dir(g, dOld, b, c.z), acc.z);
        if (c.w >= 0) acc.w = fmaf(v.w, gather_dir(g, dOld, b, c.w), acc.w);
      }
      reinterpret_cast<float4*>(q)[t0] = acc;
      part[0] = fmaf(di.x, acc.x, fmaf(di.y, acc.y, fmaf(di.z, acc.z, fmaf(di.w, acc.w, part[0]))));
    }
  } else {
    for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += stride) {
      const float di = dir(b, dOld[r], g[r]);
      dNew[r] = di;
      float acc = 0.f;
      for (int t = 0; t < K; ++t) {
        const int c = ld_stream(ellCol + (size_t)t * R + r);
        const float v = ld_stream(ellVal + (size_t)t * R + r);
        if (c >= 0) acc = fmaf(v, gather_dir(g, dOld, b, c), acc);
      }
      q[r] = acc;
      part[0] = fmaf(di, acc, part[0]);
    }
  }
  double tot[1];
  if (grid_sum<1>(part, partials, &st->ticket, tot) && threadIdx.x == 0) finish_alpha(tot[0], st);
}

// X += alpha d; g += alpha q; g'g; then the stop test and beta.
template <bool VEC>
__global__ void __launch_bounds__(kCgThreads, 4) k_cg_update(int R, float* __restrict__ X,
                                                             float* __restrict__ g,
                                                             const float* __restrict__ d,
                                                             const float* __restrict__ q,
                                                             float* partials, CgState* st) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  float part[1] = {0.f};
  if (VEC) {
    float4* X4 = reinterpret_cast<float4*>(X);
    float4* g4 = reinterpret_cast<float4*>(g);
    const float4* d4 = reinterpret_cast<const float4*>(d);
    const float4* q4 = reinterpret_cast<const float4*>(q);
    const long long n4 = R >> 2;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    // X and g of the first trip load before the wait: the SpMV kernel this
    // waits for writes only d and q (and reads g), and the update before it
    // has finished (that kernel waits for it before it lets this one start)
    float4 x[2], gi[2];
    bool have = i + stride < n4;
    if (have) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        x[u] = X4[i + u * stride];
        gi[u] = g4[i + u * stride];
      }
    }
    grid_dependency_wait();  // the direction, q and alpha of this iteration
    grid_dependency_trigger();
    if (!running(st)) return;
    const float a = (float)st->alpha;
    // two elements per trip so that 8 independent 16-byte loads are in flight
    for (; i + stride < n4; i += 2 * stride) {
      float4 di[2], qi[2];
      if (!have) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          x[u] = X4[i + u * stride];
          gi[u] = g4[i + u * stride];
        }
      }
      have = false;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        di[u] = d4[i + u * stride];
        qi[u] = q4[i + u * stride];
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        x[u].x = fmaf(a, di[u].x, x[u].x); x[u].y = fmaf(a, di[u].y, x[u].y);
        x[u].z = fmaf(a, di[u].z, x[u].z); x[u].w = fmaf(a, di[u].w, x[u].w);
        gi[u].x = fmaf(a, qi[u].x, gi[u].x); gi[u].y = fmaf(a, qi[u].y, gi[u].y);
        gi[u].z = fmaf(a, qi[u].z, gi[u].z); gi[u].w = fmaf(a, qi[u].w, gi[u].w);
        X4[i + u * stride] = x[u];
        g4[i + u * stride] = gi[u];
        part[0] = fmaf(gi[u].x, gi[u].x, fmaf(gi[u].y, gi[u].y,
                  fmaf(gi[u].z, gi[u].z, fmaf(gi[u].w, gi[u].w, part[0]))));
      }
    }
    if (i < n4) {
      float4 x = X4[i], gi = g4[i];
      const float4 di = d4[i], qi = q4[i];
      x.x = fmaf(a, di.x, x.x); x.y = fmaf(a, di.y, x.y);
      x.z = fmaf(a, di.z, x.z); x.w = fmaf(a, di.w, x.w);
      gi.x = fmaf(a, qi.x, gi.x); gi.y = fmaf(a, qi.y, gi.y);
      gi.z = fmaf(a, qi.z, gi.z); gi.w = fmaf(a, qi.w, gi.w);
      X4[i] = x;
      g4[i] = gi;
      part[0] = fmaf(gi.x, gi.x, fmaf(gi.y, gi.y, fmaf(gi.z, gi.z, fmaf(gi.w, gi.w, part[0]))));
    }
  } else {
    grid_dependency_wait();  // the direction, q and alpha of this iteration
    grid_dependency_trigger();
    if (!running(st)) return;
    const float a = (float)st->alpha;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R; i += stride) {
      X[i] = fmaf(a, d[i], X[i]);
      const float gi = fmaf(a, q[i], g[i]);
      g[i] = gi;
      part[0] = fmaf(gi, gi, part[0]);
    }
  }
  double tot[1];
  if (grid_sum<1>(part, partials, &st->ticket, tot) && threadIdx.x == 0) {
    const double ggNew = tot[0];
    st->ticket = 0;
    st->iter += 1;
    st->gnorm = sqrt(ggNew);
    if (sqrt(ggNew) <= st->stop || ggNew == 0.0) {
      __threadfence();
      st->status = kCgConverged;
    } else {
      st->beta = ggNew / st->gg;
      st->gg = ggNew;
    }
  }
}

// Blocks for a grid-stride kernel: every SM filled to its resident limit for
// that kernel (queried once per kernel slot and device), fewer for small
// inputs, at most kCgMaxBlocks (the partial-sum slots).
enum CgKernelSlot { kSlotStart, kSlotDir4, kSlotDir1, kSlotDot4, kSlotDot1, kSlotEll4, kSlotEll1,
                    kSlotUpd4, kSlotUpd1, kNumSlots };
constexpr int kCgMaxDevices = 64;

template <class Kernel>
unsigned resident_grid(Kernel kernel, int slot, long long work) {
  static int perSm[kNumSlots][kCgMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < kCgMaxDevices;
  int n = cached ? perSm[slot][dev] : 0;
  if (n <= 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kCgThreads, 0) != cudaSuccess ||
        n <= 0) {
      cudaGetLastError();
      n = 2;
    }
    if (cached) perSm[slot][dev] = n;
  }
  long long cap = (long long)n * num_sms();
  if (cap > kCgMaxBlocks) cap = kCgMaxBlocks;
  const long long want = (work + kCgThreads - 1) / kCgThreads;
  return (unsigned)(want < 1 ? 1 : want < cap ? want : cap);
}

}  // namespace

size_t cg_partials_floats() { return 2 * (size_t)kCgMaxBlocks; }

cudaError_t launch_cg_start(int R, const float* g, const float* Y, double tol, float* partials,
                            CgState* st, cudaStream_t s) {
  k_cg_start<<<resident_grid(k_cg_start, kSlotStart, R), kCgThreads, 0, s>>>(R, g, Y, tol, partials, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cg_direction(int R, const float* g, float* d, const CgState* st,
                                cudaStream_t s) {
  if ((R & 3) == 0)
    k_cg_direction<true><<<resident_grid(k_cg_direction<true>, kSlotDir4, R / 4), kCgThreads, 0, s>>>(
        R, g, d, st);
  else
    k_cg_direction<false><<<resident_grid(k_cg_direction<false>, kSlotDir1, R), kCgThreads, 0, s>>>(
        R, g, d, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cg_dot(int R, const float* d, const float* q, float* partials, CgState* st,
                          cudaStream_t s) {
  if ((R & 3) == 0)
    k_cg_dot<true><<<resident_grid(k_cg_dot<true>, kSlotDot4, R / 4), kCgThreads, 0, s>>>(R, d, q,
                                                                               partials, st);
  else
    k_cg_dot<false><<<resident_grid(k_cg_dot<false>, kSlotDot1, R), kCgThreads, 0, s>>>(R, d, q,
                                                                             partials, st);
  note_launches(1);
  return cudaGetLastError();
}

// The ELL path's two kernels per iteration go out as programmatic dependent
// launches: each waits (griddepcontrol.wait) for the kernel before it to
// complete, so the launch and the scheduling of its blocks overlap the end
// of that kernel instead of following it.
template <class Kernel, class... Args>
cudaError_t launch_dependent(Kernel kernel, unsigned grid, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCgThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_cg_ell_q(int R, int K, const int* ellCol, const float* ellVal, const float* g,
                            const float* dOld, float* dNew, float* q, float* partials,
                            CgState* st, cudaStream_t s) {
  cudaError_t e;
  if ((R & 3) == 0 && aligned16(ellCol) && aligned16(ellVal))
    e = launch_dependent(k_cg_ell_q<true>, resident_grid(k_cg_ell_q<true>, kSlotEll4, R / 4), s,
                         R, K, ellCol, ellVal, g, dOld, dNew, q, partials, st);
  else
    e = launch_dependent(k_cg_ell_q<false>, resident_grid(k_cg_ell_q<false>, kSlotEll1, R), s,
                         R, K, ellCol, ellVal, g, dOld, dNew, q, partials, st);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_cg_update(int R, float* X, float* g, const float* d, const float* q,
                             float* partials, CgState* st, cudaStream_t s) {
  cudaError_t e;
  if ((R & 3) == 0 && aligned16(X))
    e = launch_dependent(k_cg_update<true>, resident_grid(k_cg_update<true>, kSlotUpd4, R / 4), s,
                         R, X, g, d, q, partials, st);
  else
    e = launch_dependent(k_cg_update<false>, resident_grid(k_cg_update<false>, kSlotUpd1, R), s,
                         R, X, g, d, q, partials, st);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spmv
