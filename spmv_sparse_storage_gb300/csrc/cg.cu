// Conjugate gradient around the SpMV ("Sparse Matrices and Basic Formats (COO
// and CSR)", section "Background & SpMV": A·X + Y = 0 for positive-definite A
// is solved by iterating on a guess X, forming A·X + Y and correcting X along
// a direction built from the gradient; A·X + Y is that gradient). Textbook CG
// of Hestenes and Stiefel in the gradient form g = A·X + Y, d_0 = -g_0:
//   q = A d;  alpha = g'g / d'q;  X += alpha d;  g += alpha q;
//   stop when |g| <= tol |Y|;  beta = g'g_new / g'g;  d = -g + beta d.
//
// Vectors are fp32 in HBM. Every inner product is summed in fp32 inside a
// thread and a block (a short chain, then a 256-leaf tree) and in fp64 across
// blocks (one atomic per block); the last block to finish (ticket counter)
// derives alpha, beta and the stop decision on the device, so an iteration
// needs no host round trip. Once stopped, every kernel returns at entry: the
// iterate is the one of an exact stop however many iterations the host
// enqueued.
#include "internal.h"
#include "device_util.cuh"

namespace spmv {
namespace {

constexpr int kCgThreads = 256;

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
  return s;  // valid in thread 0
}

// Adds this block's partial sums into acc[0..n) (fp64); returns true in
// thread 0 of the last block to arrive, after every block's sums are in.
template <int N>
__device__ __forceinline__ bool block_accumulate(const float (&part)[N], double* acc,
                                                 unsigned* ticket, float* sRed) {
  float tot[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    tot[i] = block_sum(part[i], sRed);
    __syncthreads();
  }
  bool last = false;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) atomicAdd(acc + i, (double)tot[i]);
    __threadfence();
    last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    if (last) __threadfence();
  }
  return last;
}

// the last block reads a total and clears the accumulator for its next use
__device__ __forceinline__ double take(double* p) {
  const unsigned long long bits = atomicExch(reinterpret_cast<unsigned long long*>(p), 0ull);
  return __longlong_as_double((long long)bits);
}

__device__ __forceinline__ bool running(const CgState* st) {
  return *reinterpret_cast<const volatile int*>(&st->status) == kCgRunning;
}

// d = -g, g'g and Y'Y; decides whether X_0 already satisfies the tolerance.
__global__ void __launch_bounds__(kCgThreads) k_cg_start(int R, const float* __restrict__ g,
                                                         const float* __restrict__ Y,
                                                         float* __restrict__ d, double tol,
                                                         CgState* st) {
  __shared__ float sRed[kCgThreads / 32];
  float part[2] = {0.f, 0.f};
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R;
       i += (long long)gridDim.x * blockDim.x) {
    const float gi = g[i], yi = Y[i];
    d[i] = -gi;
    part[0] = fmaf(gi, gi, part[0]);
    part[1] = fmaf(yi, yi, part[1]);
  }
  if (block_accumulate<2>(part, st->acc, &st->ticket, sRed)) {
    const double gg = take(st->acc), yy = take(st->acc + 1);
    st->gg = gg;
    st->gnorm = sqrt(gg);
    st->stop = tol * sqrt(yy);
    st->ynorm = sqrt(yy);
    st->iter = 0;
    st->ticket = 0;
    __threadfence();
    st->status = (sqrt(gg) <= st->stop || gg == 0.0) ? kCgConverged : kCgRunning;
  }
}

// d'q after a generic SpMV (q = A d); alpha = g'g / d'q.
template <bool VEC>
__global__ void __launch_bounds__(kCgThreads) k_cg_dot(int R, const float* __restrict__ d,
                                                       const float* __restrict__ q,
                                                       CgState* st) {
  __shared__ float sRed[kCgThreads / 32];
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
  if (block_accumulate<1>(part, st->acc, &st->ticket, sRed)) {
    const double dq = take(st->acc);
    st->ticket = 0;
    if (!(dq > 0.0)) {
      __threadfence();
      st->status = kCgBreakdown;
    } else {
      st->alpha = st->gg / dq;
    }
  }
}

// q = A d with A in ELL (column-major slots, padding column -1), written
// (not accumulated), fused with d'q; alpha = g'g / d'q. Four rows per thread
// when numRows % 4 == 0 (aligned 16-byte slot loads), else one.
template <bool VEC4>
__global__ void __launch_bounds__(kCgThreads, 4) k_cg_ell_q(int R, int K,
                                                            const int* __restrict__ ellCol,
                                                            const float* __restrict__ ellVal,
                                                            const float* __restrict__ d,
                                                            float* __restrict__ q, CgState* st) {
  __shared__ float sRed[kCgThreads / 32];
  if (!running(st)) return;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  float part[1] = {0.f};
  if (VEC4) {
    const long long ld = R >> 2;
    if (t0 < ld) {
      const int4* c4 = reinterpret_cast<const int4*>(ellCol);
      const float4* v4 = reinterpret_cast<const float4*>(ellVal);
      const float4 di = reinterpret_cast<const float4*>(d)[t0];
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
          if (c[u].x >= 0) acc.x = fmaf(v[u].x, ld_x(d + c[u].x), acc.x);
          if (c[u].y >= 0) acc.y = fmaf(v[u].y, ld_x(d + c[u].y), acc.y);
          if (c[u].z >= 0) acc.z = fmaf(v[u].z, ld_x(d + c[u].z), acc.z);
          if (c[u].w >= 0) acc.w = fmaf(v[u].w, ld_x(d + c[u].w), acc.w);
        }
      }
      for (; t < K; ++t) {
        const int4 c = ld_stream(c4 + (size_t)t * ld + t0);
        const float4 v = ld_stream(v4 + (size_t)t * ld + t0);
        if (c.x >= 0) acc.x = fmaf(v.x, ld_x(d + c.x), acc.x);
        if (c.y >= 0) acc.y = fmaf(v.y, ld_x(d + c.y), acc.y);
        if (c.z >= 0) acc.z = fmaf(v.z, ld_x(d + c.z), acc.z);
        if (c.w >= 0) acc.w = fmaf(v.w, ld_x(d + c.w), acc.w);
      }
      reinterpret_cast<float4*>(q)[t0] = acc;
      part[0] = fmaf(di.x, acc.x, fmaf(di.y, acc.y, fmaf(di.z, acc.z, di.w * acc.w)));
    }
  } else if (t0 < R) {
    float acc = 0.f;
    for (int t = 0; t < K; ++t) {
      const int c = ld_stream(ellCol + (size_t)t * R + t0);
      const float v = ld_stream(ellVal + (size_t)t * R + t0);
      if (c >= 0) acc = fmaf(v, ld_x(d + c), acc);
    }
    q[t0] = acc;
    part[0] = d[t0] * acc;
  }
  if (block_accumulate<1>(part, st->acc, &st->ticket, sRed)) {
    const double dq = take(st->acc);
    st->ticket = 0;
    if (!(dq > 0.0)) {
      __threadfence();
      st->status = kCgBreakdown;
    } else {
      st->alpha = st->gg / dq;
    }
  }
}

// X += alpha d; g += alpha q; g'g; then the stop test and beta.
template <bool VEC>
__global__ void __launch_bounds__(kCgThreads) k_cg_update(int R, float* __restrict__ X,
                                                          float* __restrict__ g,
                                                          const float* __restrict__ d,
                                                          const float* __restrict__ q,
                                                          CgState* st) {
  __shared__ float sRed[kCgThreads / 32];
  if (!running(st)) return;
  const float a = (float)st->alpha;
  float part[1] = {0.f};
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (VEC) {
    float4* X4 = reinterpret_cast<float4*>(X);
    float4* g4 = reinterpret_cast<float4*>(g);
    const float4* d4 = reinterpret_cast<const float4*>(d);
    const float4* q4 = reinterpret_cast<const float4*>(q);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (R >> 2);
         i += stride) {
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
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R; i += stride) {
      X[i] = fmaf(a, d[i], X[i]);
      const float gi = fmaf(a, q[i], g[i]);
      g[i] = gi;
      part[0] = fmaf(gi, gi, part[0]);
    }
  }
  if (block_accumulate<1>(part, st->acc, &st->ticket, sRed)) {
    const double ggNew = take(st->acc);
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

// d = -g + beta d
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

// grid of a streaming kernel: enough blocks to fill every SM a few times over
unsigned stream_grid(long long work) {
  const long long want = (work + kCgThreads - 1) / kCgThreads;
  const long long cap = 8LL * num_sms();
  return (unsigned)(want < 1 ? 1 : want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_cg_start(int R, const float* g, const float* Y, float* d, double tol,
                            CgState* st, cudaStream_t s) {
  k_cg_start<<<stream_grid(R), kCgThreads, 0, s>>>(R, g, Y, d, tol, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cg_dot(int R, const float* d, const float* q, CgState* st, cudaStream_t s) {
  if ((R & 3) == 0)
    k_cg_dot<true><<<stream_grid(R / 4), kCgThreads, 0, s>>>(R, d, q, st);
  else
    k_cg_dot<false><<<stream_grid(R), kCgThreads, 0, s>>>(R, d, q, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cg_ell_q(int R, int K, const int* ellCol, const float* ellVal, const float* d,
                            float* q, CgState* st, cudaStream_t s) {
  const bool vec = (R & 3) == 0 && aligned16(ellCol) && aligned16(ellVal);
  const long long threads = vec ? R / 4 : R;
  const unsigned blocks = (unsigned)((threads + kCgThreads - 1) / kCgThreads);
  if (vec)
    k_cg_ell_q<true><<<blocks ? blocks : 1, kCgThreads, 0, s>>>(R, K, ellCol, ellVal, d, q, st);
  else
    k_cg_ell_q<false><<<blocks ? blocks : 1, kCgThreads, 0, s>>>(R, K, ellCol, ellVal, d, q, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cg_update(int R, float* X, float* g, const float* d, const float* q,
                             CgState* st, cudaStream_t s) {
  if ((R & 3) == 0 && aligned16(X))
    k_cg_update<true><<<stream_grid(R / 4), kCgThreads, 0, s>>>(R, X, g, d, q, st);
  else
    k_cg_update<false><<<stream_grid(R), kCgThreads, 0, s>>>(R, X, g, d, q, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cg_direction(int R, const float* g, float* d, const CgState* st,
                                cudaStream_t s) {
  if ((R & 3) == 0)
    k_cg_direction<true><<<stream_grid(R / 4), kCgThreads, 0, s>>>(R, g, d, st);
  else
    k_cg_direction<false><<<stream_grid(R), kCgThreads, 0, s>>>(R, g, d, st);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace spmv
