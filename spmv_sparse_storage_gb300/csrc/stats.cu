// stats.cu -- input validation, row-length statistics and the nnz-balanced
// CSR partition, all on the device.
//
// Validation follows the sanity rules of "Sparse matrix multiplication
// acceleration techniques", section 5.3: row_ptr must be monotone, every
// column index below the column count, and the array lengths consistent with
// nnz (rowPtrs[0] = 0, rowPtrs[numRows] = nnz). The statistics are the
// row-length histogram and variance of "[CUDA performance tuning] SpMV
// storage format selection and performance comparison", section 4.1, plus the
// max/mean load ratio of "Introduction to sparse computing and performance
// bottleneck location", section "Building the problem framework".
#include <climits>

#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

__global__ void k_stats_init(DevStats* st) {
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) st->histExact[i] = 0u;
  if (threadIdx.x < 33) st->histLog2[threadIdx.x] = 0ull;
  if (threadIdx.x == 0) {
    st->err = 0u;
    st->firstBadRow = INT_MAX;
    st->firstBadNnz = INT_MAX;
    st->maxLen = 0;
    st->minLen = INT_MAX;
    st->emptyRows = 0;
    st->maxWarpNnz = 0;
    st->pad0 = 0;
    st->sumSq = 0ull;
  }
}

__device__ __forceinline__ int log2_bin(int len) {
  // bin 0: len 0; bin b >= 1: len in [2^(b-1), 2^b)
  return len <= 0 ? 0 : 32 - __clz(len);
}

// One pass over rowPtrs: monotonicity, endpoints, lengths, histograms.
// Grid-stride over rows; block size 256 (a multiple of 32, so that each warp
// sees 32 consecutive rows and its lane 0 owns one 32-row group).
__global__ void __launch_bounds__(256) k_row_stats(int R, int Z, const int* __restrict__ rowPtrs,
                                                   DevStats* __restrict__ st) {
  __shared__ unsigned int sExact[kExactLenBins];
  __shared__ unsigned int sLog2[33];
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) sExact[i] = 0u;
  if (threadIdx.x < 33) sLog2[threadIdx.x] = 0u;
  __syncthreads();

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (rowPtrs[0] != 0) atomicOr(&st->err, kErrRowPtrStart);
    if (rowPtrs[R] != Z) atomicOr(&st->err, kErrRowPtrEnd);
  }

  int lmax = 0, lmin = INT_MAX, empties = 0, gmax = 0;
  unsigned long long sq = 0ull;
  bool bad = false;
  int firstBad = INT_MAX;
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long r0 = (long long)blockIdx.x * blockDim.x; r0 < R; r0 += stride) {
    const long long r = r0 + threadIdx.x;
    int len = 0;
    int exactKey = -1, logKey = -1;  // histogram bins, -1 = none
    if (r < R) {
      const int a = rowPtrs[r];
      const int b = rowPtrs[r + 1];
      if (b < a) {
        bad = true;
        firstBad = min(firstBad, (int)r);
      } else {
        len = b - a;
      }
      lmax = max(lmax, len);
      lmin = min(lmin, len);
      empties += (len == 0);
      sq += (unsigned long long)len * (unsigned long long)len;
      exactKey = len < kExactLenBins ? len : -1;
      logKey = log2_bin(len);
      if (lane == 0) {
        // 32 consecutive rows handled by one warp of a row-per-thread kernel
        const long long e = min(r + 32, (long long)R);
        const int g = rowPtrs[e] - a;
        gmax = max(gmax, g);
      }
    }
    // warp-aggregated histogram updates: rows of equal length in a warp are
    // counted by one shared-memory atomic (stencil rows share few lengths)
    const unsigned pe = __match_any_sync(kFullMask, exactKey);
    if (exactKey >= 0 && lane == __ffs(pe) - 1) atomicAdd(&sExact[exactKey], (unsigned)__popc(pe));
    const unsigned pl = __match_any_sync(kFullMask, logKey);
    if (logKey >= 0 && lane == __ffs(pl) - 1) atomicAdd(&sLog2[logKey], (unsigned)__popc(pl));
  }
  lmax = warp_max(lmax);
  lmin = warp_min(lmin);
  empties = warp_sum(empties);
  sq = warp_sum(sq);
  if (lane == 0) {
    if (lmax > 0) atomicMax(&st->maxLen, lmax);
    if (lmin != INT_MAX) atomicMin(&st->minLen, lmin);
    if (empties) atomicAdd(&st->emptyRows, empties);
    if (sq) atomicAdd(&st->sumSq, sq);
    if (gmax > 0) atomicMax(&st->maxWarpNnz, gmax);
  }
  if (bad) {
    atomicOr(&st->err, kErrRowPtrDecrease);
    atomicMin(&st->firstBadRow, firstBad);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x)
    if (sExact[i]) atomicAdd(&st->histExact[i], sExact[i]);
  if (threadIdx.x < 33 && sLog2[threadIdx.x])
    atomicAdd(&st->histLog2[threadIdx.x], (unsigned long long)sLog2[threadIdx.x]);
}

// Every column index must satisfy 0 <= c < numCols (unsigned compare catches
// negatives). VEC: colIdx is 16-byte aligned, read as int4.
template <bool VEC>
__global__ void __launch_bounds__(256) k_col_check(int Z, int C, const int* __restrict__ colIdx,
                                                   DevStats* __restrict__ st) {
  const unsigned uc = (unsigned)C;
  int firstBad = INT_MAX;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (VEC) {
    const long long nv = Z / 4;
    const int4* c4 = reinterpret_cast<const int4*>(colIdx);
    for (; i < nv; i += stride) {
      const int4 c = ld_stream(c4 + i);
      const int k = (int)(4 * i);
      if ((unsigned)c.x >= uc) firstBad = min(firstBad, k);
      if ((unsigned)c.y >= uc) firstBad = min(firstBad, k + 1);
      if ((unsigned)c.z >= uc) firstBad = min(firstBad, k + 2);
      if ((unsigned)c.w >= uc) firstBad = min(firstBad, k + 3);
    }
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long k = 4 * nv + t;
    if (k < Z && (unsigned)colIdx[k] >= uc) firstBad = min(firstBad, (int)k);
  } else {
    for (; i < Z; i += stride)
      if ((unsigned)ld_stream(colIdx + i) >= uc) firstBad = min(firstBad, (int)i);
  }
  if (firstBad != INT_MAX) {
    atomicOr(&st->err, kErrColRange);
    atomicMin(&st->firstBadNnz, firstBad);
  }
}

}  // namespace

cudaError_t launch_stats(int R, int C, int Z, const int* rowPtrs, const int* colIdx,
                         DevStats* st, cudaStream_t s) {
  k_stats_init<<<1, 256, 0, s>>>(st);
  const int sms = num_sms();
  long long rb = ((long long)R + 255) / 256;
  int gridR = (int)(rb < 1 ? 1 : (rb > 8LL * sms ? 8LL * sms : rb));
  k_row_stats<<<gridR, 256, 0, s>>>(R, Z, rowPtrs, st);
  int n = 2;
  if (Z > 0) {
    const bool vec = aligned16(colIdx);
    long long work = vec ? ((long long)Z / 4 + 1) : (long long)Z;
    long long cb = (work + 255) / 256;
    int gridC = (int)(cb < 1 ? 1 : (cb > 16LL * sms ? 16LL * sms : cb));
    if (vec)
      k_col_check<true><<<gridC, 256, 0, s>>>(Z, C, colIdx, st);
    else
      k_col_check<false><<<gridC, 256, 0, s>>>(Z, C, colIdx, st);
    ++n;
  }
  note_launches(n);
  return cudaGetLastError();
}

}  // namespace spmv
