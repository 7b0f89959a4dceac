// stats.cu -- input validation, row-length statistics and the nnz-balanced
// CSR chunk map, all on the device.
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

// One pass over rowPtrs: monotonicity, endpoints, lengths, histograms, and
// the CSR chunk map (chunkRow[c] = row holding nonzero c*kCsrChunk). A block
// takes kStatsRows consecutive rows, kStatsRowsPerThread per thread, 256
// apart so that each load instruction is coalesced, and issues all its loads
// before it uses any. Lengths below kExactLenBins go to an exact histogram
// (their log2 bins are derived from it on the host); longer rows are counted
// in the log2 bins directly.
constexpr int kStatsRowsPerThread = 8;
constexpr int kStatsRows = 256 * kStatsRowsPerThread;

__global__ void __launch_bounds__(256) k_row_stats(int R, int Z, const int* __restrict__ rowPtrs,
                                                   DevStats* __restrict__ st, int nChunks,
                                                   int* __restrict__ chunkRow) {
  __shared__ unsigned int sExact[kExactLenBins];
  __shared__ unsigned int sLog2[33];
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) sExact[i] = 0u;
  if (threadIdx.x < 33) sLog2[threadIdx.x] = 0u;
  __syncthreads();

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (rowPtrs[0] != 0) atomicOr(&st->err, kErrRowPtrStart);
    if (rowPtrs[R] != Z) atomicOr(&st->err, kErrRowPtrEnd);
    chunkRow[nChunks] = R > 0 ? R - 1 : 0;
  }
  const int lane = threadIdx.x & 31;
  const long long base = (long long)blockIdx.x * kStatsRows + threadIdx.x;
  int a[kStatsRowsPerThread], b[kStatsRowsPerThread], g[kStatsRowsPerThread];
#pragma unroll
  for (int i = 0; i < kStatsRowsPerThread; ++i) {
    const long long r = base + i * 256;
    a[i] = r < R ? rowPtrs[r] : 0;
    b[i] = r < R ? rowPtrs[r + 1] : 0;
    // 32 consecutive rows handled by one warp of a row-per-thread kernel
    g[i] = (r < R && lane == 0) ? rowPtrs[min(r + 32, (long long)R)] : 0;
  }
  int lmax = 0, lmin = INT_MAX, empties = 0, gmax = 0;
  unsigned long long sq = 0ull;
  int firstBad = INT_MAX;
#pragma unroll
  for (int i = 0; i < kStatsRowsPerThread; ++i) {
    const long long r = base + i * 256;
    const bool live = r < R;
    int len = 0;
    if (live) {
      if (b[i] < a[i])
        firstBad = min(firstBad, (int)r);
      else
        len = b[i] - a[i];
      lmax = max(lmax, len);
      lmin = min(lmin, len);
      empties += (len == 0);
      sq += (unsigned long long)len * (unsigned long long)len;
      if (lane == 0) gmax = max(gmax, g[i] - a[i]);
      if (len >= kExactLenBins) atomicAdd(&sLog2[32 - __clz(len)], 1u);
      // chunks whose first nonzero lies in this row (bounds-checked: runs
      // before the validation result is known)
      if (a[i] >= 0 && b[i] <= Z && b[i] > a[i]) {
        const int c0 = (a[i] + kCsrChunk - 1) / kCsrChunk;
        const int c1 = min((b[i] - 1) / kCsrChunk, nChunks - 1);
        for (int c = c0; c <= c1; ++c) chunkRow[c] = (int)r;
      }
    }
    // warp-aggregated exact histogram: one shared atomic per distinct length
    const int key = (live && len < kExactLenBins) ? len : -1;
    const unsigned peers = __match_any_sync(kFullMask, key);
    if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sExact[key], (unsigned)__popc(peers));
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
  if (firstBad != INT_MAX) {
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
                         DevStats* st, int nChunks, int* chunkRow, cudaStream_t s) {
  k_stats_init<<<1, 256, 0, s>>>(st);
  const int sms = num_sms();
  const long long rb = ((long long)R + kStatsRows - 1) / kStatsRows;
  k_row_stats<<<(unsigned)(rb < 1 ? 1 : rb), 256, 0, s>>>(R, Z, rowPtrs, st, nChunks, chunkRow);
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
