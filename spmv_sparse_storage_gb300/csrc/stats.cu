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

constexpr int kStatsRowsPerThread = 8;
constexpr int kStatsRows = 256 * kStatsRowsPerThread;
constexpr int kColUnroll = 4;  // column check: vectors in flight per thread

__global__ void k_stats_init(DevStats* st, unsigned* histRep) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  for (int i = t; i < kStatsReplicas * kExactLenBins; i += gridDim.x * blockDim.x) histRep[i] = 0u;
  if (blockIdx.x == 0) {
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
      st->gatherLines = 0ull;
      st->gatherSets = 0ull;
    }
  }
}

// One pass over rowPtrs: monotonicity, endpoints, lengths, histograms, and
// the CSR chunk map (desc[c].lo = row holding nonzero c*kCsrChunk). A block
// takes kStatsRows consecutive rows, kStatsRowsPerThread per thread, 256
// apart so that each load instruction is coalesced, and issues all its loads
// before it uses any. The block's maxima, minima and sums go to its own
// partial record (no atomics); lengths below kExactLenBins are counted in a
// shared histogram that is added to one of kStatsReplicas global copies;
// longer rows are counted in the log2 bins directly (their log2 bins for
// shorter rows are derived on the host from the exact histogram).
__global__ void __launch_bounds__(256) k_row_stats(int R, int Z, const int* __restrict__ rowPtrs,
                                                   DevStats* __restrict__ st,
                                                   StatsPartial* __restrict__ partials,
                                                   unsigned* __restrict__ histRep, int nChunks,
                                                   CsrChunkDesc* __restrict__ desc) {
  __shared__ unsigned int sExact[kExactLenBins];
  __shared__ int sRed[5][8];
  __shared__ unsigned long long sSq[8];
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) sExact[i] = 0u;
  __syncthreads();

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (rowPtrs[0] != 0) atomicOr(&st->err, kErrRowPtrStart);
    if (rowPtrs[R] != Z) atomicOr(&st->err, kErrRowPtrEnd);
    if (nChunks > 0) desc[nChunks - 1].hi = R > 0 ? R - 1 : 0;
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
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
      if (len >= kExactLenBins) atomicAdd(&st->histLog2[32 - __clz(len)], 1ull);
      // CSR chunk records (bounds-checked: this runs before the validation
      // result is known). A nonempty row is `lo` of every chunk whose first
      // nonzero it holds (and `hi` of the chunk before), and sets the bit of
      // its start position in the chunk where it starts; an empty row inside
      // a chunk flags that chunk.
      if (a[i] >= 0 && b[i] <= Z && b[i] > a[i]) {
        const int c0 = (a[i] + kCsrChunk - 1) / kCsrChunk;
        const int c1 = min((b[i] - 1) / kCsrChunk, nChunks - 1);
        for (int c = c0; c <= c1; ++c) {
          desc[c].lo = (int)r;
          if (c > 0) desc[c - 1].hi = (int)r;
        }
        const int pos = a[i] % kCsrChunk;
        if (pos != 0) {
          unsigned* m = reinterpret_cast<unsigned*>(&desc[a[i] / kCsrChunk].mask);
          atomicOr(m + (pos >> 5), 1u << (pos & 31));
        }
      } else if (a[i] == b[i] && a[i] > 0 && a[i] < Z && a[i] % kCsrChunk != 0) {
        atomicOr(&desc[a[i] / kCsrChunk].flags, kCsrChunkHasEmptyRow);
      }
    }
    // warp-aggregated exact histogram: when all 32 rows share one length
    // (stencils, uniform rows) one shared atomic; otherwise one per distinct
    // length found with a warp match
    const int key = (live && len < kExactLenBins) ? len : -1;
    const int kmin = __reduce_min_sync(kFullMask, key);
    const int kmax = __reduce_max_sync(kFullMask, key);
    if (kmin == kmax) {
      if (lane == 0 && key >= 0) atomicAdd(&sExact[key], 32u);
    } else {
      const unsigned peers = __match_any_sync(kFullMask, key);
      if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sExact[key], (unsigned)__popc(peers));
    }
  }
  lmax = warp_max(lmax);
  lmin = warp_min(lmin);
  empties = warp_sum(empties);
  sq = warp_sum(sq);
  gmax = warp_max(gmax);
  firstBad = warp_min(firstBad);
  if (lane == 0) {
    sRed[0][wid] = lmax;
    sRed[1][wid] = lmin;
    sRed[2][wid] = empties;
    sRed[3][wid] = gmax;
    sRed[4][wid] = firstBad;
    sSq[wid] = sq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    StatsPartial p;
    p.maxLen = 0; p.minLen = INT_MAX; p.emptyRows = 0; p.maxWarpNnz = 0;
    p.firstBadRow = INT_MAX; p.pad0 = 0; p.sumSq = 0ull;
    for (int w = 0; w < 8; ++w) {
      p.maxLen = max(p.maxLen, sRed[0][w]);
      p.minLen = min(p.minLen, sRed[1][w]);
      p.emptyRows += sRed[2][w];
      p.maxWarpNnz = max(p.maxWarpNnz, sRed[3][w]);
      p.firstBadRow = min(p.firstBadRow, sRed[4][w]);
      p.sumSq += sSq[w];
    }
    partials[blockIdx.x] = p;
  }
  unsigned* rep = histRep + (size_t)(blockIdx.x % kStatsReplicas) * kExactLenBins;
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x)
    if (sExact[i]) atomicAdd(rep + i, sExact[i]);
}

// Fold the per-block partials and the histogram replicas into DevStats.
__global__ void __launch_bounds__(1024) k_stats_reduce(int nBlocks,
                                                       const StatsPartial* __restrict__ partials,
                                                       const unsigned* __restrict__ histRep,
                                                       DevStats* __restrict__ st) {
  __shared__ int sRed[5][32];
  __shared__ unsigned long long sSq[32];
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) {
    unsigned v = 0u;
    for (int r = 0; r < kStatsReplicas; ++r) v += histRep[(size_t)r * kExactLenBins + i];
    st->histExact[i] = v;
  }
  int mx = 0, mn = INT_MAX, emp = 0, gm = 0, fb = INT_MAX;
  unsigned long long sq = 0ull;
  for (int i = threadIdx.x; i < nBlocks; i += blockDim.x) {
    const StatsPartial p = partials[i];
    mx = max(mx, p.maxLen);
    mn = min(mn, p.minLen);
    emp += p.emptyRows;
    gm = max(gm, p.maxWarpNnz);
    fb = min(fb, p.firstBadRow);
    sq += p.sumSq;
  }
  mx = warp_max(mx);
  mn = warp_min(mn);
  emp = warp_sum(emp);
  gm = warp_max(gm);
  fb = warp_min(fb);
  sq = warp_sum(sq);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) {
    sRed[0][wid] = mx; sRed[1][wid] = mn; sRed[2][wid] = emp; sRed[3][wid] = gm; sRed[4][wid] = fb;
    sSq[wid] = sq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int nw = blockDim.x / 32;
    for (int w = 0; w < nw; ++w) {
      mx = max(mx, sRed[0][w]);
      mn = min(mn, sRed[1][w]);
      gm = max(gm, sRed[3][w]);
      fb = min(fb, sRed[4][w]);
    }
    emp = 0;
    sq = 0ull;
    for (int w = 0; w < nw; ++w) {
      emp += sRed[2][w];
      sq += sSq[w];
    }
    st->maxLen = mx;
    st->minLen = mn;
    st->emptyRows = emp;
    st->maxWarpNnz = gm;
    st->sumSq = sq;
    if (fb != INT_MAX) {
      st->err |= kErrRowPtrDecrease;
      st->firstBadRow = fb;
    }
  }
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
  const bool sample = blockIdx.x < kGatherSampleBlocks;
  unsigned long long lines = 0ull, sets = 0ull;
  if (VEC) {
    const long long nv = Z / 4;
    const int4* c4 = reinterpret_cast<const int4*>(colIdx);
    // kColUnroll vectors per thread per iteration, all loaded before any is
    // checked; all lanes of a warp run the same number of iterations (the
    // bound only depends on the warp's first index), so the warp match below
    // is uniform
    long long i0 = i - (threadIdx.x & 31);
    for (; i0 < nv; i += kColUnroll * stride, i0 += kColUnroll * stride) {
      int4 c[kColUnroll];
#pragma unroll
      for (int u = 0; u < kColUnroll; ++u)
        c[u] = i + u * stride < nv ? ld_stream(c4 + i + u * stride) : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kColUnroll; ++u) {
        const long long iu = i + u * stride;
        if (iu < nv) {
          const int k = (int)(4 * iu);
          if ((unsigned)c[u].x >= uc) firstBad = min(firstBad, k);
          if ((unsigned)c[u].y >= uc) firstBad = min(firstBad, k + 1);
          if ((unsigned)c[u].z >= uc) firstBad = min(firstBad, k + 2);
          if ((unsigned)c[u].w >= uc) firstBad = min(firstBad, k + 3);
        }
      }
      if (sample) {
        // distinct 128-byte lines of x among the 32 gathers of one warp load
        const bool in = i < nv;
        const unsigned ln = in ? ((unsigned)c[0].x >> 5) : 0xffffffffu;
        const unsigned peers = __match_any_sync(kFullMask, ln);
        const bool leader = (threadIdx.x & 31) == __ffs(peers) - 1;
        if (i0 + 32 <= nv) {  // full sets only
          if (leader) ++lines;
          if ((threadIdx.x & 31) == 0) ++sets;
        }
      }
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
  if (VEC && sample) {
    __shared__ unsigned long long sL[8], sS[8];
    lines = warp_sum(lines);
    sets = warp_sum(sets);
    if ((threadIdx.x & 31) == 0) {
      sL[threadIdx.x >> 5] = lines;
      sS[threadIdx.x >> 5] = sets;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long L = 0ull, S = 0ull;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        L += sL[w];
        S += sS[w];
      }
      if (S) {
        atomicAdd(&st->gatherLines, L);
        atomicAdd(&st->gatherSets, S);
      }
    }
  }
}

}  // namespace

size_t stats_scratch_bytes(int R) {
  const long long nb = ((long long)R + kStatsRows - 1) / kStatsRows;
  return (size_t)(nb < 1 ? 1 : nb) * sizeof(StatsPartial) +
         (size_t)kStatsReplicas * kExactLenBins * sizeof(unsigned);
}

cudaError_t launch_stats(int R, int C, int Z, const int* rowPtrs, const int* colIdx,
                         DevStats* st, void* scratch, int nChunks, CsrChunkDesc* desc,
                         cudaStream_t s) {
  const long long rb = ((long long)R + kStatsRows - 1) / kStatsRows;
  const int nb = (int)(rb < 1 ? 1 : rb);
  unsigned* histRep = static_cast<unsigned*>(scratch);
  StatsPartial* partials =
      reinterpret_cast<StatsPartial*>(histRep + (size_t)kStatsReplicas * kExactLenBins);
  k_stats_init<<<32, 256, 0, s>>>(st, histRep);
  k_row_stats<<<nb, 256, 0, s>>>(R, Z, rowPtrs, st, partials, histRep, nChunks, desc);
  int n = 3;
  const int sms = num_sms();
  if (Z > 0) {
    const bool vec = aligned16(colIdx);
    long long work = vec ? ((long long)Z / 4 + 1) : (long long)Z;
    long long cb = (work + 255) / 256;
    int gridC = (int)(cb < 1 ? 1 : (cb > 8LL * sms ? 8LL * sms : cb));
    if (vec)
      k_col_check<true><<<gridC, 256, 0, s>>>(Z, C, colIdx, st);
    else
      k_col_check<false><<<gridC, 256, 0, s>>>(Z, C, colIdx, st);
    ++n;
  }
  k_stats_reduce<<<1, 1024, 0, s>>>(nb, partials, histRep, st);
  note_launches(n);
  return cudaGetLastError();
}

}  // namespace spmv
