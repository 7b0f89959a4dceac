// stats.cu -- input validation, row-length statistics and the nnz-balanced
// CSR chunk records, all on the device, in one kernel launch.
//
// Validation follows the sanity rules of "Sparse matrix multiplication
// acceleration techniques", section 5.3: row_ptr must be monotone, every
// column index below the column count, and the array lengths consistent with
// nnz (rowPtrs[0] = 0, rowPtrs[numRows] = nnz). The statistics are the
// row-length histogram and variance of "[CUDA performance tuning] SpMV
// storage format selection and performance comparison", section 4.1, plus the
// max/mean load ratio of "Introduction to sparse computing and performance
// bottleneck location", section "Building the problem framework".
//
// One grid does everything: its first blocks walk rowPtrs, the others walk
// colIdx (both streams at once), each block writes a partial record, and the
// last block to finish folds the records into DevStats (no inter-block wait:
// a block learns it is last from an atomic ticket).
#include <climits>

#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

constexpr int kStatsRowsPerThread = 8;
constexpr int kStatsRows = 256 * kStatsRowsPerThread;  // rows per row block
constexpr int kColUnroll = 4;                           // column check: vectors in flight
constexpr int kStatsReplicaCount = 8;                   // copies of the exact histogram

struct ColPartial {
  int firstBad;
  int pad0;
  unsigned long long lines, sets;
};

// Work area layout (one allocation, zeroed up to `zero_bytes`):
//   DevStats | ticket (16 B) | histogram replicas | row partials | column partials
struct WorkLayout {
  size_t ticket, rep, rowPart, colPart, zero, total;
};

__host__ __device__ inline WorkLayout work_layout(int nbRow, int nbCol) {
  WorkLayout L;
  L.ticket = (sizeof(DevStats) + 15) / 16 * 16;
  L.rep = L.ticket + 16;
  L.rowPart = L.rep + (size_t)kStatsReplicaCount * kExactLenBins * sizeof(unsigned);
  L.zero = L.rowPart;
  L.colPart = L.rowPart + (size_t)nbRow * sizeof(StatsPartial);
  L.total = L.colPart + (size_t)(nbCol > 0 ? nbCol : 1) * sizeof(ColPartial);
  return L;
}

// Row blocks: at most kRowBlocksPerSm per SM, each walking several
// kStatsRows-row tiles, so that a block's fixed tail (shared-memory
// histogram, reductions, fence, ticket) is paid once per block rather than
// once per tile.
constexpr int kRowBlocksPerSm = 2;
long long row_tiles(int R) {
  const long long t = ((long long)R + kStatsRows - 1) / kStatsRows;
  return t < 1 ? 1 : t;
}
int row_blocks(int R) {
  const long long t = row_tiles(R);
  const long long cap = (long long)kRowBlocksPerSm * num_sms();
  return (int)(t < cap ? t : cap);
}

int col_blocks(int Z, bool vec) {
  if (Z <= 0) return 0;
  const long long work = vec ? ((long long)Z / 4 + 1) : (long long)Z;
  const long long cb = (work + 255) / 256;
  const long long cap = 8LL * num_sms();
  return (int)(cb < 1 ? 1 : (cb > cap ? cap : cb));
}

// Row part. A block walks tiles blk, blk + nbRow, ... of kStatsRows
// consecutive rows, kStatsRowsPerThread per thread, 256 apart so that each
// load is coalesced, and issues all of a tile's loads before it uses any:
// monotonicity, lengths, min/max/sum of squares,
// the max nonzeros of any 32 consecutive rows, an exact length histogram
// (lengths < kExactLenBins; longer rows go to the log2 bins), and the CSR
// chunk records (bounds-checked: they are written before validation is
// known). A nonempty row is `lo` of every chunk whose first nonzero it holds
// (and `hi` of the chunk before) and sets the bit of its start position in
// the chunk where it starts; an empty row inside a chunk flags that chunk.
__device__ void row_part(int blk, int nbRow, int R, int Z, const int* __restrict__ rowPtrs,
                         DevStats* __restrict__ st, StatsPartial* __restrict__ partials,
                         unsigned* __restrict__ histRep, int nChunks,
                         CsrChunkDesc* __restrict__ desc) {
  __shared__ unsigned int sExact[kExactLenBins];
  __shared__ int sRed[5][8];
  __shared__ unsigned long long sSq[8];
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) sExact[i] = 0u;
  __syncthreads();

  if (blk == 0 && threadIdx.x == 0) {
    if (rowPtrs[0] != 0) atomicOr(&st->err, kErrRowPtrStart);
    if (rowPtrs[R] != Z) atomicOr(&st->err, kErrRowPtrEnd);
    if (nChunks > 0) desc[nChunks - 1].hi = R > 0 ? R - 1 : 0;
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int lmax = 0, lmin = INT_MAX, empties = 0, gmax = 0;
  unsigned long long sq = 0ull;
  int firstBad = INT_MAX;
  const long long nTiles = ((long long)R + kStatsRows - 1) / kStatsRows;
  for (long long tile = blk; tile < (nTiles > 0 ? nTiles : 1); tile += nbRow) {
    const long long base = tile * kStatsRows + threadIdx.x;
    int a[kStatsRowsPerThread], b[kStatsRowsPerThread], g[kStatsRowsPerThread];
#pragma unroll
    for (int i = 0; i < kStatsRowsPerThread; ++i) {
      const long long r = base + i * 256;
      a[i] = r < R ? rowPtrs[r] : 0;
      b[i] = r < R ? rowPtrs[r + 1] : 0;
      // 32 consecutive rows handled by one warp of a row-per-thread kernel
      g[i] = (r < R && lane == 0) ? rowPtrs[min(r + 32, (long long)R)] : 0;
    }
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
    partials[blk] = p;
  }
  unsigned* rep = histRep + (size_t)(blk % kStatsReplicaCount) * kExactLenBins;
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x)
    if (sExact[i]) atomicAdd(rep + i, sExact[i]);
}

// Column part: every column index must satisfy 0 <= c < numCols (unsigned
// compare catches negatives). VEC: colIdx is 16-byte aligned, read as int4,
// kColUnroll vectors per thread in flight. The first kGatherSampleBlocks
// column blocks also sample the x-gather spread: distinct 128-byte lines of x
// among the 32 gathers of one warp load.
template <bool VEC>
__device__ void col_part(int cblk, int nbCol, int Z, int C, const int* __restrict__ colIdx,
                         ColPartial* __restrict__ colPart) {
  const unsigned uc = (unsigned)C;
  int firstBad = INT_MAX;
  const long long stride = (long long)nbCol * blockDim.x;
  long long i = (long long)cblk * blockDim.x + threadIdx.x;
  const bool sample = cblk < kGatherSampleBlocks;
  unsigned long long lines = 0ull, sets = 0ull;
  if (VEC) {
    const long long nv = Z / 4;
    const int4* c4 = reinterpret_cast<const int4*>(colIdx);
    // all lanes of a warp run the same number of iterations (the bound only
    // depends on the warp's first index), so the warp match below is uniform
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
    const long long t = (long long)cblk * blockDim.x + threadIdx.x;
    const long long k = 4 * nv + t;
    if (k < Z && (unsigned)colIdx[k] >= uc) firstBad = min(firstBad, (int)k);
  } else {
    for (; i < Z; i += stride)
      if ((unsigned)ld_stream(colIdx + i) >= uc) firstBad = min(firstBad, (int)i);
  }
  __shared__ unsigned long long sL[8], sS[8];
  __shared__ int sB[8];
  firstBad = warp_min(firstBad);
  lines = warp_sum(lines);
  sets = warp_sum(sets);
  if ((threadIdx.x & 31) == 0) {
    sL[threadIdx.x >> 5] = lines;
    sS[threadIdx.x >> 5] = sets;
    sB[threadIdx.x >> 5] = firstBad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ColPartial p;
    p.firstBad = INT_MAX;
    p.pad0 = 0;
    p.lines = 0ull;
    p.sets = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      p.firstBad = min(p.firstBad, sB[w]);
      p.lines += sL[w];
      p.sets += sS[w];
    }
    colPart[cblk] = p;
  }
}

// The last block: fold row partials, column partials and histogram replicas.
__device__ void finalize(int nbRow, int nbCol, DevStats* __restrict__ st,
                         const StatsPartial* __restrict__ partials,
                         const ColPartial* __restrict__ colPart,
                         const unsigned* __restrict__ histRep) {
  __shared__ int sRed[6][8];
  __shared__ unsigned long long sU[3][8];
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x) {
    unsigned v = 0u;
#pragma unroll
    for (int r = 0; r < kStatsReplicaCount; ++r) v += histRep[(size_t)r * kExactLenBins + i];
    st->histExact[i] = v;
  }
  int mx = 0, mn = INT_MAX, emp = 0, gm = 0, fb = INT_MAX, fc = INT_MAX;
  unsigned long long sq = 0ull, ln = 0ull, ss = 0ull;
  for (int i = threadIdx.x; i < nbRow; i += blockDim.x) {
    const StatsPartial p = partials[i];
    mx = max(mx, p.maxLen);
    mn = min(mn, p.minLen);
    emp += p.emptyRows;
    gm = max(gm, p.maxWarpNnz);
    fb = min(fb, p.firstBadRow);
    sq += p.sumSq;
  }
  for (int i = threadIdx.x; i < nbCol; i += blockDim.x) {
    const ColPartial p = colPart[i];
    fc = min(fc, p.firstBad);
    ln += p.lines;
    ss += p.sets;
  }
  mx = warp_max(mx);
  mn = warp_min(mn);
  emp = warp_sum(emp);
  gm = warp_max(gm);
  fb = warp_min(fb);
  fc = warp_min(fc);
  sq = warp_sum(sq);
  ln = warp_sum(ln);
  ss = warp_sum(ss);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) {
    sRed[0][wid] = mx; sRed[1][wid] = mn; sRed[2][wid] = emp;
    sRed[3][wid] = gm; sRed[4][wid] = fb; sRed[5][wid] = fc;
    sU[0][wid] = sq; sU[1][wid] = ln; sU[2][wid] = ss;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mx = 0; mn = INT_MAX; emp = 0; gm = 0; fb = INT_MAX; fc = INT_MAX;
    sq = ln = ss = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      mx = max(mx, sRed[0][w]);
      mn = min(mn, sRed[1][w]);
      emp += sRed[2][w];
      gm = max(gm, sRed[3][w]);
      fb = min(fb, sRed[4][w]);
      fc = min(fc, sRed[5][w]);
      sq += sU[0][w];
      ln += sU[1][w];
      ss += sU[2][w];
    }
    st->maxLen = mx;
    st->minLen = mn;
    st->emptyRows = emp;
    st->maxWarpNnz = gm;
    st->sumSq = sq;
    st->gatherLines = ln;
    st->gatherSets = ss;
    st->firstBadRow = fb;
    st->firstBadNnz = fc;
    unsigned err = st->err;
    if (fb != INT_MAX) err |= kErrRowPtrDecrease;
    if (fc != INT_MAX) err |= kErrColRange;
    st->err = err;
  }
}

template <bool VEC>
__global__ void __launch_bounds__(256) k_validate_stats(int R, int C, int Z,
                                                        const int* __restrict__ rowPtrs,
                                                        const int* __restrict__ colIdx,
                                                        unsigned char* __restrict__ work,
                                                        int nbRow, int nbCol, int nChunks,
                                                        CsrChunkDesc* __restrict__ desc) {
  const WorkLayout L = work_layout(nbRow, nbCol);
  DevStats* st = reinterpret_cast<DevStats*>(work);
  unsigned* ticket = reinterpret_cast<unsigned*>(work + L.ticket);
  unsigned* histRep = reinterpret_cast<unsigned*>(work + L.rep);
  StatsPartial* partials = reinterpret_cast<StatsPartial*>(work + L.rowPart);
  ColPartial* colPart = reinterpret_cast<ColPartial*>(work + L.colPart);
  if ((int)blockIdx.x < nbRow)
    row_part(blockIdx.x, nbRow, R, Z, rowPtrs, st, partials, histRep, nChunks, desc);
  else
    col_part<VEC>(blockIdx.x - nbRow, nbCol, Z, C, colIdx, colPart);
  // publish this block's results, then take a ticket; the last block folds
  __shared__ bool sLast;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sLast = atomicAdd(ticket, 1u) == (unsigned)(nbRow + nbCol - 1);
  __syncthreads();
  if (sLast) {
    __threadfence();
    finalize(nbRow, nbCol, st, partials, colPart, histRep);
  }
}

}  // namespace

size_t stats_work_bytes(int R, int Z, const int* colIdx) {
  return work_layout(row_blocks(R), col_blocks(Z, aligned16(colIdx))).total;
}

size_t stats_zero_bytes() { return work_layout(1, 1).zero; }

cudaError_t launch_stats(int R, int C, int Z, const int* rowPtrs, const int* colIdx, void* work,
                         int nChunks, CsrChunkDesc* desc, cudaStream_t s) {
  const bool vec = aligned16(colIdx);
  const int nbRow = row_blocks(R);
  const int nbCol = col_blocks(Z, vec);
  unsigned char* w = static_cast<unsigned char*>(work);
  if (vec)
    k_validate_stats<true><<<nbRow + nbCol, 256, 0, s>>>(R, C, Z, rowPtrs, colIdx, w, nbRow,
                                                         nbCol, nChunks, desc);
  else
    k_validate_stats<false><<<nbRow + nbCol, 256, 0, s>>>(R, C, Z, rowPtrs, colIdx, w, nbRow,
                                                          nbCol, nChunks, desc);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace spmv
