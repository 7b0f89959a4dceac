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
// colIdx (both streams at once), and each block adds its results into the
// zeroed DevStats record with atomics (maxima, sums, histogram bins) as it
// finishes, so that nothing is left to fold after the last block.
#include <climits>

#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

constexpr int kStatsRowsPerThread = 8;
constexpr int kStatsRows = 256 * kStatsRowsPerThread;  // rows per row block
constexpr int kColUnroll = 4;                           // column check: vectors in flight

// Work area: the DevStats record alone (zeroed before the launch).
constexpr size_t kWorkBytes = (sizeof(DevStats) + 255) / 256 * 256;

// Row blocks: at most kRowBlocksPerSm per SM, each walking several
// kStatsRows-row tiles, so that a block's fixed tail (shared-memory
// histogram flush, reductions, atomics) is paid once per block rather than
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

// Word W of the flat bit array of chunk masks: bit p (nonzero position p)
// is bit p % 32 of word p / 32, kept in the mask of chunk p / kCsrChunk.
__device__ __forceinline__ unsigned* mask_word(CsrChunkDesc* desc, long long W) {
  return reinterpret_cast<unsigned*>(&desc[W >> 2].mask) + (W & 3);
}

// Row part. A block walks tiles blk, blk + nbRow, ... of kStatsRows
// consecutive rows; a lane takes kStatsRowsPerThread consecutive rows, whose
// kStatsRowsPerThread + 1 row pointers come from two 16-byte loads and one
// shuffle (when rowPtrs is 16-byte aligned and the tile whole; scalar loads
// otherwise). From them, in registers: monotonicity, lengths, min/max/sum of
// squares, the nonzeros of each 32 consecutive rows (4 lanes), an exact
// length histogram (lengths < kExactLenBins; one shared add per warp when its
// 256 rows share a length, else one per run of equal lengths; longer rows go
// to the log2 bins), and the CSR chunk records (bounds-checked: they are
// written before validation is known). A nonempty row is `lo` of every chunk
// whose first nonzero it holds (and `hi` of the chunk before) and sets the
// bit of its start position in the chunk where it starts; a lane gathers its
// rows' bits in a 64-bit window and ORs at most two words into the records.
// An empty row inside a chunk flags that chunk.
__device__ void row_part(int blk, int nbRow, int R, int Z, bool rowVec,
                         const int* __restrict__ rowPtrs,
                         DevStats* __restrict__ st, int nChunks,
                         CsrChunkDesc* __restrict__ desc) {
  constexpr int E = kStatsRowsPerThread;
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
  for (long long tile = blk; tile < nTiles; tile += nbRow) {
    const long long r0 = tile * kStatsRows + (long long)threadIdx.x * E;
    const bool wholeTile = (tile + 1) * kStatsRows <= (long long)R;  // block-uniform
    // p[e] = rowPtrs[r0 + e]; past rowPtrs[R] it is INT_MAX (never a start)
    int p[E + 1];
    int nLive;  // rows r0 .. r0 + nLive - 1 exist
    if (rowVec && wholeTile) {
      const int4 u = *reinterpret_cast<const int4*>(rowPtrs + r0);
      const int4 v = *reinterpret_cast<const int4*>(rowPtrs + r0 + 4);
      const int last = lane == 31 ? __ldg(rowPtrs + r0 + E) : 0;
      p[0] = u.x; p[1] = u.y; p[2] = u.z; p[3] = u.w;
      p[4] = v.x; p[5] = v.y; p[6] = v.z; p[7] = v.w;
      const int next = __shfl_down_sync(kFullMask, p[0], 1);
      p[E] = lane == 31 ? last : next;
      nLive = E;
    } else {
#pragma unroll
      for (int e = 0; e <= E; ++e) p[e] = r0 + e <= R ? rowPtrs[r0 + e] : INT_MAX;
      const long long left = (long long)R - r0;
      nLive = left <= 0 ? 0 : (left >= E ? E : (int)left);
    }
    // per-row statistics (lengths are recomputed from p where needed)
    int kmn = INT_MAX, kmx = -1;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool live = e < nLive;
      // monotonicity by comparison, not by the sign of a 32-bit difference
      // (which wraps for far-apart values); with rowPtrs[0] = 0 and
      // rowPtrs[R] = nnz it confines every row pointer to [0, nnz]
      const bool dec = p[e + 1] < p[e];
      if (live && dec) firstBad = min(firstBad, (int)(r0 + e));
      int l = dec ? 0 : (int)((unsigned)p[e + 1] - (unsigned)p[e]);
      l = l > 0 ? l : 0;
      if (live) {
        lmax = max(lmax, l);
        lmin = min(lmin, l);
        empties += l == 0;
        sq += (unsigned long long)(unsigned)l * (unsigned)l;
        kmn = min(kmn, l);
        kmx = max(kmx, l);
      }
    }
    // nonzeros of each aligned group of 32 rows (4 lanes)
    const int pBeg = p[0];
    int pEnd = pBeg;  // p[nLive], by selects (no dynamic register index)
#pragma unroll
    for (int e = 1; e <= E; ++e) pEnd = e <= nLive ? p[e] : pEnd;
    int groupNnz = nLive > 0 ? (int)((unsigned)pEnd - (unsigned)pBeg) : 0;
    groupNnz += __shfl_xor_sync(kFullMask, groupNnz, 1);
    groupNnz += __shfl_xor_sync(kFullMask, groupNnz, 2);
    gmax = max(gmax, groupNnz);
    // exact histogram
    const int wmn = __reduce_min_sync(kFullMask, kmn);
    const int wmx = __reduce_max_sync(kFullMask, kmx);
    if (wmn == wmx && wmx < kExactLenBins) {  // one length (wmx >= 0: some row lives)
      const int rows = __reduce_add_sync(kFullMask, (unsigned)nLive);
      if (lane == 0) atomicAdd(&sExact[wmx], (unsigned)rows);
    } else {
      int cur = -1;
      unsigned cnt = 0u;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        int l = -1;  // as in the statistics loop above
        if (e < nLive && p[e + 1] >= p[e]) l = max((int)((unsigned)p[e + 1] - (unsigned)p[e]), 0);
        else if (e < nLive) l = 0;
        if (l >= kExactLenBins) atomicAdd(&st->histLog2[32 - __clz(l)], 1ull);
        const int key = l < kExactLenBins ? l : -1;
        if (key != cur) {
          if (cur >= 0) atomicAdd(&sExact[cur], cnt);
          cur = key;
          cnt = 0u;
        }
        ++cnt;
      }
      if (cur >= 0) atomicAdd(&sExact[cur], cnt);
    }
    // chunk records; only on a consistent lane range (always, for valid input)
    if (nLive > 0 && 0 <= pBeg && pBeg < pEnd && pEnd <= Z) {
      // lo/hi of the chunks whose first position q lies in [pBeg, pEnd): the
      // row holding q is the last of the lane's rows starting at or before q
      const int cLast = min((pEnd - 1) / kCsrChunk, nChunks - 1);
      for (int c = (pBeg + kCsrChunk - 1) / kCsrChunk; c <= cLast; ++c) {
        const int q = c * kCsrChunk;
        int e = 0;
#pragma unroll
        for (int k = 1; k < E; ++k) e += (k < nLive && p[k] <= q);
        const int r = (int)(r0 + e);
        desc[c].lo = r;
        if (c > 0) desc[c - 1].hi = r;
      }
      // start bits of nonempty rows, in a 64-bit window from word pBeg / 32
      const long long W0 = pBeg >> 5;
      unsigned long long win = 0ull;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int a = p[e];
        const bool live = e < nLive;
        if (live && p[e + 1] > a && (a & (kCsrChunk - 1)) != 0 && a >= 0 && p[e + 1] <= Z) {
          const long long off = (long long)a - (W0 << 5);
          if (off >= 0 && off < 64)  // (off < 0 only on invalid input)
            win |= 1ull << off;
          else
            atomicOr(mask_word(desc, a >> 5), 1u << (a & 31));
        } else if (live && p[e + 1] <= a && a > 0 && a < Z && (a & (kCsrChunk - 1)) != 0) {
          atomicOr(&desc[a / kCsrChunk].flags, kCsrChunkHasEmptyRow);
        }
      }
      if ((unsigned)win) atomicOr(mask_word(desc, W0), (unsigned)win);
      if ((unsigned)(win >> 32)) atomicOr(mask_word(desc, W0 + 1), (unsigned)(win >> 32));
    } else if (nLive > 0) {
      // empty lane range: every live row is empty (or the input is invalid)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int a = p[e];
        if (e < nLive && p[e + 1] <= a && a > 0 && a < Z && (a & (kCsrChunk - 1)) != 0)
          atomicOr(&desc[a / kCsrChunk].flags, kCsrChunkHasEmptyRow);
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
    int mx = 0, mn = INT_MAX, emp = 0, gm = 0, fb = INT_MAX;
    unsigned long long sqs = 0ull;
    for (int w = 0; w < 8; ++w) {
      mx = max(mx, sRed[0][w]);
      mn = min(mn, sRed[1][w]);
      emp += sRed[2][w];
      gm = max(gm, sRed[3][w]);
      fb = min(fb, sRed[4][w]);
      sqs += sSq[w];
    }
    if (mx) atomicMax(&st->maxLen, mx);
    if (mn != INT_MAX) atomicMax(&st->minLenKey, INT_MAX - mn);
    if (emp) atomicAdd(&st->emptyRows, emp);
    if (gm) atomicMax(&st->maxWarpNnz, gm);
    if (fb != INT_MAX) atomicMax(&st->badRowKey, INT_MAX - fb);
    if (sqs) atomicAdd(&st->sumSq, sqs);
  }
  for (int i = threadIdx.x; i < kExactLenBins; i += blockDim.x)
    if (sExact[i]) atomicAdd(&st->histExact[i], sExact[i]);
}

// Column part: every column index must satisfy 0 <= c < numCols (unsigned
// compare catches negatives). VEC: colIdx is 16-byte aligned, read as int4,
// kColUnroll vectors per thread in flight. The first kGatherSampleBlocks
// column blocks also sample the x-gather spread: distinct 128-byte lines of x
// among the 32 gathers of one warp load.
template <bool VEC>
__device__ void col_part(int cblk, int nbCol, int Z, int C, const int* __restrict__ colIdx,
                         DevStats* __restrict__ st) {
  const unsigned uc = (unsigned)C;
  int firstBad = INT_MAX;
  const bool sample = cblk < kGatherSampleBlocks;
  unsigned nLines = 0u, nSets = 0u;
  if (VEC) {
    // 32-bit indices: nv < 2^29 and the grid stride is small
    const int nv = Z / 4;
    const int stride = nbCol * (int)blockDim.x;
    const int4* c4 = reinterpret_cast<const int4*>(colIdx);
    int i = cblk * (int)blockDim.x + (int)threadIdx.x;
    // all lanes of a warp run the same number of iterations (the bound only
    // depends on the warp's first index), so the warp match below is uniform
    int i0 = i - (int)(threadIdx.x & 31);
    for (; i0 < nv; i += kColUnroll * stride, i0 += kColUnroll * stride) {
      int4 c[kColUnroll];
#pragma unroll
      for (int u = 0; u < kColUnroll; ++u)
        c[u] = i + u * stride < nv ? ld_stream(c4 + i + u * stride) : make_int4(0, 0, 0, 0);
      // any entry out of range? (the zero fill is in range: C > 0 when Z > 0)
      bool bad = false;
#pragma unroll
      for (int u = 0; u < kColUnroll; ++u)
        bad |= ((unsigned)c[u].x >= uc) | ((unsigned)c[u].y >= uc) | ((unsigned)c[u].z >= uc) |
               ((unsigned)c[u].w >= uc);
      if (bad) {  // the first bad position (only on invalid input)
#pragma unroll
        for (int u = 0; u < kColUnroll; ++u) {
          const int iu = i + u * stride;
          if (iu < nv) {
            const int k = 4 * iu;
            if ((unsigned)c[u].x >= uc) firstBad = min(firstBad, k);
            if ((unsigned)c[u].y >= uc) firstBad = min(firstBad, k + 1);
            if ((unsigned)c[u].z >= uc) firstBad = min(firstBad, k + 2);
            if ((unsigned)c[u].w >= uc) firstBad = min(firstBad, k + 3);
          }
        }
      }
      if (sample) {
        const bool in = i < nv;
        const unsigned ln = in ? ((unsigned)c[0].x >> 5) : 0xffffffffu;
        const unsigned peers = __match_any_sync(kFullMask, ln);
        const bool leader = (threadIdx.x & 31) == __ffs(peers) - 1;
        if (i0 + 32 <= nv) {  // full sets only
          if (leader) ++nLines;
          if ((threadIdx.x & 31) == 0) ++nSets;
        }
      }
    }
    const long long t = (long long)cblk * blockDim.x + threadIdx.x;
    const long long k = 4LL * nv + t;
    if (k < Z && (unsigned)colIdx[k] >= uc) firstBad = min(firstBad, (int)k);
  } else {
    const long long stride = (long long)nbCol * blockDim.x;
    for (long long i = (long long)cblk * blockDim.x + threadIdx.x; i < Z; i += stride)
      if ((unsigned)ld_stream(colIdx + i) >= uc) firstBad = min(firstBad, (int)i);
  }
  unsigned long long lines = nLines, sets = nSets;
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
    int fb = INT_MAX;
    unsigned long long ln = 0ull, ss = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      fb = min(fb, sB[w]);
      ln += sL[w];
      ss += sS[w];
    }
    if (fb != INT_MAX) atomicMax(&st->badNnzKey, INT_MAX - fb);
    if (ln) atomicAdd(&st->gatherLines, ln);
    if (ss) atomicAdd(&st->gatherSets, ss);
  }
}

template <bool VEC>
__global__ void __launch_bounds__(256) k_validate_stats(int R, int C, int Z,
                                                        const int* __restrict__ rowPtrs,
                                                        const int* __restrict__ colIdx,
                                                        DevStats* __restrict__ st, int nbRow,
                                                        int nbCol, int nChunks,
                                                        CsrChunkDesc* __restrict__ desc,
                                                        bool rowVec) {
  if ((int)blockIdx.x < nbRow)
    row_part(blockIdx.x, nbRow, R, Z, rowVec, rowPtrs, st, nChunks, desc);
  else
    col_part<VEC>(blockIdx.x - nbRow, nbCol, Z, C, colIdx, st);
}

// Column blocks: up to 8 per SM, each walking the column array grid-stride;
// blocks beyond those resident start as row blocks finish.
int col_blocks(int Z, bool vec) {
  if (Z <= 0) return 0;
  const long long work = vec ? ((long long)Z / 4 + 1) : (long long)Z;
  const long long cb = (work + 255) / 256;
  const long long cap = 8LL * num_sms();
  return (int)(cb < 1 ? 1 : (cb > cap ? cap : cb));
}

}  // namespace

size_t stats_work_bytes(int, int, const int*) { return kWorkBytes; }


cudaError_t launch_stats(int R, int C, int Z, const int* rowPtrs, const int* colIdx, void* work,
                         int nChunks, CsrChunkDesc* desc, cudaStream_t s) {
  const bool vec = aligned16(colIdx);
  const bool rowVec = aligned16(rowPtrs);
  const int nbRow = row_blocks(R);
  const int nbCol = col_blocks(Z, vec);
  DevStats* w = static_cast<DevStats*>(work);
  if (vec)
    k_validate_stats<true><<<nbRow + nbCol, 256, 0, s>>>(R, C, Z, rowPtrs, colIdx, w, nbRow,
                                                         nbCol, nChunks, desc, rowVec);
  else
    k_validate_stats<false><<<nbRow + nbCol, 256, 0, s>>>(R, C, Z, rowPtrs, colIdx, w, nbRow,
                                                          nbCol, nChunks, desc, rowVec);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace spmv
