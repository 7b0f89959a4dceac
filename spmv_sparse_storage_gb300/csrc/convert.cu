// convert.cu -- on-device conversion of a CSR matrix into the other storage
// formats, plus the device scans and the stable row sort they use.
//
// Formats (PMPP notes):
//   COO -- "Sparse Matrices and Basic Formats (COO and CSR)", section "COO
//          format and SpMV": every nonzero carries its row index.
//   ELL -- "Regularized Formats (ELL, Hybrid ELL-COO and JDS)", section "ELL
//          format: padding + transposition": rows padded to a common width,
//          stored column-major (slot t*numRows + row).
//   HYB -- same page, section "Hybrid ELL-COO format": surplus entries of
//          long rows move to a COO part in row order.
//   JDS -- same page, section "JDS format": rows sorted by length (longest
//          first), a row permutation, jagged diagonals starting at iterPtr[t].
#include <climits>

#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

// ---------------------------------------------------------------------------
// Warp-cooperative segmented expansion (the HYB tail). A warp owns 32
// consecutive segments (rows) whose outputs are contiguous: segment j covers
// output positions [start_j, start_{j+1}). The warp walks its output range 32
// positions at a time (coalesced writes); each lane finds its segment by a
// 5-step binary search over the 32 starts held one per lane.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int find_segment(int start, int k) {
  // largest lane j with start_j <= k (starts non-decreasing over lanes)
  int j = 0;
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {
    const int sc = __shfl_sync(kFullMask, start, j + step);
    if (sc <= k) j += step;
  }
  return j;
}

// HYB COO part: row r's entries at in-row positions >= K, written at
// tailPtr[r] ... in row order (warp-cooperative expansion as above).
template <class T>
__global__ void __launch_bounds__(256) k_hyb_tail_copy(int R, int K, const int* __restrict__ rowPtrs,
                                                       const int* __restrict__ colIdx,
                                                       const T* __restrict__ value,
                                                       const int* __restrict__ tailPtr,
                                                       int* __restrict__ cooRow,
                                                       int* __restrict__ cooCol,
                                                       T* __restrict__ cooVal) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long r0 = warp * 32;
  if (r0 >= R) return;
  const long long r = r0 + lane;
  const int start = r < R ? tailPtr[r] : INT_MAX;
  const int src = r < R ? rowPtrs[r] + K : 0;
  const int A = __shfl_sync(kFullMask, start, 0);
  const int B = tailPtr[min(r0 + 32, (long long)R)];
  // 64-bit counter: B may lie within one step of INT32_MAX
  for (long long base = A; base < B; base += 32) {
    const int o = (int)min(base + lane, (long long)B);  // o == B: no entry
    const int j = find_segment(start, o);
    const int sj = __shfl_sync(kFullMask, start, j);
    const int srcj = __shfl_sync(kFullMask, src, j);
    if (o < B) {
      const int k = srcj + (o - sj);
      cooRow[o] = (int)(r0 + j);
      cooCol[o] = colIdx[k];
      cooVal[o] = value[k];
    }
  }
}

// ---------------------------------------------------------------------------
// Exclusive scan (reduce, scan of block sums, apply), no inter-block waits.
// Input is produced by a functor so that lengths need not be materialised.
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

struct ArrayIn {
  const int* p;
  __device__ int operator()(long long i) const { return p[i]; }
};

struct TailLenIn {  // max(0, len(r) - K)
  const int* rowPtrs;
  int K;
  __device__ int operator()(long long i) const {
    const int len = rowPtrs[i + 1] - rowPtrs[i];
    return len > K ? len - K : 0;
  }
};

__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* sWarp) {
  // exclusive scan of one value per thread across a 256-thread block
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFullMask, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sWarp[w] = inc;
  __syncthreads();
  if (w == 0) {
    int s = lane < kScanThreads / 32 ? sWarp[lane] : 0;
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFullMask, si, off);
      if (lane >= off) si += o;
    }
    if (lane < kScanThreads / 32) sWarp[lane] = si - s;
    if (lane == kScanThreads / 32 - 1) sWarp[kScanThreads / 32] = si;
  }
  __syncthreads();
  const int res = inc - v + sWarp[w];
  *total = sWarp[kScanThreads / 32];
  __syncthreads();
  return res;
}

template <class In>
__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(In in, long long n, int* blockSums) {
  __shared__ int sWarp[kScanThreads / 32 + 1];
  const long long base = (long long)blockIdx.x * kScanTile + (long long)threadIdx.x * kScanItems;
  int s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) s += in(base + i);
  int total;
  block_exclusive_scan(s, &total, sWarp);
  if (threadIdx.x == 0) blockSums[blockIdx.x] = total;
}

// Single block: exclusive scan of nb block sums in chunks with a carry.
__global__ void __launch_bounds__(kScanThreads) k_scan_block_sums(int* sums, long long nb) {
  __shared__ int sWarp[kScanThreads / 32 + 1];
  int carry = 0;
  for (long long c = 0; c < nb; c += kScanTile) {
    const long long base = c + (long long)threadIdx.x * kScanItems;
    int v[kScanItems];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      v[i] = base + i < nb ? sums[base + i] : 0;
      s += v[i];
    }
    int total;
    int ex = block_exclusive_scan(s, &total, sWarp) + carry;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      if (base + i < nb) sums[base + i] = ex;
      ex += v[i];
    }
    carry += total;
  }
}

// In-place exclusive scan of a small array (n <= kSmallScan) by one block of
// 1024 threads, 16384 entries per pass: a thread holds 16 consecutive entries
// in registers (four 16-byte loads when the array is 16-byte aligned), scans
// them, the warp scans the thread totals with shuffles, one warp scans the 32
// warp totals through shared memory (two barriers per pass), and the thread
// writes its 16 results back. (Staging the pass through shared memory with 8
// consecutive entries per thread made 8-way bank conflicts: 10.5 us for
// 16384 entries, bound by the shared-memory pipe.)
constexpr int kSmallScanThreads = 1024;
constexpr int kSmallScanItems = 16;
constexpr int kSmallScanPass = kSmallScanThreads * kSmallScanItems;
__global__ void __launch_bounds__(kSmallScanThreads) k_scan_small(int* __restrict__ a, int n) {
  __shared__ int sWarp[kSmallScanThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const bool vec = (reinterpret_cast<uintptr_t>(a) & 15u) == 0;
  int carry = 0;
  for (int base0 = 0; base0 < n; base0 += kSmallScanPass) {
    const int first = base0 + threadIdx.x * kSmallScanItems;
    int v[kSmallScanItems];
    if (vec && first + kSmallScanItems <= n) {
#pragma unroll
      for (int q = 0; q < kSmallScanItems / 4; ++q) {
        const int4 c = reinterpret_cast<const int4*>(a + first)[q];
        v[4 * q] = c.x; v[4 * q + 1] = c.y; v[4 * q + 2] = c.z; v[4 * q + 3] = c.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kSmallScanItems; ++i) v[i] = first + i < n ? a[first + i] : 0;
    }
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kSmallScanItems; ++i) sum += v[i];
    int inc = sum;  // inclusive scan of the thread totals over the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFullMask, inc, off);
      if (lane >= off) inc += o;
    }
    if (lane == 31) sWarp[w] = inc;
    __syncthreads();
    if (w == 0) {
      int x = sWarp[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFullMask, x, off);
        if (lane >= off) x += o;
      }
      sWarp[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    int ex = carry + (w > 0 ? sWarp[w - 1] : 0) + inc - sum;
    const int total = sWarp[kSmallScanThreads / 32 - 1];
#pragma unroll
    for (int i = 0; i < kSmallScanItems; ++i) {
      const int t = v[i];
      v[i] = ex;
      ex += t;
    }
    if (vec && first + kSmallScanItems <= n) {
#pragma unroll
      for (int q = 0; q < kSmallScanItems / 4; ++q)
        reinterpret_cast<int4*>(a + first)[q] =
            make_int4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < kSmallScanItems; ++i)
        if (first + i < n) a[first + i] = v[i];
    }
    carry += total;
    __syncthreads();  // sWarp is reused by the next pass
  }
}

template <class In>
__global__ void __launch_bounds__(kScanThreads) k_scan_apply(In in, long long n, const int* blockOffs,
                                                             int* out) {
  __shared__ int sWarp[kScanThreads / 32 + 1];
  const long long base = (long long)blockIdx.x * kScanTile + (long long)threadIdx.x * kScanItems;
  int v[kScanItems];
  int s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = base + i < n ? in(base + i) : 0;
    s += v[i];
  }
  int total;
  int ex = block_exclusive_scan(s, &total, sWarp) + blockOffs[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if (base + i < n) out[base + i] = ex;
    ex += v[i];
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == kScanThreads - 1) out[n] = ex;
}

// out[0..n] = exclusive scan of in(0..n-1), out[n] = total. scratch holds
// scan_scratch_ints(n) ints.
template <class In>
cudaError_t exclusive_scan(In in, long long n, int* out, int* scratch, cudaStream_t s) {
  const long long nb = n > 0 ? (n + kScanTile - 1) / kScanTile : 1;
  k_scan_reduce<In><<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, scratch);
  k_scan_block_sums<<<1, kScanThreads, 0, s>>>(scratch, nb);
  k_scan_apply<In><<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, scratch, out);
  note_launches(3);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// JDS: stable least-significant-digit radix sort of the rows on the key
// maxLen - len (ascending key = longest row first; equal lengths keep their
// original order because every pass is stable).
// ---------------------------------------------------------------------------
constexpr int kSortThreads = 256;
constexpr int kSortRounds = 8;
constexpr int kSortTile = kSortThreads * kSortRounds;  // rows per tile
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr long long kSmallScan = 32768;  // histograms up to this size: one-block scan

// Key sources of the radix sort: pass 0 derives (key, item) from the input,
// later passes read the previous pass's output (keysIn/valsIn).
struct SortIn {
  // pass 0 reads keys from rowPtrs (items are the rows themselves)
  const int* rowPtrs;
  int maxLen;
  const int* keysIn;  // later passes
  const int* valsIn;
  __device__ void get(long long i, int& key, int& val) const {
    if (keysIn) {
      key = keysIn[i];
      val = valsIn[i];
    } else {
      key = maxLen - (rowPtrs[i + 1] - rowPtrs[i]);
      val = (int)i;
    }
  }
};

struct ChunkKeyIn {
  // pass 0: key = column chunk of nonzero i (items are the nonzeros)
  const int* colIdx;
  int B;
  const int* keysIn;
  const int* valsIn;
  __device__ void get(long long i, int& key, int& val) const {
    if (keysIn) {
      key = keysIn[i];
      val = valsIn[i];
    } else {
      key = colIdx[i] / B;
      val = (int)i;
    }
  }
};

// Per tile, count keys per digit; hist is digit-major: hist[d * nTiles + tile].
// All of a thread's keys are loaded before any is counted; equal digits in a
// warp are counted with one shared atomic (warp match).
template <class In>
__global__ void __launch_bounds__(kSortThreads) k_radix_hist(In in, int R, int shift, int nBuckets,
                                                             int nTiles, int* __restrict__ hist) {
  __shared__ int sCount[kRadix];
  for (int d = threadIdx.x; d < nBuckets; d += kSortThreads) sCount[d] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long base = (long long)blockIdx.x * kSortTile;
  int key[kSortRounds];
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const long long i = base + rd * kSortThreads + threadIdx.x;
    int val;
    key[rd] = 0;
    if (i < R) in.get(i, key[rd], val);
  }
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const long long i = base + rd * kSortThreads + threadIdx.x;
    const int digit = i < R ? (key[rd] >> shift) & (nBuckets - 1) : kRadix;
    const unsigned peers = __match_any_sync(kFullMask, digit);
    if (digit < kRadix && lane == __ffs(peers) - 1) atomicAdd(&sCount[digit], __popc(peers));
  }
  __syncthreads();
  for (int d = threadIdx.x; d < nBuckets; d += kSortThreads)
    hist[(long long)d * nTiles + blockIdx.x] = sCount[d];
}

// Stable scatter. Warp w of a tile owns the tile's items [256w, 256w + 256)
// (8 rounds of 32 consecutive items, all loaded before the first is used).
// Rank of an item among equal digits = tile offset (from the scanned
// histogram) + items of that digit in earlier warps + earlier rounds of this
// warp + earlier lanes of this round (warp match). Each warp first counts its
// own digits in a warp-private shared-memory row, one pass over the digits
// turns the rows into starting positions, and each warp then walks its items
// again, advancing its private cursors: two block barriers per tile. The
// last pass also writes the inverse permutation (invOut[item] = sorted
// position) when invOut is given; keysOut may be null when the sorted keys
// are not needed.
template <class In>
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter(In in, int R, int shift,
                                                                int nBuckets, int nTiles,
                                                                const int* __restrict__ offs,
                                                                int* __restrict__ keysOut,
                                                                int* __restrict__ valsOut,
                                                                int* __restrict__ invOut) {
  constexpr int kWarps = kSortThreads / 32;
  constexpr int kPerWarp = kSortTile / kWarps;  // = 32 * kSortRounds
  __shared__ int sCur[kWarps][kRadix];          // counts, then running positions
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int d = lane; d < nBuckets; d += 32) sCur[w][d] = 0;
  const long long wbase = (long long)blockIdx.x * kSortTile + (long long)w * kPerWarp;
  int key[kSortRounds], val[kSortRounds], digit[kSortRounds];
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const long long i = wbase + rd * 32 + lane;
    key[rd] = 0;
    val[rd] = 0;
    if (i < R) in.get(i, key[rd], val[rd]);
    digit[rd] = i < R ? (key[rd] >> shift) & (nBuckets - 1) : kRadix;  // kRadix: no one shares
  }
  __syncwarp();
  // this warp's count of every digit
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const unsigned peers = __match_any_sync(kFullMask, digit[rd]);
    if (digit[rd] < kRadix && lane == __ffs(peers) - 1) sCur[w][digit[rd]] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // counts -> where each warp's items of each digit start
  for (int d = threadIdx.x; d < nBuckets; d += kSortThreads) {
    int run = offs[(long long)d * nTiles + blockIdx.x];
#pragma unroll
    for (int q = 0; q < kWarps; ++q) {
      const int cnt = sCur[q][d];
      sCur[q][d] = run;
      run += cnt;
    }
  }
  __syncthreads();
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const int dg = digit[rd];
    const unsigned peers = __match_any_sync(kFullMask, dg);
    const bool valid = dg < kRadix;
    const int start = valid ? sCur[w][dg] : 0;
    __syncwarp();
    if (valid) {
      const int pos = start + __popc(peers & lanemask_lt());
      if (keysOut) keysOut[pos] = key[rd];
      valsOut[pos] = val[rd];
      if (invOut) invOut[val[rd]] = pos;
      if (lane == __ffs(peers) - 1) sCur[w][dg] = start + __popc(peers);
    }
    __syncwarp();
  }
}

// Single-pass form (every key below kSortMaxBuckets, at most kSortMaxGroups
// groups of tiles):
// two kernels instead of five (the histogram, three scan kernels for a large
// histogram, the scatter), and no block waits on another. k_radix_count1
// writes each tile's digit counts (tile-major) and adds them into the sums of
// its group of kSortGroup tiles (zeroed before the launch). k_radix_scatter1,
// a programmatic dependent launch, loads its keys and counts its warps' digits
// while the counts finish, then finds its tile's start for every digit by
// itself: the digit's start (an exclusive scan over the digits of the group
// sums' totals) plus the groups before its group plus the tiles before it in
// its group, read by all 256 threads (256 / nBuckets per digit). It then
// scatters as k_radix_scatter does.
constexpr int kSortGroup = 32;
// bounds of the single-pass form: at most kSortMaxGroups groups (2048 tiles,
// 4,194,304 items) and kSortMaxBuckets digits, so that each thread's share of
// the prefix reads is a few loads issued together; larger sorts (the
// x-blocked list's chunk sort, with thousands of tiles) take the general form
constexpr int kSortMaxGroups = 64;
constexpr int kSortMaxBuckets = 32;
__host__ __device__ inline long long sort_groups(long long nTiles) {
  return (nTiles + kSortGroup - 1) / kSortGroup;
}

template <class In>
__global__ void __launch_bounds__(kSortThreads) k_radix_count1(In in, int R, int nBuckets,
                                                               int* __restrict__ tileHist,
                                                               int* __restrict__ groupSum) {
  grid_dependency_trigger();  // the scatter may load its keys meanwhile
  __shared__ int sCount[kRadix];
  for (int d = threadIdx.x; d < nBuckets; d += kSortThreads) sCount[d] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long base = (long long)blockIdx.x * kSortTile;
  int key[kSortRounds];
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const long long i = base + rd * kSortThreads + threadIdx.x;
    int val;
    key[rd] = 0;
    if (i < R) in.get(i, key[rd], val);
  }
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const long long i = base + rd * kSortThreads + threadIdx.x;
    const int digit = i < R ? key[rd] & (nBuckets - 1) : kRadix;
    const unsigned peers = __match_any_sync(kFullMask, digit);
    if (digit < kRadix && lane == __ffs(peers) - 1) atomicAdd(&sCount[digit], __popc(peers));
  }
  __syncthreads();
  int* grp = groupSum + (long long)(blockIdx.x / kSortGroup) * nBuckets;
  for (int d = threadIdx.x; d < nBuckets; d += kSortThreads) {
    const int c = sCount[d];
    tileHist[(long long)blockIdx.x * nBuckets + d] = c;
    if (c) atomicAdd(grp + d, c);
  }
}

template <class In>
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter1(
    In in, int R, int nBuckets, int nTiles, const int* __restrict__ tileHist,
    const int* __restrict__ groupSum, int* __restrict__ keysOut, int* __restrict__ valsOut,
    int* __restrict__ invOut) {
  constexpr int kWarps = kSortThreads / 32;
  constexpr int kPerWarp = kSortTile / kWarps;  // = 32 * kSortRounds
  __shared__ int sCur[kWarps][kRadix];          // counts, then running positions
  __shared__ int sBefore[kSortThreads], sTotal[kSortThreads];
  __shared__ int sStart[kRadix];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int d = lane; d < nBuckets; d += 32) sCur[w][d] = 0;
  const long long wbase = (long long)blockIdx.x * kSortTile + (long long)w * kPerWarp;
  int key[kSortRounds], val[kSortRounds], digit[kSortRounds];
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const long long i = wbase + rd * 32 + lane;
    key[rd] = 0;
    val[rd] = 0;
    if (i < R) in.get(i, key[rd], val[rd]);
    digit[rd] = i < R ? key[rd] & (nBuckets - 1) : kRadix;  // kRadix: no one shares
  }
  __syncwarp();
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const unsigned peers = __match_any_sync(kFullMask, digit[rd]);
    if (digit[rd] < kRadix && lane == __ffs(peers) - 1) sCur[w][digit[rd]] += __popc(peers);
    __syncwarp();
  }
  grid_dependency_wait();  // the counts are complete and visible
  // partial sums: thread (digit d, part p) takes the groups g = p mod P and the
  // tiles of its group before this one, t = p mod P
  const int P = kSortThreads / nBuckets;  // nBuckets: a power of two <= kRadix
  const int d = threadIdx.x % nBuckets, p = threadIdx.x / nBuckets;
  const int tile = blockIdx.x, myGroup = tile / kSortGroup;
  const int nGroups = (int)sort_groups(nTiles);
  // at most kSortMaxGroups / P group sums and kSortGroup / P tile counts per
  // thread (P >= kSortThreads / kSortMaxBuckets), all loaded together
  constexpr int kG = kSortMaxGroups / (kSortThreads / kSortMaxBuckets);
  constexpr int kT = kSortGroup / (kSortThreads / kSortMaxBuckets);
  int gv[kG], tv[kT];
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const int g = p + k * P;
    gv[k] = g < nGroups ? __ldcg(groupSum + (long long)g * nBuckets + d) : 0;
  }
#pragma unroll
  for (int k = 0; k < kT; ++k) {
    const int t = myGroup * kSortGroup + p + k * P;
    tv[k] = t < tile ? __ldcg(tileHist + (long long)t * nBuckets + d) : 0;
  }
  int before = 0, total = 0;
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    total += gv[k];
    if (p + k * P < myGroup) before += gv[k];
  }
#pragma unroll
  for (int k = 0; k < kT; ++k) before += tv[k];
  sBefore[threadIdx.x] = before;
  sTotal[threadIdx.x] = total;
  __syncthreads();
  if (threadIdx.x < nBuckets) {
    int b = 0, t = 0;
    for (int q = 1; q < P; ++q) {
      b += sBefore[q * nBuckets + threadIdx.x];
      t += sTotal[q * nBuckets + threadIdx.x];
    }
    sBefore[threadIdx.x] += b;
    sTotal[threadIdx.x] += t;
  }
  __syncthreads();
  // digit starts: exclusive scan of the totals (lane l takes nBuckets / 32
  // consecutive digits, or one)
  if (w == 0) {
    const int per = (nBuckets + 31) / 32;
    const int lo = lane * per;
    int own = 0;
    for (int k = 0; k < per && lo + k < nBuckets; ++k) own += sTotal[lo + k];
    int incl = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - own;
    for (int k = 0; k < per && lo + k < nBuckets; ++k) {
      const int v = sTotal[lo + k];
      sStart[lo + k] = run;
      run += v;
    }
  }
  __syncthreads();
  // counts -> where each warp's items of each digit start
  for (int dd = threadIdx.x; dd < nBuckets; dd += kSortThreads) {
    int run = sStart[dd] + sBefore[dd];
#pragma unroll
    for (int q = 0; q < kWarps; ++q) {
      const int cnt = sCur[q][dd];
      sCur[q][dd] = run;
      run += cnt;
    }
  }
  __syncthreads();
#pragma unroll
  for (int rd = 0; rd < kSortRounds; ++rd) {
    const int dg = digit[rd];
    const unsigned peers = __match_any_sync(kFullMask, dg);
    const bool valid = dg < kRadix;
    const int start = valid ? sCur[w][dg] : 0;
    __syncwarp();
    if (valid) {
      const int pos = start + __popc(peers & lanemask_lt());
      if (keysOut) keysOut[pos] = key[rd];
      valsOut[pos] = val[rd];
      if (invOut) invOut[val[rd]] = pos;
      if (lane == __ffs(peers) - 1) sCur[w][dg] = start + __popc(peers);
    }
    __syncwarp();
  }
}

// Diagonal widths from the sorted lengths: width(t) = #{s : len(s) > t}. With
// lengths non-increasing over s, width(t) = s+1 for t in [len(s+1), len(s)).
// (Used when some row is at least kExactLenBins long; otherwise iterPtr comes
// from the exact length histogram.)
__global__ void k_jds_widths(int R, int maxLen, const int* __restrict__ sortedKeys,
                             int* __restrict__ width) {
  const long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= R) return;
  const int len = maxLen - sortedKeys[s];
  const int next = s + 1 < R ? maxLen - sortedKeys[s + 1] : 0;
  for (int t = next; t < len; ++t) width[t] = (int)(s + 1);
}

// Jagged scatter, in sorted order: thread s takes sorted row s (original row
// perm[s]) and writes its entry t to iterPtr[t] + s. Rows are sorted longest
// first, so for every t the lanes of a warp that still have an entry are a
// prefix of the warp and their stores are contiguous (walking rows in their
// original order instead split a warp's stores wherever the length changed:
// 392 us per launch on the 27-point stencil). A thread copies the first
// kJdsCoop entries of its row. The longer rows are the first wLong sorted
// rows; their entries from kJdsCoop on are cut into segments of kJdsSeg,
// one segment per warp of the blocks after the first mainBlocks (a warp per
// long row would serialise the longest rows, which sit together). The first
// kJdsScatterSmem entries of iterPtr are staged in shared memory.
constexpr int kJdsScatterSmem = 1024;
constexpr int kJdsSeg = 1024;
// iterPtr passed by value when the host knows it and it is short (longest
// row below kIpArg): block 0 writes it to memory, every block reads it from
// its arguments. n = 0: iterPtr is already in memory.
constexpr int kIpArg = 256;
struct IterPtrArg {
  int n;
  int v[kIpArg];
};
template <class T>
__global__ void __launch_bounds__(256) k_jds_scatter(int R, int maxLen, int mainBlocks,
                                                     int wLong, int nSegs,
                                                     const int* __restrict__ rowPtrs,
                                                     const int* __restrict__ colIdx,
                                                     const T* __restrict__ value,
                                                     const int* __restrict__ perm,
                                                     int* __restrict__ iterPtr,
                                                     const __grid_constant__ IterPtrArg ipArg,
                                                     int* __restrict__ jdsCol,
                                                     T* __restrict__ jdsVal) {
  __shared__ int sIp[kJdsScatterSmem];
  const int nIp = maxLen < kJdsScatterSmem ? maxLen : kJdsScatterSmem;
  if (ipArg.n > 0) {  // n = maxLen + 1 <= kIpArg
    for (int t = threadIdx.x; t < nIp; t += blockDim.x) sIp[t] = ipArg.v[t];
    if (blockIdx.x == 0)
      for (int t = threadIdx.x; t < ipArg.n; t += blockDim.x) iterPtr[t] = ipArg.v[t];
  } else {
    for (int t = threadIdx.x; t < nIp; t += blockDim.x) sIp[t] = iterPtr[t];
  }
  __syncthreads();
  if ((int)blockIdx.x < mainBlocks) {
    const long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // sorted row
    if (s >= R) return;
    const int r = perm[s];
    const int a = rowPtrs[r];
    const int len = rowPtrs[r + 1] - a;
    const int lim = len < kJdsCoop ? len : kJdsCoop;
    for (int t = 0; t < lim; ++t) {
      const long long o = (long long)sIp[t] + s;
      jdsCol[o] = colIdx[a + t];
      jdsVal[o] = value[a + t];
    }
  } else {
    // one segment of one long row per warp, one entry per lane
    const long long item = (long long)(blockIdx.x - mainBlocks) * (blockDim.x >> 5) +
                           (threadIdx.x >> 5);
    const long long s = item / nSegs;
    if (s >= wLong) return;
    const int r = perm[s];
    const int a = rowPtrs[r];
    const int len = rowPtrs[r + 1] - a;
    const long long t0 = kJdsCoop + (item % nSegs) * (long long)kJdsSeg;
    const long long t1 = min(t0 + kJdsSeg, (long long)len);
    for (long long t = t0 + (threadIdx.x & 31); t < t1; t += 32) {
      const int ip = t < kJdsScatterSmem ? sIp[t] : __ldg(iterPtr + t);
      const long long o = (long long)ip + s;
      jdsCol[o] = colIdx[a + t];
      jdsVal[o] = value[a + t];
    }
  }
}

// Warp-staged jagged scatter for a longest row in [kStageMinK, kStageMaxK<T>]
// (the 27-point stencil): warp w takes sorted rows s0 .. s0 + 31 and copies
// their entries into its shared buffers, then each lane writes its own row's
// entries to iterPtr[t] + s from there (reading them straight from global
// memory, a warp's load of the rows' t-th entries touches a sector per lane).
// When the 32 rows are consecutive original rows (the sort is stable, so a
// run of rows of one length stays together), their entries are one
// contiguous range, staged as for the ELL scatter (warp_stage_entries:
// 16-byte asynchronous copies). Otherwise the warp copies row by row, lane t
// taking entry t of the row (asynchronous 4- or 8-byte copies, coalesced
// within the row), rows maxLen rounded up to an odd count apart so that the
// lanes' reads fall in different banks. Either way all copies are in flight
// before one wait.
template <class T, bool VEC>
__global__ void __launch_bounds__(32 * kStageWarps) k_jds_scatter_staged(
    int R, int maxLen, const int* __restrict__ rowPtrs, const int* __restrict__ colIdx,
    const T* __restrict__ value, const int* __restrict__ perm, int* __restrict__ iterPtr,
    const __grid_constant__ IterPtrArg ipArg, int* __restrict__ jdsCol, T* __restrict__ jdsVal) {
  __shared__ int sIp[kStageMaxK<float>];
  extern __shared__ int4 sRaw[];
  if (ipArg.n > 0) {  // n = maxLen + 1
    for (int t = threadIdx.x; t < maxLen; t += blockDim.x) sIp[t] = ipArg.v[t];
    if (blockIdx.x == 0)
      for (int t = threadIdx.x; t < ipArg.n; t += blockDim.x) iterPtr[t] = ipArg.v[t];
  } else {
    for (int t = threadIdx.x; t < maxLen; t += blockDim.x) sIp[t] = iterPtr[t];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stride = maxLen | 1;
  const int cap = 32 * stride + 8;  // a multiple of 4 when stride is odd plus 8: see below
  int* sCol = reinterpret_cast<int*>(sRaw) + warp * cap;
  T* sVal = reinterpret_cast<T*>(reinterpret_cast<int*>(sRaw) + kStageWarps * cap) + warp * cap;
  const long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // sorted row
  const long long s0 = s - lane;
  if (s0 >= R) return;  // warp-uniform
  int r = -1, a = 0, len = 0;
  if (s < R) {
    r = perm[s];
    a = rowPtrs[r];
    len = min(rowPtrs[r + 1] - a, maxLen);
  }
  const int r0 = __shfl_sync(kFullMask, r, 0);
  const int nRows = (int)min(32LL, (long long)R - s0);
  // consecutive original rows: one contiguous range [a0, a1)
  const bool run = __all_sync(kFullMask, lane >= nRows || r == r0 + lane) && VEC;
  int off;
  if (run) {
    const int a0 = __shfl_sync(kFullMask, a, 0);
    const int a1 = __ldg(rowPtrs + r0 + nRows);  // a1 - a0 <= 32 * maxLen
    warp_stage_entries<T, true>(colIdx, value, a0, a1, lane, sCol, sVal);
    off = (int)(a - (a0 & ~3LL));
  } else {
    for (int j = 0; j < 32; ++j) {
      const int aj = __shfl_sync(kFullMask, a, j);
      const int lj = __shfl_sync(kFullMask, len, j);
      if (lane < lj) {
        cp_async_small<4>(sCol + j * stride + lane, colIdx + aj + lane);
        cp_async_small<(int)sizeof(T)>(sVal + j * stride + lane, value + aj + lane);
      }
    }
    cp_async_wait_all();
    off = lane * stride;
  }
  __syncwarp();
  if (s >= R) return;
  for (int t = 0; t < len; ++t) {
    const long long o = (long long)sIp[t] + s;
    jdsCol[o] = sCol[off + t];
    jdsVal[o] = sVal[off + t];
  }
}

}  // namespace

// Threads per block of the HYB tail copy (128 and 64 measured slower: the
// HYB conversion of the skewed matrix 197 / 218 / 209 us with 256 / 128 / 64
// threads).
constexpr int kTailBlock = 256;

size_t scan_scratch_ints(long long n) { return (size_t)((n + kScanTile - 1) / kScanTile + 1); }

cudaError_t launch_tail_scan(int R, int K, const int* rowPtrs, int* tailPtr, int* scratch,
                             cudaStream_t s) {
  return exclusive_scan(TailLenIn{rowPtrs, K}, (long long)R, tailPtr, scratch, s);
}

template <class T>
cudaError_t launch_hyb_tail_copy(int R, int K, const int* rowPtrs, const int* colIdx,
                                 const T* value, const int* tailPtr, int* cooRow,
                                 int* cooCol, T* cooVal, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const long long warps = ((long long)R + 31) / 32;
  const long long blocks = (warps * 32 + kTailBlock - 1) / kTailBlock;
  k_hyb_tail_copy<T><<<(unsigned)blocks, kTailBlock, 0, s>>>(R, K, rowPtrs, colIdx, value,
                                                             tailPtr, cooRow, cooCol, cooVal);
  note_launches(1);
  return cudaGetLastError();
}

// Scratch layout for the JDS build (all int32):
//   keysA[R] valsA[R] keysB[R] inv[R] hist[sort_hist_ints(nTiles)] scanScratch[...] width[maxLen]
// (hist: the tiles' digit counts, then the single-pass form's group sums)
long long sort_hist_ints(long long nTiles) {
  if (nTiles < 1) nTiles = 1;
  return (long long)kRadix * (nTiles + sort_groups(nTiles)) + 1;
}
size_t jds_sort_scratch_bytes(int R, int maxLen) {
  const long long nTiles = ((long long)R + kSortTile - 1) / kSortTile;
  const long long nh = (long long)kRadix * (nTiles > 0 ? nTiles : 1);
  const long long scanN = nh > maxLen ? nh : maxLen;
  const long long ints = 4LL * R + sort_hist_ints(nTiles) + (long long)scan_scratch_ints(scanN) +
                         maxLen + 16;
  return (size_t)ints * sizeof(int);
}

// Stable sort of the rows by length, longest first (LSD radix on maxLen - len
// with 8-bit digits): perm[s] = row at sorted position s, and, when invOut is
// given, inv[row] = s. The sorted keys are left in keysB when needKeys (else
// they are not written).
// Scratch (int32): keysA[R] valsA[R] keysB[R] inv[R] hist[sort_hist_ints(nTiles)] scan.
template <class In>
static cudaError_t radix_sort(In first, int R, int maxLen, int* perm, int* scratch,
                              bool needKeys, const int** sortedKeys, int** invOut,
                              int** scanScratchOut, cudaStream_t s) {
  const long long nTiles = ((long long)R + kSortTile - 1) / kSortTile;
  int* keysA = scratch;
  int* valsA = keysA + R;
  int* keysB = valsA + R;
  int* inv = keysB + R;
  int* hist = inv + R;
  int* scanScratch = hist + sort_hist_ints(nTiles);
  if (invOut) *invOut = inv;
  *scanScratchOut = scanScratch;
  int bits = 0;
  while (bits < 31 && (1LL << bits) <= maxLen) ++bits;
  const int passes = bits == 0 ? 1 : (bits + kRadixBits - 1) / kRadixBits;
  if (passes == 1 && (1 << bits) <= kSortMaxBuckets && sort_groups(nTiles) <= kSortMaxGroups) {
    const int nBuckets = 1 << bits;
    int* tileHist = hist;
    int* groupSum = hist + (long long)kRadix * nTiles;
    cudaError_t err = cudaMemsetAsync(groupSum, 0,
                                      sizeof(int) * (size_t)(sort_groups(nTiles) * nBuckets), s);
    if (err != cudaSuccess) return err;
    k_radix_count1<<<(unsigned)nTiles, kSortThreads, 0, s>>>(first, R, nBuckets, tileHist,
                                                             groupSum);
    note_launches(1);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nTiles);
    cfg.blockDim = dim3(kSortThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, k_radix_scatter1<In>, first, R, nBuckets, (int)nTiles,
                             (const int*)tileHist, (const int*)groupSum,
                             needKeys ? keysB : nullptr, perm, invOut ? inv : nullptr);
    note_launches(1);
    if (err != cudaSuccess) return err;
    *sortedKeys = keysB;
    return cudaGetLastError();
  }
  // Ping-pong so that the last pass writes perm (values) and keysB (keys).
  int* kBuf[2] = {keysA, keysB};
  int* vBuf[2] = {valsA, perm};
  int outSlot = (passes % 2 == 1) ? 1 : 0;
  const int* kIn = nullptr;
  const int* vIn = nullptr;
  cudaError_t err = cudaSuccess;
  for (int p = 0; p < passes; ++p) {
    In in = first;
    in.keysIn = kIn;
    in.valsIn = vIn;
    const int shift = p * kRadixBits;
    // only the buckets this pass's digit can take (the last digit may be narrower)
    const int digitBits = bits - shift < kRadixBits ? (bits - shift > 0 ? bits - shift : 0)
                                                     : kRadixBits;
    const int nBuckets = 1 << digitBits;
    const long long nhp = (long long)nBuckets * nTiles;
    k_radix_hist<<<(unsigned)nTiles, kSortThreads, 0, s>>>(in, R, shift, nBuckets, (int)nTiles,
                                                           hist);
    note_launches(1);
    if (nhp <= kSmallScan) {  // one block scans the whole histogram in place
      k_scan_small<<<1, kSmallScanThreads, 0, s>>>(hist, (int)nhp);
      note_launches(1);
    } else {
      err = exclusive_scan(ArrayIn{hist}, nhp, hist, scanScratch, s);
      if (err != cudaSuccess) return err;
    }
    const bool last = p == passes - 1;
    k_radix_scatter<<<(unsigned)nTiles, kSortThreads, 0, s>>>(
        in, R, shift, nBuckets, (int)nTiles, hist, (last && !needKeys) ? nullptr : kBuf[outSlot],
        vBuf[outSlot], (last && invOut) ? inv : nullptr);
    note_launches(1);
    kIn = kBuf[outSlot];
    vIn = vBuf[outSlot];
    outSlot ^= 1;
  }
  *sortedKeys = kIn;
  return cudaGetLastError();
}

static cudaError_t row_sort(int R, int maxLen, const int* rowPtrs, int* perm, int* scratch,
                            bool needKeys, const int** sortedKeys, int** invOut,
                            int** scanScratchOut, cudaStream_t s) {
  return radix_sort(SortIn{rowPtrs, maxLen, nullptr, nullptr}, R, maxLen, perm, scratch,
                    needKeys, sortedKeys, invOut, scanScratchOut, s);
}

template <class T>
cudaError_t launch_jds_build(int R, int maxLen, int wLong, const int* rowPtrs,
                             const int* colIdx, const T* value, int* perm, int* iterPtr,
                             int* jdsCol, T* jdsVal, void* scratch, const int* hostIterPtr,
                             cudaStream_t s) {
  if (R <= 0) {
    // iterPtr has maxLen + 1 = 1 entry
    return cudaMemsetAsync(iterPtr, 0, sizeof(int), s);
  }
  const long long nTiles = ((long long)R + kSortTile - 1) / kSortTile;
  const long long nh = (long long)kRadix * nTiles;
  const long long scanN = nh > maxLen ? nh : maxLen;
  const int* sortedKeys = nullptr;
  int* scanScratch = nullptr;
  // the scatter walks rows in sorted order (perm): no inverse permutation
  cudaError_t err = row_sort(R, maxLen, rowPtrs, perm, static_cast<int*>(scratch),
                             hostIterPtr == nullptr, &sortedKeys, nullptr, &scanScratch, s);
  if (err != cudaSuccess) return err;
  int* width = scanScratch + scan_scratch_ints(scanN);
  if (maxLen > 0) {
    IterPtrArg ipArg;
    ipArg.n = 0;
    if (hostIterPtr && maxLen + 1 <= kIpArg) {
      // known exactly on the host from the length histogram: kernel argument
      ipArg.n = maxLen + 1;
      for (int t = 0; t <= maxLen; ++t) ipArg.v[t] = hostIterPtr[t];
    } else if (hostIterPtr) {
      err = cudaMemcpyAsync(iterPtr, hostIterPtr, sizeof(int) * ((size_t)maxLen + 1),
                            cudaMemcpyHostToDevice, s);
      if (err != cudaSuccess) return err;
    } else {
      k_jds_widths<<<(unsigned)(((long long)R + 255) / 256), 256, 0, s>>>(R, maxLen, sortedKeys,
                                                                         width);
      note_launches(1);
      err = exclusive_scan(ArrayIn{width}, (long long)maxLen, iterPtr, scanScratch, s);
      if (err != cudaSuccess) return err;
    }
    // a thread per sorted row, then a warp per kJdsSeg-entry segment of the
    // wLong rows longer than kJdsCoop
    const long long mainBlocks = ((long long)R + 255) / 256;
    const int nSegs = maxLen > kJdsCoop ? (maxLen - kJdsCoop + kJdsSeg - 1) / kJdsSeg : 1;
    const long long tailBlocks = ((long long)wLong * nSegs + 7) / 8;
    if (maxLen >= kStageMinK && maxLen <= kStageMaxK<T>) {  // wLong = 0: no row past kJdsCoop
      constexpr int threads = 32 * kStageWarps;
      const unsigned blocks = (unsigned)(((long long)R + threads - 1) / threads);
      const size_t smem =
          (size_t)kStageWarps * (32 * (size_t)(maxLen | 1) + 8) * (sizeof(int) + sizeof(T));
      if (aligned16(colIdx) && aligned16(value))
        k_jds_scatter_staged<T, true><<<blocks, threads, smem, s>>>(
            R, maxLen, rowPtrs, colIdx, value, perm, iterPtr, ipArg, jdsCol, jdsVal);
      else
        k_jds_scatter_staged<T, false><<<blocks, threads, smem, s>>>(
            R, maxLen, rowPtrs, colIdx, value, perm, iterPtr, ipArg, jdsCol, jdsVal);
      note_launches(1);
      return cudaGetLastError();
    }
    k_jds_scatter<T><<<(unsigned)(mainBlocks + tailBlocks), 256, 0, s>>>(
        R, maxLen, (int)mainBlocks, wLong, nSegs, rowPtrs, colIdx, value, perm, iterPtr, ipArg,
        jdsCol, jdsVal);
    note_launches(1);
  } else {
    err = cudaMemsetAsync(iterPtr, 0, sizeof(int), s);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Sectioned ELL ("Regularized Formats ...", section "JDS format", variant
// paragraph): the rows sorted as for JDS, cut into sections of S sorted rows,
// each section an ELL padded to its own longest row, column-major inside the
// section: slot t of the j-th row of section k at secPtr[k] + t*h_k + j.
// ---------------------------------------------------------------------------
// the row sort's scratch, then the scratch of the scan of section sizes
size_t sell_scratch_bytes(int R, int maxLen, long long nsec) {
  return jds_sort_scratch_bytes(R, maxLen) + sizeof(int) * (size_t)scan_scratch_ints(nsec);
}

struct SellSlotsIn {  // slots of section k: h_k * length of its first sorted row
  const int* rowPtrs;
  const int* perm;
  int R, S;
  __device__ int operator()(long long k) const {
    const long long s0 = k * S;
    const int h = R - s0 < S ? (int)(R - s0) : S;
    const int r = perm[s0];
    return h * (rowPtrs[r + 1] - rowPtrs[r]);
  }
};

cudaError_t launch_sell_offsets(int R, int S, int maxLen, long long nsec, const int* rowPtrs,
                                const int* perm, int* secPtr, void* scratch, cudaStream_t s) {
  if (nsec <= 0) return cudaMemsetAsync(secPtr, 0, sizeof(int), s);
  int* scanScratch = reinterpret_cast<int*>(static_cast<char*>(scratch) +
                                            jds_sort_scratch_bytes(R, maxLen));
  return exclusive_scan(SellSlotsIn{rowPtrs, perm, R, S}, nsec, secPtr, scanScratch, s);
}

cudaError_t launch_sell_sort(int R, int maxLen, const int* rowPtrs, int* perm, void* scratch,
                             cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const int* sortedKeys = nullptr;
  int* inv = nullptr;
  int* scanScratch = nullptr;
  return row_sort(R, maxLen, rowPtrs, perm, static_cast<int*>(scratch), false, &sortedKeys,
                  &inv, &scanScratch, s);
}

// width of section k = length of its first sorted row
__global__ void k_sell_widths(int R, int S, int nsec, const int* __restrict__ rowPtrs,
                              const int* __restrict__ perm, int* __restrict__ widths) {
  const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= nsec) return;
  const int r = perm[k * S];
  widths[k] = rowPtrs[r + 1] - rowPtrs[r];
}

cudaError_t launch_sell_widths(int R, int S, int nsec, const int* rowPtrs, const int* perm,
                               int* widths, cudaStream_t s) {
  if (nsec <= 0) return cudaSuccess;
  k_sell_widths<<<(unsigned)(((long long)nsec + 255) / 256), 256, 0, s>>>(R, S, nsec, rowPtrs,
                                                                         perm, widths);
  note_launches(1);
  return cudaGetLastError();
}

// Row-side scatter: original row r (sorted position inv[r], section k, row j
// of the section) writes its w_k slots, real entries then padding (column -1,
// value +0.0f). A thread writes the first kJdsCoop slots; the warp then writes
// each wider section's remaining slots of its rows together, one per lane.
template <class T>
__global__ void __launch_bounds__(256) k_sell_scatter(int R, int S, const int* __restrict__ rowPtrs,
                                                      const int* __restrict__ colIdx,
                                                      const T* __restrict__ value,
                                                      const int* __restrict__ inv,
                                                      const int* __restrict__ secPtr,
                                                      int cap, int* __restrict__ sellCol,
                                                      T* __restrict__ sellVal) {
  const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  int a = 0, len = 0, w = 0, h = 1, j = 0, base = 0;
  if (r < R) {
    a = rowPtrs[r];
    len = rowPtrs[r + 1] - a;
    const int sidx = inv[r];
    const int k = sidx / S;
    j = sidx - k * S;
    h = min(S, R - k * S);
    base = secPtr[k];
    const int end = secPtr[k + 1];
    w = end <= cap ? (end - base) / h : 0;  // offsets past the arrays: write nothing
    const int lim = w < kJdsCoop ? w : kJdsCoop;
    for (int t = 0; t < lim; ++t) {
      const long long o = (long long)base + (long long)t * h + j;
      const bool real = t < len;
      sellCol[o] = real ? colIdx[a + t] : -1;
      sellVal[o] = real ? value[a + t] : T(0);
    }
  }
  unsigned wide = __ballot_sync(kFullMask, w > kJdsCoop);
  while (wide) {
    const int src = __ffs(wide) - 1;
    wide &= wide - 1;
    const int la = __shfl_sync(kFullMask, a, src);
    const int ll = __shfl_sync(kFullMask, len, src);
    const int lw = __shfl_sync(kFullMask, w, src);
    const int lh = __shfl_sync(kFullMask, h, src);
    const int lj = __shfl_sync(kFullMask, j, src);
    const int lb = __shfl_sync(kFullMask, base, src);
    for (long long t = kJdsCoop + lane; t < lw; t += 32) {  // 64-bit: lw may be near INT32_MAX
      const long long o = (long long)lb + t * lh + lj;
      const bool real = t < ll;
      sellCol[o] = real ? colIdx[la + t] : -1;
      sellVal[o] = real ? value[la + t] : T(0);
    }
  }
}

// Warp-staged form for a longest row of kStageMinK to kStageMaxK entries
// (every section at most that wide, below kJdsCoop: no cooperative part): a
// warp's 32 consecutive original rows are one contiguous CSR range, copied
// into its shared memory with asynchronous 16-byte copies
// (warp_stage_entries), then each lane writes its row's slots from there, as
// k_csr_to_ell_staged does. A warp whose rows hold more than 32 * K entries
// reads directly.
template <class T, bool VEC>
__global__ void __launch_bounds__(32 * kStageWarps) k_sell_scatter_staged(
    int R, int S, int K, const int* __restrict__ rowPtrs, const int* __restrict__ colIdx,
    const T* __restrict__ value, const int* __restrict__ inv, const int* __restrict__ secPtr,
    int cap, int* __restrict__ sellCol, T* __restrict__ sellVal) {
  extern __shared__ int4 sRaw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bufCap = 32 * K + 8;  // a multiple of 4: every warp's buffers start 16-byte aligned
  int* sCol = reinterpret_cast<int*>(sRaw) + warp * bufCap;
  T* sVal = reinterpret_cast<T*>(reinterpret_cast<int*>(sRaw) + kStageWarps * bufCap) +
            warp * bufCap;
  const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long w0 = r - lane;  // the warp's first row
  if (w0 >= R) return;            // warp-uniform
  const long long wEnd = w0 + 32 < R ? w0 + 32 : R;
  const int a0 = __ldg(rowPtrs + w0);
  const int a1 = __ldg(rowPtrs + wEnd);
  int a = 0, len = 0, w = 0, h = 1, j = 0, base = 0;
  if (r < R) {
    a = __ldg(rowPtrs + r);
    len = __ldg(rowPtrs + r + 1) - a;
    const int sidx = inv[r];
    const int k = sidx / S;
    j = sidx - k * S;
    h = min(S, R - k * S);
    base = secPtr[k];
    const int end = secPtr[k + 1];
    w = end <= cap ? (end - base) / h : 0;  // offsets past the arrays: write nothing
  }
  const bool staged = (long long)a1 - a0 <= 32LL * K;  // warp-uniform
  if (staged) warp_stage_entries<T, VEC>(colIdx, value, a0, a1, lane, sCol, sVal);
  __syncwarp();
  if (r >= R) return;
  const int off = (int)(a - (a0 & ~3LL));
  for (int t = 0; t < w; ++t) {
    const long long o = (long long)base + (long long)t * h + j;
    int c = -1;
    T v = T(0);
    if (t < len) {
      c = staged ? sCol[off + t] : colIdx[a + t];
      v = staged ? sVal[off + t] : value[a + t];
    }
    sellCol[o] = c;
    sellVal[o] = v;
  }
}

template <class T>
cudaError_t launch_sell_scatter(int R, int S, int maxLen, const int* rowPtrs, const int* colIdx,
                                const T* value, const void* scratch, const int* secPtr,
                                int slots, int* sellCol, T* sellVal, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const int* inv = static_cast<const int*>(scratch) + 3LL * R;  // row_sort's layout
  if (maxLen >= kStageMinK && maxLen <= kStageMaxK<T>) {
    constexpr int threads = 32 * kStageWarps;
    const unsigned blocks = (unsigned)(((long long)R + threads - 1) / threads);
    const size_t smem = warp_stage_smem<T>(maxLen);
    if (aligned16(colIdx) && aligned16(value))
      k_sell_scatter_staged<T, true><<<blocks, threads, smem, s>>>(
          R, S, maxLen, rowPtrs, colIdx, value, inv, secPtr, slots, sellCol, sellVal);
    else
      k_sell_scatter_staged<T, false><<<blocks, threads, smem, s>>>(
          R, S, maxLen, rowPtrs, colIdx, value, inv, secPtr, slots, sellCol, sellVal);
    note_launches(1);
    return cudaGetLastError();
  }
  k_sell_scatter<T><<<(unsigned)(((long long)R + 255) / 256), 256, 0, s>>>(
      R, S, rowPtrs, colIdx, value, inv, secPtr, slots, sellCol, sellVal);
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// x-blocked list ("Introduction to sparse computing and performance
// bottleneck location", section "Building the problem framework": split x
// into chunks, a thread block handles only the nonzeros whose columns fall in
// one chunk). Chunk c (columns [cB, (c+1)B)) holds its nonzeros in CSR order
// from chunkPtr[c]: row, 16-bit local column, value; padded to 4 entries.
// Build: per-chunk counts, the unpadded and padded chunk starts (scans), a
// stable radix sort of the nonzeros by chunk (rank of each nonzero), then a
// scatter in CSR order and the padding.
// ---------------------------------------------------------------------------
constexpr int kXbCountThreads = 256;
constexpr int kXbSmemBins = 8192;

__global__ void __launch_bounds__(kXbCountThreads) k_xb_count(int Z, int B, int nch,
                                                              const int* __restrict__ colIdx,
                                                              int* __restrict__ cnt) {
  __shared__ int sCnt[kXbSmemBins];
  const bool local = nch <= kXbSmemBins;
  if (local) {
    for (int c = threadIdx.x; c < nch; c += blockDim.x) sCnt[c] = 0;
    __syncthreads();
  }
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < Z;
       k += (long long)gridDim.x * blockDim.x) {
    const int c = colIdx[k] / B;
    if (local)
      atomicAdd(&sCnt[c], 1);
    else
      atomicAdd(cnt + c, 1);
  }
  if (local) {
    __syncthreads();
    for (int c = threadIdx.x; c < nch; c += blockDim.x)
      if (sCnt[c]) atomicAdd(cnt + c, sCnt[c]);
  }
}

struct Pad4In {  // chunk sizes rounded up to 4 entries
  const int* p;
  __device__ int operator()(long long i) const { return (p[i] + 3) & ~3; }
};

template <class T>
__global__ void __launch_bounds__(256) k_xb_scatter(int Z, int B, const int* __restrict__ colIdx,
                                                    const T* __restrict__ value,
                                                    const int* __restrict__ rowIdx,
                                                    const int* __restrict__ inv,
                                                    const int* __restrict__ ustart,
                                                    const int* __restrict__ chunkPtr,
                                                    int* __restrict__ xbRow,
                                                    unsigned short* __restrict__ xbCol,
                                                    T* __restrict__ xbVal) {
  const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= Z) return;
  const int col = colIdx[k];
  const int c = col / B;
  const long long p = (long long)chunkPtr[c] + (inv[k] - ustart[c]);
  xbRow[p] = rowIdx[k];
  xbCol[p] = (unsigned short)(col - c * B);
  xbVal[p] = value[k];
}

template <class T>
__global__ void k_xb_pad(int nch, const int* __restrict__ cnt, const int* __restrict__ chunkPtr,
                         int* __restrict__ xbRow, unsigned short* __restrict__ xbCol,
                         T* __restrict__ xbVal) {
  const long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= nch) return;
  for (long long i = (long long)chunkPtr[c] + cnt[c]; i < chunkPtr[c + 1]; ++i) {
    xbRow[i] = -1;
    xbCol[i] = 0;
    xbVal[i] = T(0);
  }
}

// Tiled build, for at most kXbTileChunks chunks: tiles of kXbTile consecutive
// nonzeros. (1) k_xb_tile_count: each tile's nonzeros per chunk, chunk-major
// (tileCnt[c * nTiles + t]); a thread counts its 8 consecutive entries in runs
// of equal chunk (a row's columns ascend) and adds each run with one shared
// atomic. (2) An exclusive scan of tileCnt: tile t's first position among
// chunk c's nonzeros, unpadded. (3) k_xb_chunk_ptr: chunk sizes and their
// padded starts. (4) k_xb_tile_scatter: each tile ranks its entries by chunk
// (stable: peer masks per 32 entries, warps in order), sorts them by chunk in
// shared memory, and writes every chunk's run of entries contiguously. The
// rows come from the CSR chunk records (no expanded row array). The earlier
// build sorted every nonzero by chunk with the general radix sort and then
// scattered each one by itself (a store instruction's 32 lanes on up to 32
// chunks): 1.09 ms on the skewed rows' 30.6M nonzeros and 1.63 ms on the
// 27-point stencil.
constexpr int kXbTile = 2048;
constexpr int kXbTileThreads = 256;

// col / B without a division: with M = ceil(2^64 / B), the high 64 bits of
// col * M are col / B + col * e / 2^64 for some e in [0, 1), and col < 2^31
// keeps that excess below 2^-33, under the 1/B gap to the next integer
// (B < 2^17). B = 1 is passed as M = 0.
struct ChunkDiv {
  unsigned long long m;
  int b;
  __device__ int operator()(int col) const {
    return m ? (int)__umul64hi((unsigned long long)(unsigned)col, m) : col;
  }
};
inline ChunkDiv chunk_div(int B) {
  ChunkDiv d;
  d.b = B;
  d.m = B <= 1 ? 0ull : (~0ull) / (unsigned long long)B + 1ull;  // ceil(2^64 / B), B > 1
  return d;
}
constexpr int kXbTileRounds = kXbTile / kXbTileThreads;  // 8
static_assert(kXbTileChunks <= 256, "chunk ids are kept in one byte");

template <bool VEC>
__global__ void __launch_bounds__(kXbTileThreads) k_xb_tile_count(int Z, ChunkDiv div, int nch,
                                                                  int nTiles,
                                                                  const int* __restrict__ colIdx,
                                                                  int* __restrict__ tileCnt) {
  __shared__ int sCnt[kXbTileChunks];
  for (int c = threadIdx.x; c < nch; c += kXbTileThreads) sCnt[c] = 0;
  const long long k0 = (long long)blockIdx.x * kXbTile + (long long)threadIdx.x * kXbTileRounds;
  int cols[kXbTileRounds];
  if (VEC && k0 + kXbTileRounds <= Z) {  // 16-byte aligned: tiles start on multiples of 2048
    const int4 a = ld_stream(reinterpret_cast<const int4*>(colIdx + k0));
    const int4 b = ld_stream(reinterpret_cast<const int4*>(colIdx + k0) + 1);
    cols[0] = a.x; cols[1] = a.y; cols[2] = a.z; cols[3] = a.w;
    cols[4] = b.x; cols[5] = b.y; cols[6] = b.z; cols[7] = b.w;
  } else {
#pragma unroll
    for (int e = 0; e < kXbTileRounds; ++e)
      cols[e] = k0 + e < Z ? ld_stream(colIdx + k0 + e) : 0;
  }
  __syncthreads();
  int cur = -1, run = 0;
#pragma unroll
  for (int e = 0; e < kXbTileRounds; ++e) {
    const long long k = k0 + e;
    if (k < Z) {
      const int c = div(cols[e]);
      if (c != cur) {
        if (run) atomicAdd(&sCnt[cur], run);
        cur = c;
        run = 0;
      }
      ++run;
    }
  }
  if (run) atomicAdd(&sCnt[cur], run);
  __syncthreads();
  for (int c = threadIdx.x; c < nch; c += kXbTileThreads)
    tileCnt[(long long)c * nTiles + blockIdx.x] = sCnt[c];
}

// One block: cnt[c] from the scanned tile counts (start of chunk c's first
// tile to the next chunk's), chunkPtr = exclusive scan of cnt rounded up to 4.
__global__ void __launch_bounds__(kScanThreads) k_xb_chunk_ptr(int Z, int nch, int nTiles,
                                                               const int* __restrict__ tileOff,
                                                               int* __restrict__ cnt,
                                                               int* __restrict__ chunkPtr) {
  __shared__ int sWarp[kScanThreads / 32 + 1];
  const int c = threadIdx.x;  // nch <= kXbTileChunks <= kScanThreads
  int padded = 0;
  if (c < nch) {
    const int a = tileOff[(long long)c * nTiles];
    const int b = c + 1 < nch ? tileOff[(long long)(c + 1) * nTiles] : Z;
    cnt[c] = b - a;
    padded = (b - a + 3) & ~3;
  }
  int total = 0;
  const int ex = block_exclusive_scan(padded, &total, sWarp);
  if (c < nch) chunkPtr[c] = ex;
  if (c == 0) chunkPtr[nch] = total;
}

// Row of nonzero k from its chunk record: lo plus the row starts at or
// before k's position (a binary search on rowPtrs in a chunk that holds an
// empty row).
__device__ __forceinline__ int xb_row_of(const CsrChunkDesc& d, long long k,
                                         const int* __restrict__ rowPtrs) {
  if (!(d.flags & kCsrChunkHasEmptyRow)) {
    const int pos = (int)(k & (kCsrChunk - 1));
    const int wd = pos >> 5;
    const unsigned mw = wd == 0 ? d.mask.x : wd == 1 ? d.mask.y : wd == 2 ? d.mask.z : d.mask.w;
    const int before = (wd > 0 ? __popc(d.mask.x) : 0) + (wd > 1 ? __popc(d.mask.y) : 0) +
                       (wd > 2 ? __popc(d.mask.z) : 0);
    return d.lo + before + __popc(mw & ((2u << (pos & 31)) - 1u));
  }
  int r = d.lo, b = d.hi;
  while (r < b) {
    const int m = (r + b + 1) >> 1;
    if (__ldg(rowPtrs + m) <= k) r = m; else b = m - 1;
  }
  return r;
}

// Lanes of the warp holding the same value v < 2^nbits (nbits warp-uniform).
// BALLOTS: one ballot per bit of v; otherwise __match_any_sync. The launch
// takes ballots for scattered columns (many chunks among 32 consecutive
// entries), the match otherwise. Measured on the tile scatter: skewed rows
// 459 us with the match (ncu: its pipe at 75 % of peak, DRAM at 17 %) and
// 393 us with ballots; 27-point stencil (one or two chunks per 32 entries)
// 952 us with the match and 1291 us with ballots. Choosing per 32 entries
// (by the number of value changes between neighbouring lanes) cost more than
// it saved: 420 and 1030 us.
template <bool BALLOTS>
__device__ __forceinline__ unsigned warp_peers(unsigned v, int nbits) {
  if (!BALLOTS) return __match_any_sync(kFullMask, v);
  unsigned peers = kFullMask;
  for (int b = 0; b < nbits; ++b) {
    const unsigned bit = (v >> b) & 1u;
    const unsigned bal = __ballot_sync(kFullMask, bit);
    peers &= bit ? bal : ~bal;
  }
  return peers;
}

template <class T, bool BALLOTS>
__global__ void __launch_bounds__(kXbTileThreads, 6) k_xb_tile_scatter(
    int Z, ChunkDiv div, int nch, int nTiles, const int* __restrict__ rowPtrs,
    const CsrChunkDesc* __restrict__ desc, const int* __restrict__ colIdx,
    const T* __restrict__ value, const int* __restrict__ tileOff,
    const int* __restrict__ chunkPtr, int* __restrict__ xbRow, unsigned short* __restrict__ xbCol,
    T* __restrict__ xbVal) {
  constexpr int kWarps = kXbTileThreads / 32;
  constexpr int kPerWarp = kXbTile / kWarps;  // 32 * kXbTileRounds
  __shared__ int sCur[kWarps][kXbTileChunks];  // counts, then running positions in the tile
  __shared__ int sBase[kXbTileChunks];         // output position of the tile's first entry of c
  __shared__ int sRow[kXbTile];
  __shared__ T sVal[kXbTile];
  __shared__ unsigned short sLoc[kXbTile];
  __shared__ unsigned char sChk[kXbTile];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int c = lane; c < nch; c += 32) sCur[w][c] = 0;
  // output start of this tile's entries of chunk threadIdx.x, loaded while
  // the entries load
  int outBase = 0;
  if ((int)threadIdx.x < nch) {
    const long long row0 = (long long)threadIdx.x * nTiles;
    outBase = __ldg(chunkPtr + threadIdx.x) + (__ldg(tileOff + row0 + blockIdx.x) -
                                               __ldg(tileOff + row0));
  }
  const long long tileBase = (long long)blockIdx.x * kXbTile;
  const long long wbase = tileBase + (long long)w * kPerWarp;
  int chk[kXbTileRounds], row[kXbTileRounds], loc[kXbTileRounds];
  T val[kXbTileRounds];
#pragma unroll
  for (int rd = 0; rd < kXbTileRounds; ++rd) {
    const long long k = wbase + rd * 32 + lane;
    chk[rd] = nch;  // no entry: a value no chunk takes
    row[rd] = 0;
    loc[rd] = 0;
    val[rd] = T(0);
    if (k < Z) {
      const int col = __ldcs(colIdx + k);
      val[rd] = __ldcs(value + k);
      const int c = div(col);
      chk[rd] = c;
      loc[rd] = col - c * div.b;
      row[rd] = xb_row_of(desc[k >> 7], k, rowPtrs);  // 32 lanes, one record
    }
  }
  __syncwarp();
  const int nbits = 32 - __clz(nch);  // bits of the values 0 .. nch
#pragma unroll
  for (int rd = 0; rd < kXbTileRounds; ++rd) {
    const unsigned peers = warp_peers<BALLOTS>((unsigned)chk[rd], nbits);
    if (chk[rd] < nch && lane == __ffs(peers) - 1) sCur[w][chk[rd]] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // tile-local starts of the chunks (scan over the chunks of the tile's
  // counts), each warp's start inside its chunk, and the output position of
  // the tile's first entry of each chunk
  __shared__ int sWarp[kScanThreads / 32 + 1];
  {
    const int c = threadIdx.x;  // nch <= kXbTileChunks <= kXbTileThreads
    int tot = 0;
    if (c < nch)
#pragma unroll
      for (int q = 0; q < kWarps; ++q) tot += sCur[q][c];
    int all = 0;
    const int lstart = block_exclusive_scan(tot, &all, sWarp);
    if (c < nch) {
      int run = lstart;
#pragma unroll
      for (int q = 0; q < kWarps; ++q) {
        const int cntq = sCur[q][c];
        sCur[q][c] = run;
        run += cntq;
      }
      sBase[c] = outBase - lstart;
    }
  }
  __syncthreads();
#pragma unroll
  for (int rd = 0; rd < kXbTileRounds; ++rd) {
    const int c = chk[rd];
    const unsigned peers = warp_peers<BALLOTS>((unsigned)c, nbits);
    const bool valid = c < nch;
    const int start = valid ? sCur[w][c] : 0;
    __syncwarp();
    if (valid) {
      const int q = start + __popc(peers & lanemask_lt());
      sRow[q] = row[rd];
      sVal[q] = val[rd];
      sLoc[q] = (unsigned short)loc[rd];
      sChk[q] = (unsigned char)c;
      if (lane == __ffs(peers) - 1) sCur[w][c] = start + __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();
  // out: the tile's entries in chunk order; a chunk's entries are
  // consecutive here and in the output
  const int n = (int)(Z - tileBase < kXbTile ? Z - tileBase : kXbTile);
  for (int q = threadIdx.x; q < n; q += kXbTileThreads) {
    const long long p = (long long)sBase[sChk[q]] + q;
    __stcs(xbRow + p, sRow[q]);
    __stcs(xbCol + p, sLoc[q]);
    __stcs(xbVal + p, sVal[q]);
  }
}

size_t xb_scratch_bytes(int Z, int nch) {
  if (nch <= kXbTileChunks) {
    // cnt[nch], tileCnt[nch * nTiles + 1], scan scratch for it
    const long long nTiles = ((long long)Z + kXbTile - 1) / kXbTile;
    const long long n = (long long)nch * (nTiles > 0 ? nTiles : 1);
    return sizeof(int) * (size_t)(nch + n + 1 + (long long)scan_scratch_ints(n) + 16);
  }
  // cnt[nch], ustart[nch + 1], scan scratch for nch, the sort's item order
  // perm[Z], then the radix sort's own scratch for Z items
  const size_t ints = 2 * (size_t)nch + 1 + (size_t)scan_scratch_ints(nch) + (size_t)Z;
  return ints * sizeof(int) + jds_sort_scratch_bytes(Z, nch > 0 ? nch - 1 : 0);
}

template <class T>
cudaError_t launch_xb_build(int Z, int B, int nch, const int* rowPtrs, const CsrChunkDesc* desc,
                            const int* colIdx, const T* value, const int* rowIdx, bool scattered,
                            int* chunkPtr, int* xbRow, unsigned short* xbCol, T* xbVal,
                            void* scratch, cudaStream_t s) {
  if (nch <= 0) return cudaMemsetAsync(chunkPtr, 0, sizeof(int), s);
  if (nch <= kXbTileChunks && Z > 0) {
    const long long nTiles = ((long long)Z + kXbTile - 1) / kXbTile;
    const long long n = (long long)nch * nTiles;
    int* cnt = static_cast<int*>(scratch);
    int* tileCnt = cnt + nch;
    int* scanScratch = tileCnt + n + 1;
    const ChunkDiv div = chunk_div(B);
    if (aligned16(colIdx))
      k_xb_tile_count<true><<<(unsigned)nTiles, kXbTileThreads, 0, s>>>(Z, div, nch, (int)nTiles,
                                                                        colIdx, tileCnt);
    else
      k_xb_tile_count<false><<<(unsigned)nTiles, kXbTileThreads, 0, s>>>(Z, div, nch,
                                                                         (int)nTiles, colIdx,
                                                                         tileCnt);
    note_launches(1);
    cudaError_t err = exclusive_scan(ArrayIn{tileCnt}, n, tileCnt, scanScratch, s);
    if (err != cudaSuccess) return err;
    k_xb_chunk_ptr<<<1, kScanThreads, 0, s>>>(Z, nch, (int)nTiles, tileCnt, cnt, chunkPtr);
    if (scattered)
      k_xb_tile_scatter<T, true><<<(unsigned)nTiles, kXbTileThreads, 0, s>>>(
          Z, div, nch, (int)nTiles, rowPtrs, desc, colIdx, value, tileCnt, chunkPtr, xbRow,
          xbCol, xbVal);
    else
      k_xb_tile_scatter<T, false><<<(unsigned)nTiles, kXbTileThreads, 0, s>>>(
          Z, div, nch, (int)nTiles, rowPtrs, desc, colIdx, value, tileCnt, chunkPtr, xbRow,
          xbCol, xbVal);
    k_xb_pad<T><<<(unsigned)((nch + 255) / 256), 256, 0, s>>>(nch, cnt, chunkPtr, xbRow, xbCol,
                                                             xbVal);
    note_launches(3);
    return cudaGetLastError();
  }
  int* cnt = static_cast<int*>(scratch);
  int* ustart = cnt + nch;
  int* scanScratch = ustart + nch + 1;
  int* sortScratch = scanScratch + scan_scratch_ints(nch);
  cudaError_t err = cudaMemsetAsync(cnt, 0, sizeof(int) * (size_t)nch, s);
  if (err != cudaSuccess) return err;
  if (Z > 0) {
    long long blocks = ((long long)Z + kXbCountThreads * 16 - 1) / (kXbCountThreads * 16);
    const long long cap = 8LL * num_sms();
    k_xb_count<<<(unsigned)(blocks < cap ? blocks : cap), kXbCountThreads, 0, s>>>(Z, B, nch,
                                                                                 colIdx, cnt);
    note_launches(1);
  }
  err = exclusive_scan(ArrayIn{cnt}, nch, ustart, scanScratch, s);
  if (err == cudaSuccess) err = exclusive_scan(Pad4In{cnt}, nch, chunkPtr, scanScratch, s);
  if (err != cudaSuccess || Z <= 0) {
    if (err == cudaSuccess) {
      k_xb_pad<T><<<(unsigned)((nch + 255) / 256), 256, 0, s>>>(nch, cnt, chunkPtr, xbRow, xbCol,
                                                            xbVal);
      note_launches(1);
      err = cudaGetLastError();
    }
    return err;
  }
  // stable rank of every nonzero among the nonzeros of its chunk
  int* perm = sortScratch;  // sorted item order (not used beyond the sort)
  const int* sortedKeys = nullptr;
  int* inv = nullptr;
  int* unusedScan = nullptr;
  err = radix_sort(ChunkKeyIn{colIdx, B, nullptr, nullptr}, Z, nch - 1, perm, sortScratch + Z,
                   false, &sortedKeys, &inv, &unusedScan, s);
  if (err != cudaSuccess) return err;
  k_xb_scatter<T><<<(unsigned)(((long long)Z + 255) / 256), 256, 0, s>>>(
      Z, B, colIdx, value, rowIdx, inv, ustart, chunkPtr, xbRow, xbCol, xbVal);
  k_xb_pad<T><<<(unsigned)((nch + 255) / 256), 256, 0, s>>>(nch, cnt, chunkPtr, xbRow, xbCol,
                                                           xbVal);
  note_launches(2);
  return cudaGetLastError();
}

// the two value types
#define SPMV_INSTANTIATE(T)                                                                      \
  template cudaError_t launch_hyb_tail_copy<T>(int, int, const int*, const int*, const T*,      \
                                               const int*, int*, int*, T*, cudaStream_t);        \
  template cudaError_t launch_jds_build<T>(int, int, int, const int*, const int*, const T*,     \
                                           int*, int*, int*, T*, void*, const int*,              \
                                           cudaStream_t);                                        \
  template cudaError_t launch_sell_scatter<T>(int, int, int, const int*, const int*, const T*,  \
                                              const void*, const int*, int, int*, T*,            \
                                              cudaStream_t);                                     \
  template cudaError_t launch_xb_build<T>(int, int, int, const int*, const CsrChunkDesc*,       \
                                          const int*, const T*, const int*, bool, int*, int*,   \
                                          unsigned short*, T*, void*, cudaStream_t);
SPMV_INSTANTIATE(float)
SPMV_INSTANTIATE(double)
#undef SPMV_INSTANTIATE

}  // namespace spmv
