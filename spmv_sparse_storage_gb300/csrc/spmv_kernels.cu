// spmv_kernels.cu -- y <- A*x + y for each storage format.
//
// Operation: sparse matrix-vector multiplication and accumulation (PMPP
// notes, "Sparse Matrices and Basic Formats (COO and CSR)", section
// "Background & SpMV"). Every kernel is memory-bound: per nonzero it moves a
// 4-byte value and a 4-byte column index and does one multiply-add ("Regularized
// Formats (ELL, Hybrid ELL-COO and JDS)", section "Summary": 0.25 op/byte),
// so the designs below are about streaming those bytes at HBM speed, keeping
// the gathered x resident in L2, and balancing the work.
#include <climits>
#include <type_traits>

#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

// Across lanes: each lane holds a run of consecutive entries summarised as
// its head run (row rh, sum sh), its tail run (row rt, sum st) and whether
// the whole lane is one run (single); runs strictly inside a lane are the
// caller's. Adds the head and tail runs into y, joining runs that continue
// across lanes with a segmented shuffle scan, one atomicAdd per joined run.
template <class T>
__device__ __forceinline__ void warp_join_runs(int rh, int rt, T sh, T st, bool single,
                                               T* __restrict__ y, bool waitFirst) {
  const int lane = threadIdx.x & 31;
  // w = tail-run sum carried to the right while lanes continue one run
  const int prevRt = __shfl_up_sync(kFullMask, rt, 1);
  const bool connected = lane > 0 && prevRt == rh;
  const unsigned heads = __ballot_sync(kFullMask, !(single && connected));
  const int segStart = 31 - __clz(heads & (0xffffffffu >> (31 - lane)));
  T w = st;
  if constexpr (sizeof(T) == 8) {
    // 8-byte values: the kernels are bound by the fp64 adds, so only as many
    // doubling steps as the longest run of lanes needs (one on a 5-point
    // stencil, none when no run crosses a lane). With 4-byte values the
    // kernels are bound by memory latency and keep the unrolled five steps
    // (no reduction on each warp's critical path).
    const int span = __reduce_max_sync(kFullMask, lane - segStart);
    for (int off = 1; off <= span; off <<= 1) {  // warp-uniform bound
      const T o = __shfl_up_sync(kFullMask, w, off);
      if (lane - off >= segStart) w += o;
    }
  } else {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const T o = __shfl_up_sync(kFullMask, w, off);
      if (lane - off >= segStart) w += o;
    }
  }
  const T wPrev = __shfl_up_sync(kFullMask, w, 1);
  const T carryIn = connected ? wPrev : T(0);
  const int nextRh = __shfl_down_sync(kFullMask, rh, 1);
  const bool tailEnds = (lane == 31) || nextRh != rt;

  if (waitFirst) grid_dependency_wait();
  if (single) {
    if (tailEnds && rt >= 0) atomicAdd(y + rt, st + carryIn);
  } else {
    if (rh >= 0) atomicAdd(y + rh, sh + carryIn);
    if (tailEnds && rt >= 0) atomicAdd(y + rt, st);
  }
}

// ===========================================================================
// Warp-level segmented add. Each lane holds 4 consecutive entries of a
// 128-entry chunk (entry 4*lane + e) and their row `row[e]` (-1 = no entry).
// Runs of equal row are summed inside the lane, then across lanes with a
// segmented shuffle scan, and each run is added into y with ONE atomicAdd (a
// fire-and-forget reduction in L2). Only adjacent equal rows merge, so any
// entry order is correct; rows grouped together give one atomic per row per
// chunk. `waitFirst`: wait for the preceding kernel of the stream
// (programmatic dependent launch) before the first write to y.
// ===========================================================================
// s[e] = sum of the lane's run that ends at entry e
template <class T>
__device__ __forceinline__ void segmented_add_runs(const int (&row)[4], const T (&s)[4],
                                                   T* __restrict__ y, bool waitFirst) {
  const int hEnd = row[1] != row[0] ? 0 : row[2] != row[1] ? 1 : row[3] != row[2] ? 2 : 3;
  const bool single = (hEnd == 3);
  warp_join_runs(row[0], row[3], s[hEnd], s[3], single, y, waitFirst);
  if (!single) {
#pragma unroll
    for (int e = 1; e < 3; ++e)  // runs strictly inside the lane
      if (e > hEnd && row[e] != row[e + 1] && row[e] >= 0) atomicAdd(y + row[e], s[e]);
  }
}

// From the products p[e] (0 for no entry): the in-lane sums are adds.
template <class T>
__device__ __forceinline__ void warp_segmented_add(const int (&row)[4], const T (&p)[4],
                                                   T* __restrict__ y, bool waitFirst) {
  T s[4];
  s[0] = p[0];
#pragma unroll
  for (int e = 1; e < 4; ++e) s[e] = (row[e] == row[e - 1]) ? s[e - 1] + p[e] : p[e];
  segmented_add_runs(row, s, y, waitFirst);
}

// From the values v[e] and gathered x xg[e] (0 for no entry): the in-lane
// sums are fused multiply-adds, 4 operations for 4 entries instead of 7. Used
// with 8-byte values, where the fp64 rate bounds the kernel; with 4-byte
// values the product form measured faster (COO on a 5-point stencil 45.7 vs
// 47.7 us, on a 27-point stencil 207 vs 219 us).
template <class T>
__device__ __forceinline__ void warp_segmented_fma(const int (&row)[4], const T (&v)[4],
                                                   const T (&xg)[4], T* __restrict__ y,
                                                   bool waitFirst) {
  T s[4];
  s[0] = v[0] * xg[0];
#pragma unroll
  for (int e = 1; e < 4; ++e) s[e] = fma_t(v[e], xg[e], row[e] == row[e - 1] ? s[e - 1] : T(0));
  segmented_add_runs(row, s, y, waitFirst);
}

// ===========================================================================
// CSR, nnz-balanced.
//
// The pages' CSR kernels give a row to a thread ("CSR format and SpMV") or a
// warp ("[CUDA performance tuning] ...", section 2.2); both idle threads when
// row lengths differ, and the remedy named in "Introduction to sparse
// computing ...", section "Building the problem framework", is to split the
// work by nonzero count and to split very long rows. Here the nonzeros are
// cut into chunks of kCsrChunk = 128 whatever rows they belong to: a
// 5000-entry row spreads over 40 chunks, an empty row costs nothing.
//
// Row ids come from a 32-byte record per chunk built once at handle
// creation: lo = the row holding the chunk's first nonzero and mask = the
// chunk positions where a later row starts. The row of entry p is lo plus
// the number of mask bits at positions <= p (popcounts), so the kernel reads
// 0.25 byte of index per nonzero and never waits on rowPtrs; a chunk in
// which an empty row sits (flagged) binary-searches rowPtrs instead.
// ===========================================================================

// The CSR kernel: kCsrLane = 8 consecutive entries per lane. A warp takes
// 256 nonzeros (two chunks); lane l takes the entries at 8l, which sit in
// chunk l/16 at position 8(l%16): one byte of one mask word. The lane's
// first row is lo + the set bits up to that position, and the row advances
// at every further set bit. Runs of equal row are summed in the lane
// with one multiply-add per entry (a run that starts and ends inside the lane
// goes to y directly), and the lane's head and tail runs are joined across
// lanes once per 256 entries (warp_join_runs). The decode, the join and the
// loop are paid once per 8 entries and the accumulation is one fused
// multiply-add per entry, so the kernel is not bound by instruction issue
// (with 4 entries per lane it was, in a shared-memory (bulk copy) pipeline as
// well: 214 warp instructions per 128 entries). Loads are direct 16-byte
// vectors. A chunk that holds an empty row is decoded by a binary search on
// rowPtrs.
constexpr int kCsrLane = 8;
constexpr int kCsrSuper = 32 * kCsrLane;             // entries per warp
constexpr int kCsrLanesPerChunk = kCsrChunk / kCsrLane;

// Rows of a lane's kCsrLane consecutive entries starting at `base`, which
// sit in chunk base / kCsrChunk at position kCsrLane * (lane % 16): one byte
// of one mask word (the row advances at every set bit after lo + the set
// bits up to that position). Entries at or past Z get -1. A chunk holding an
// empty row is decoded by a binary search on rowPtrs instead.
__device__ __forceinline__ void lane_rows(const CsrChunkDesc& d, long long base, int lane, int Z,
                                          const int* __restrict__ rowPtrs, int (&row)[kCsrLane]) {
  const bool full = base + kCsrLane <= Z;
  if (!(d.flags & kCsrChunkHasEmptyRow)) {
    const int q0 = kCsrLane * (lane % kCsrLanesPerChunk);  // position in the chunk
    const int wd = q0 >> 5;
    const unsigned mw = wd == 0 ? d.mask.x : wd == 1 ? d.mask.y : wd == 2 ? d.mask.z : d.mask.w;
    const int before = (wd > 0 ? __popc(d.mask.x) : 0) + (wd > 1 ? __popc(d.mask.y) : 0) +
                       (wd > 2 ? __popc(d.mask.z) : 0);
    const int sh = q0 & 31;  // the lane's entries are bits sh .. sh + kCsrLane - 1 of mw
    int r = d.lo + before + __popc(mw & ((2u << sh) - 1u));
    const unsigned bits = mw >> sh;
#pragma unroll
    for (int e = 0; e < kCsrLane; ++e) {
      if (e > 0) r += (bits >> e) & 1u;
      row[e] = (full || base + e < Z) ? r : -1;
    }
  } else {
    const int hi = d.hi;
    int r = d.lo;
    if (base < Z) {
      int b = hi;
      while (r < b) {
        const int m = (r + b + 1) >> 1;
        if (__ldg(rowPtrs + m) <= (int)base) r = m; else b = m - 1;
      }
    }
    int nextStart = r < hi ? __ldg(rowPtrs + r + 1) : INT_MAX;
#pragma unroll
    for (int e = 0; e < kCsrLane; ++e) {
      const long long k = base + e;
      while (k >= nextStart) {  // skips empty rows; bounded by hi
        ++r;
        nextStart = r < hi ? __ldg(rowPtrs + r + 1) : INT_MAX;
      }
      row[e] = k < Z ? r : -1;
    }
  }
}

template <class T, bool VEC>
__global__ void __launch_bounds__(256) k_spmv_csr_wide(int Z, const int* __restrict__ rowPtrs,
                                                       const int* __restrict__ colIdx,
                                                       const T* __restrict__ value,
                                                       const CsrChunkDesc* __restrict__ desc,
                                                       const T* __restrict__ x,
                                                       T* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long g = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (g * kCsrSuper >= Z) return;  // warp-uniform
  const long long base = g * kCsrSuper + (long long)lane * kCsrLane;
  const bool any = base < Z;
  const bool full = base + kCsrLane <= Z;
  // the lane's chunk record (chunk index < nChunks whenever base < Z)
  CsrChunkDesc d = {};
  if (any) d = desc[(g * kCsrSuper + (long long)lane * kCsrLane) / kCsrChunk];
  int col[kCsrLane];
  T val[kCsrLane];
  if (VEC && full) {
#pragma unroll
    for (int q = 0; q < kCsrLane / 4; ++q) {
      const int4 c4 = ld_stream(reinterpret_cast<const int4*>(colIdx + base) + q);
      col[4 * q] = c4.x; col[4 * q + 1] = c4.y; col[4 * q + 2] = c4.z; col[4 * q + 3] = c4.w;
      const Vec4<T> v4 = ld4_stream(value + base + 4 * q);
      val[4 * q] = v4.x; val[4 * q + 1] = v4.y; val[4 * q + 2] = v4.z; val[4 * q + 3] = v4.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kCsrLane; ++e) {
      const bool in = base + e < Z;
      col[e] = in ? ld_stream(colIdx + base + e) : 0;
      val[e] = in ? ld_stream(value + base + e) : T(0);
    }
  }
  // rows of the lane's entries (-1 past nnz)
  int row[kCsrLane];
  lane_rows(d, base, lane, Z, rowPtrs, row);
  // gathers, all issued before the multiply-adds
  T xg[kCsrLane];
#pragma unroll
  for (int e = 0; e < kCsrLane; ++e) xg[e] = row[e] >= 0 ? ld_x(x + col[e]) : T(0);
  // runs inside the lane
  T run = T(0), head = T(0);
  bool boundary = false;
#pragma unroll
  for (int e = 0; e < kCsrLane; ++e) {
    const bool cont = e == 0 || row[e] == row[e - 1];
    if (!cont) {
      if (boundary) {
        if (row[e - 1] >= 0) atomicAdd(y + row[e - 1], run);  // a row that ended in the lane
      } else {
        head = run;
        boundary = true;
      }
    }
    run = fma_t(val[e], xg[e], cont ? run : T(0));
  }
  warp_join_runs(row[0], row[kCsrLane - 1], boundary ? head : run, run, !boundary, y, false);
}

// CSR -> COO ("Sparse Matrices and Basic Formats ...", section "COO format
// and SpMV"): rowIdx[k] = r for rowPtrs[r] <= k < rowPtrs[r+1]. The layout of
// the CSR kernel: per 256 nonzeros, each lane takes 8 consecutive ones,
// decodes their rows from its chunk record (lane_rows) and stores them with
// two 16-byte stores (VEC: rowIdx is 16-byte aligned). A warp takes
// kExpandSupers consecutive blocks of 256 and loads all their chunk records
// before decoding any, so that one load round trip serves them all (the
// kernel has nothing else to wait on).
constexpr int kExpandSupers = 4;
template <bool VEC>
__global__ void __launch_bounds__(256) k_expand_rows(int Z, const int* __restrict__ rowPtrs,
                                                     const CsrChunkDesc* __restrict__ desc,
                                                     int* __restrict__ rowIdx) {
  const int lane = threadIdx.x & 31;
  const long long g = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long first = g * kExpandSupers * kCsrSuper + (long long)lane * kCsrLane;
  if (first >= Z) return;  // no shuffles below: lanes may leave
  CsrChunkDesc d[kExpandSupers];
#pragma unroll
  for (int k = 0; k < kExpandSupers; ++k) {
    const long long base = first + (long long)k * kCsrSuper;
    if (base < Z) d[k] = desc[base / kCsrChunk];
  }
#pragma unroll
  for (int k = 0; k < kExpandSupers; ++k) {
    const long long base = first + (long long)k * kCsrSuper;
    if (base >= Z) break;
    int row[kCsrLane];
    lane_rows(d[k], base, lane, Z, rowPtrs, row);
    if (VEC && base + kCsrLane <= Z) {
      int4* out = reinterpret_cast<int4*>(rowIdx + base);
      __stcs(out, make_int4(row[0], row[1], row[2], row[3]));
      __stcs(out + 1, make_int4(row[4], row[5], row[6], row[7]));
    } else {
#pragma unroll
      for (int e = 0; e < kCsrLane; ++e)
        if (base + e < Z) rowIdx[base + e] = row[e];
    }
  }
}

// Chunk records: hi from the next chunk's lo, and the positions where rows
// start inside the chunk (or the empty-row flag). Thread per chunk, walking
// the rows that start in it (at most kCsrChunk + 1 steps). Bounds are checked
// so that this kernel, which runs before validation is known, stays in
// bounds on invalid input.
__global__ void k_csr_chunk_masks(int R, int Z, const int* __restrict__ rowPtrs, int nChunks,
                                  CsrChunkDesc* __restrict__ desc) {
  const long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= nChunks) return;
  const int lo = desc[c].lo;
  const int hi = c + 1 < nChunks ? desc[c + 1].lo : (R > 0 ? R - 1 : 0);
  const long long cb = c * kCsrChunk;
  unsigned m[4] = {0u, 0u, 0u, 0u};
  int flags = 0;
  if (lo >= 0 && lo < R) {
    int next = rowPtrs[lo + 1];
    for (int r = lo + 1; r < R; ++r) {
      const int st = next;
      if (st >= cb + kCsrChunk || st >= Z) break;
      next = rowPtrs[r + 1];
      if (next == st) {  // row r is empty and sits inside the chunk
        flags |= kCsrChunkHasEmptyRow;
        break;
      }
      const long long pos = st - cb;
      if (pos > 0 && pos < kCsrChunk) m[pos >> 5] |= 1u << (pos & 31);
    }
  } else {
    flags |= kCsrChunkHasEmptyRow;  // invalid input: take the searching path
  }
  CsrChunkDesc d;
  d.lo = lo;
  d.hi = hi;
  d.flags = flags;
  d.pad0 = 0;
  d.mask = make_uint4(m[0], m[1], m[2], m[3]);
  desc[c] = d;
}

// ===========================================================================
// ELL ("Regularized Formats ...", section "ELL format: padding +
// transposition"): thread per row, slot t of row r at t*numRows + r, so a
// warp reads consecutive slots (coalesced). The loop runs over all K slots;
// padding slots (column -1) skip the x gather and add nothing, so nnzPerRow
// is never read. VEC4: numRows % 4 == 0 and 16-byte aligned arrays, a thread
// handles 4 consecutive rows with 16-byte loads.
// ===========================================================================
template <class T, bool VEC4>
__global__ void __launch_bounds__(256, 4) k_spmv_ell(int R, int K, const int* __restrict__ ellCol,
                                                     const T* __restrict__ ellVal,
                                                     const T* __restrict__ x,
                                                     T* __restrict__ y) {
  // let a programmatically dependent kernel (the COO part of HYB) start its
  // loads; it waits for this grid to finish before it writes y
  grid_dependency_trigger();
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (VEC4) {
    const long long ld = R >> 2;
    if (q >= ld) return;
    const int4* c4 = reinterpret_cast<const int4*>(ellCol);
    const Vec4<T> y0 = ld4(y + 4 * q);
    Vec4<T> acc = {T(0), T(0), T(0), T(0)};
    int t = 0;
    for (; t + 4 <= K; t += 4) {
      int4 c[4];
      Vec4<T> v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c[u] = ld_stream(c4 + (size_t)(t + u) * ld + q);
        v[u] = ld4_stream(ellVal + 4 * ((size_t)(t + u) * ld + q));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c[u].x >= 0) acc.x = fma_t(v[u].x, ld_x(x + c[u].x), acc.x);
        if (c[u].y >= 0) acc.y = fma_t(v[u].y, ld_x(x + c[u].y), acc.y);
        if (c[u].z >= 0) acc.z = fma_t(v[u].z, ld_x(x + c[u].z), acc.z);
        if (c[u].w >= 0) acc.w = fma_t(v[u].w, ld_x(x + c[u].w), acc.w);
      }
    }
    for (; t < K; ++t) {
      const int4 c = ld_stream(c4 + (size_t)t * ld + q);
      const Vec4<T> v = ld4_stream(ellVal + 4 * ((size_t)t * ld + q));
      if (c.x >= 0) acc.x = fma_t(v.x, ld_x(x + c.x), acc.x);
      if (c.y >= 0) acc.y = fma_t(v.y, ld_x(x + c.y), acc.y);
      if (c.z >= 0) acc.z = fma_t(v.z, ld_x(x + c.z), acc.z);
      if (c.w >= 0) acc.w = fma_t(v.w, ld_x(x + c.w), acc.w);
    }
    st4(y + 4 * q, Vec4<T>{y0.x + acc.x, y0.y + acc.y, y0.z + acc.z, y0.w + acc.w});
  } else {
    if (q >= R) return;
    const T y0 = y[q];
    T acc = T(0);
    int t = 0;
    for (; t + 4 <= K; t += 4) {
      int c[4];
      T v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c[u] = ld_stream(ellCol + (size_t)(t + u) * R + q);
        v[u] = ld_stream(ellVal + (size_t)(t + u) * R + q);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c[u] >= 0) acc = fma_t(v[u], ld_x(x + c[u]), acc);
    }
    for (; t < K; ++t) {
      const int c = ld_stream(ellCol + (size_t)t * R + q);
      const T v = ld_stream(ellVal + (size_t)t * R + q);
      if (c >= 0) acc = fma_t(v, ld_x(x + c), acc);
    }
    y[q] = y0 + acc;
  }
}

// ===========================================================================
// COO ("Sparse Matrices and Basic Formats ...", section "COO format and
// SpMV" uses one atomicAdd per nonzero, and same-row nonzeros contend). Here
// a warp takes 128 consecutive entries, 4 per lane (16-byte loads when
// aligned) and adds each run of equal row index with one atomicAdd (see
// warp_segmented_add). `dependent`: launched as a programmatic dependent of
// the ELL part of HYB, the kernel loads and reduces before waiting for that
// kernel, and only then touches y.
// ===========================================================================
template <class T, bool VEC>
__global__ void __launch_bounds__(256) k_spmv_coo(int Z, const int* __restrict__ rowIdx,
                                                  const int* __restrict__ colIdx,
                                                  const T* __restrict__ value,
                                                  const T* __restrict__ x,
                                                  T* __restrict__ y, int dependent) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long base = warp * 128 + 4 * lane;

  int row[4];
  if constexpr (sizeof(T) == 4) {
    T p[4];
    if (VEC && base + 4 <= Z) {
      const int4 r4 = ld_stream(reinterpret_cast<const int4*>(rowIdx + base));
      const int4 c4 = ld_stream(reinterpret_cast<const int4*>(colIdx + base));
      const Vec4<T> v4 = ld4_stream(value + base);
      row[0] = r4.x; row[1] = r4.y; row[2] = r4.z; row[3] = r4.w;
      p[0] = v4.x * ld_x(x + c4.x);
      p[1] = v4.y * ld_x(x + c4.y);
      p[2] = v4.z * ld_x(x + c4.z);
      p[3] = v4.w * ld_x(x + c4.w);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const long long k = base + e;
        if (k < Z) {
          row[e] = ld_stream(rowIdx + k);
          p[e] = ld_stream(value + k) * ld_x(x + ld_stream(colIdx + k));
        } else {
          row[e] = -1;  // sentinel: no entry
          p[e] = T(0);
        }
      }
    }
    warp_segmented_add(row, p, y, dependent != 0);
  } else {
    T v[4], xg[4];
    if (VEC && base + 4 <= Z) {
      const int4 r4 = ld_stream(reinterpret_cast<const int4*>(rowIdx + base));
      const int4 c4 = ld_stream(reinterpret_cast<const int4*>(colIdx + base));
      const Vec4<T> v4 = ld4_stream(value + base);
      row[0] = r4.x; row[1] = r4.y; row[2] = r4.z; row[3] = r4.w;
      v[0] = v4.x; v[1] = v4.y; v[2] = v4.z; v[3] = v4.w;
      xg[0] = ld_x(x + c4.x);
      xg[1] = ld_x(x + c4.y);
      xg[2] = ld_x(x + c4.z);
      xg[3] = ld_x(x + c4.w);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const long long k = base + e;
        if (k < Z) {
          row[e] = ld_stream(rowIdx + k);
          v[e] = ld_stream(value + k);
          xg[e] = ld_x(x + ld_stream(colIdx + k));
        } else {
          row[e] = -1;  // sentinel: no entry
          v[e] = T(0);
          xg[e] = T(0);
        }
      }
    }
    warp_segmented_fma(row, v, xg, y, dependent != 0);
  }
}

// ===========================================================================
// JDS ("Regularized Formats ...", section "JDS format": a thread takes a
// sorted row and walks the jagged diagonals from iterPtr; the page leaves the
// kernel as an exercise). Diagonal t holds one entry for every sorted row
// s < width(t), contiguous in s, so a warp's loads are coalesced. Widths only
// shrink with t; the first tSplit diagonals (those at least
// kJdsSplitMinWidth wide, at most kJdsSplitMaxDiag of them) run one thread
// per sorted row (two with 4-byte values: rows 32 apart): a warp's 32 rows of
// a diagonal are 32 consecutive entries, so 4-byte loads are coalesced
// wherever the diagonal starts, and a thread loads a group of diagonals
// before it gathers any x. (4 consecutive rows per thread with 16-byte loads
// needed a shuffle realignment per diagonal and 64 registers.)
// The remaining diagonals belong to the few
// longest rows (s < wTail) and would serialise one thread over thousands of
// entries, so they are split into blocks of kJdsTailRows rows x
// kJdsTailDiags diagonals that run in parallel and add their partial sums
// atomically. The result of sorted row s goes straight to y[perm[s]] (the
// page permutes the result back with the row array). With at most
// kJdsParamDiags row-parallel diagonals their iterPtr entries come with the
// launch (from the host's length histogram): a block then starts its loads at
// once instead of first copying them into shared memory behind a barrier
// (cold L2: 5-point Laplacian 45.0 -> 43.0 us, uniform random rows 29.7 ->
// 26.6 us, skewed rows 168.6 -> 163.8 us; 64-thread blocks gained nothing
// more).
// ===========================================================================
// diagonals whose loads a thread issues together: 8 with 4-byte values (32
// registers; laplace2d 45.1 us, 27-point stencil 148 us, against 53.3 and
// 152 with 4), 5 with 8-byte values (8 needs 48 registers: 27-point stencil
// 251 us against 227)
template <class T>
constexpr int kJdsGroup = sizeof(T) == 4 ? 8 : 5;
// iterPtr[0 .. tSplit] as a launch parameter (PARAM kernels): read through the
// constant cache, so that a block starts its row loads at once. Otherwise
// the block first copies them into shared memory and synchronises, one more
// round trip on the path of a short-lived block.
struct JdsIterPtrs {
  int v[kJdsParamDiags + 1];
};
// RPT sorted rows per thread: rows warpBase + 32 j + lane, j < RPT, so that
// every load of a warp is still 32 consecutive entries of a diagonal and a
// thread keeps RPT rows' loads in flight. Diagonals are loaded
// kJdsRowGroup<T, RPT> at a time.
template <class T, int RPT>
constexpr int kJdsRowGroup = RPT == 1 ? kJdsGroup<T> : 4;
template <class T, bool PARAM, int RPT>
__global__ void __launch_bounds__(256) k_spmv_jds(int R, int maxLen, int tSplit, int wTail,
                                                     int nMainBlocks, int tailRowBlocks,
                                                     const int* __restrict__ iterPtr,
                                                     const __grid_constant__ JdsIterPtrs ipArg,
                                                     const int* __restrict__ perm,
                                                     const int* __restrict__ jdsCol,
                                                     const T* __restrict__ jdsVal,
                                                     const T* __restrict__ x,
                                                     T* __restrict__ y) {
  __shared__ int sIpBuf[PARAM ? 1 : kJdsSplitMaxDiag + 1];
  const int* sIp = PARAM ? ipArg.v : sIpBuf;
  if ((int)blockIdx.x < nMainBlocks) {
    if (!PARAM) {
      for (int t = threadIdx.x; t <= tSplit; t += blockDim.x) sIpBuf[t] = iterPtr[t];
      __syncthreads();
    }
    constexpr int G = kJdsRowGroup<T, RPT>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long warpFirst =
        ((long long)blockIdx.x * (blockDim.x >> 5) + warp) * (32LL * RPT);  // sorted row
    long long s[RPT];
    int r[RPT];
    T y0[RPT], acc[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      s[j] = warpFirst + 32 * j + lane;
      r[j] = s[j] < R ? __ldg(perm + s[j]) : -1;
      acc[j] = T(0);
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) y0[j] = (r[j] >= 0 && s[j] >= wTail) ? y[r[j]] : T(0);
    // G diagonals at a time: all their column and value loads are issued
    // before the gathers, and all gathers before the multiply-adds
    for (int t0 = 0; t0 < tSplit; t0 += G) {
      if (warpFirst >= sIp[t0 + 1] - sIp[t0]) break;  // widths shrink
      int c[RPT][G];
      T v[RPT][G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int t = t0 + g;
        const int a = t < tSplit ? sIp[t] : 0;
        const int wd = t < tSplit ? sIp[t + 1] - a : 0;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
          c[j][g] = -1;
          v[j][g] = T(0);
          if (s[j] < wd) {
            c[j][g] = ld_stream(jdsCol + a + s[j]);
            v[j][g] = ld_stream(jdsVal + a + s[j]);
          }
        }
      }
      T xg[RPT][G];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < RPT; ++j) xg[j][g] = c[j][g] >= 0 ? ld_x(x + c[j][g]) : T(0);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < RPT; ++j) acc[j] = fma_t(v[j][g], xg[j][g], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      if (r[j] >= 0) {
        if (s[j] < wTail)
          atomicAdd(y + r[j], acc[j]);  // the tail blocks add to this row too
        else
          y[r[j]] = y0[j] + acc[j];
      }
    }
  } else {
    // a tile of kJdsTailRows rows x kJdsTailDiags diagonals, walked by the
    // block's threads (a row per thread per pass, whatever the block size)
    const int b = blockIdx.x - nMainBlocks;
    const int rb = b % tailRowBlocks;
    const int tb = b / tailRowBlocks;
    const int tBeg = tSplit + tb * kJdsTailDiags;
    const int tEnd = min(tBeg + kJdsTailDiags, maxLen);
    const long long sEnd = min((long long)(rb + 1) * kJdsTailRows, (long long)wTail);
    for (long long s = (long long)rb * kJdsTailRows + threadIdx.x; s < sEnd; s += blockDim.x) {
      T acc = T(0);
      bool any = false;
      for (int t = tBeg; t < tEnd; ++t) {
        const int a = __ldg(iterPtr + t);
        const int wdt = __ldg(iterPtr + t + 1) - a;
        if (s >= wdt) break;  // widths shrink: no later diagonal reaches s
        const long long i = (long long)a + s;
        acc = fma_t(ld_stream(jdsVal + i), ld_x(x + ld_stream(jdsCol + i)), acc);
        any = true;
      }
      if (any) atomicAdd(y + perm[s], acc);
    }
  }
}

}  // namespace

// Threads per block of the short-lived kernels (each thread or warp streams
// its share once and exits). A block's slot on an SM frees only when its
// last warp ends, so smaller blocks keep more warps resident. Measured with
// 256 / 128 / 64 threads (cold L2): CSR on the 27-point stencil 191.6 /
// 178.8 / 172.1 us; ELL on the 5-point Laplacian 38.9 / 36.9 / 36.9 us and
// on the 27-point stencil 144.0 / 139.0 / 137.9 us; COO on the 27-point
// stencil 209.5 / 205.1 / 221.8 us; the COO row expansion on the Laplacian
// 24.2 / 23.3 / 22.4 us; SELL on the Laplacian 47.1 / 44.6 / 43.7 us and on
// the skewed matrix 138.9 / 133.0 / 131.7 us. JDS stays at 256: no gain on
// the stencils, and its long-row tail tiles of kJdsTailRows rows lose
// threads (skewed matrix 169.6 / 217.1 / 309.2 us).
constexpr int kCsrBlock = 64;
constexpr int kCooBlock = 128;
constexpr int kEllBlock = 64;
constexpr int kExpandBlock = 64;
constexpr int kJdsBlock = 256;
constexpr int kSellBlock = 64;

cudaError_t launch_expand_rows(int R, int Z, const int* rowPtrs, const CsrChunkDesc* desc,
                               int* rowIdx, cudaStream_t s) {
  if (R <= 0 || Z <= 0) return cudaSuccess;
  const long long perWarp = (long long)kExpandSupers * kCsrSuper;
  const long long warps = ((long long)Z + perWarp - 1) / perWarp;
  const unsigned grid = (unsigned)((warps * 32 + kExpandBlock - 1) / kExpandBlock);
  if (aligned16(rowIdx))
    k_expand_rows<true><<<grid, kExpandBlock, 0, s>>>(Z, rowPtrs, desc, rowIdx);
  else
    k_expand_rows<false><<<grid, kExpandBlock, 0, s>>>(Z, rowPtrs, desc, rowIdx);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_csr_chunk_masks(int R, int Z, const int* rowPtrs, int nChunks,
                                   CsrChunkDesc* desc, cudaStream_t s) {
  if (nChunks <= 0) return cudaSuccess;
  k_csr_chunk_masks<<<(unsigned)(((long long)nChunks + 255) / 256), 256, 0, s>>>(R, Z, rowPtrs,
                                                                                nChunks, desc);
  note_launches(1);
  return cudaGetLastError();
}

template <class T>
cudaError_t launch_spmv_csr(int R, int Z, const int* rowPtrs, const int* colIdx,
                            const T* value, const CsrChunkDesc* desc, const T* x,
                            T* y, cudaStream_t s) {
  if (Z <= 0 || R <= 0) return cudaSuccess;
  const bool vec = aligned16(colIdx) && aligned16(value);
  const long long warps = ((long long)Z + kCsrSuper - 1) / kCsrSuper;
  const unsigned blocks = (unsigned)((warps * 32 + kCsrBlock - 1) / kCsrBlock);
  if (vec)
    k_spmv_csr_wide<T, true><<<blocks, kCsrBlock, 0, s>>>(Z, rowPtrs, colIdx, value, desc, x, y);
  else
    k_spmv_csr_wide<T, false><<<blocks, kCsrBlock, 0, s>>>(Z, rowPtrs, colIdx, value, desc, x, y);
  note_launches(1);
  return cudaGetLastError();
}

template <class T>
cudaError_t launch_spmv_coo(int Z, const int* rowIdx, const int* colIdx, const T* value,
                            const T* x, T* y, bool dependent, cudaStream_t s) {
  if (Z <= 0) return cudaSuccess;
  const long long warps = ((long long)Z + 127) / 128;
  const long long blocks = (warps * 32 + kCooBlock - 1) / kCooBlock;
  const bool vec = aligned16(rowIdx) && aligned16(colIdx) && aligned16(value);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCooBlock);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const int dep = dependent ? 1 : 0;
  cudaError_t err;
  if (vec)
    err = cudaLaunchKernelEx(&cfg, k_spmv_coo<T, true>, Z, rowIdx, colIdx, value, x, y, dep);
  else
    err = cudaLaunchKernelEx(&cfg, k_spmv_coo<T, false>, Z, rowIdx, colIdx, value, x, y, dep);
  note_launches(1);
  return err;
}

template <class T>
cudaError_t launch_spmv_ell(int R, int K, const int* ellCol, const T* ellVal,
                            const T* x, T* y, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const bool vec4 = (R % 4 == 0) && aligned16(ellCol) && aligned16(ellVal) && aligned16(y);
  const long long threads = vec4 ? R / 4 : R;
  const long long blocks = (threads + kEllBlock - 1) / kEllBlock;
  if (vec4)
    k_spmv_ell<T, true><<<(unsigned)blocks, kEllBlock, 0, s>>>(R, K, ellCol, ellVal, x, y);
  else
    k_spmv_ell<T, false><<<(unsigned)blocks, kEllBlock, 0, s>>>(R, K, ellCol, ellVal, x, y);
  note_launches(1);
  return cudaGetLastError();
}

// sorted rows per thread of the JDS kernel's main part: 2 with 4-byte values
// (cold L2: 27-point stencil 147.1 -> 143.4 us against 1, the 5-point
// Laplacian unchanged at 43.0 us; 4 rows took 64 registers and measured
// 148.1 and 49.2 us), 1 with 8-byte values (bound by the fp64 adds)
template <class T>
constexpr int kJdsRowsPerThread = sizeof(T) == 4 ? 2 : 1;

template <class T>
cudaError_t launch_spmv_jds(int R, int maxLen, int tSplit, int wTail, const int* iterPtr,
                            const int* hostIterPtr, const int* perm, const int* jdsCol,
                            const T* jdsVal, const T* x, T* y, cudaStream_t s) {
  if (R <= 0 || maxLen <= 0) return cudaSuccess;
  // kJdsRowsPerThread<T> sorted rows per thread
  constexpr int rpt = kJdsRowsPerThread<T>;
  const long long mainBlocks = ((long long)R + (long long)kJdsBlock * rpt - 1) /
                               ((long long)kJdsBlock * rpt);
  long long tailBlocks = 0;
  int tailRowBlocks = 1;
  if (tSplit < maxLen && wTail > 0) {
    tailRowBlocks = (wTail + kJdsTailRows - 1) / kJdsTailRows;
    const long long diagBlocks = ((long long)(maxLen - tSplit) + kJdsTailDiags - 1) / kJdsTailDiags;
    tailBlocks = (long long)tailRowBlocks * diagBlocks;
  }
  JdsIterPtrs ip;
  // 4-byte values only: with 8-byte values the parameter form measured slower
  // (27-point stencil 227 -> 240 us, 5-point Laplacian 63.5 -> 72 us)
  const bool param = sizeof(T) == 4 && hostIterPtr != nullptr && tSplit <= kJdsParamDiags;
  for (int t = 0; t <= kJdsParamDiags; ++t) ip.v[t] = param && t <= tSplit ? hostIterPtr[t] : 0;
  if (param)
    k_spmv_jds<T, true, rpt><<<(unsigned)(mainBlocks + tailBlocks), kJdsBlock, 0, s>>>(
        R, maxLen, tSplit, wTail, (int)mainBlocks, tailRowBlocks, iterPtr, ip, perm, jdsCol,
        jdsVal, x, y);
  else
    k_spmv_jds<T, false, rpt><<<(unsigned)(mainBlocks + tailBlocks), kJdsBlock, 0, s>>>(
        R, maxLen, tSplit, wTail, (int)mainBlocks, tailRowBlocks, iterPtr, ip, perm, jdsCol,
        jdsVal, x, y);
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Sectioned ELL ("Regularized Formats (ELL, Hybrid ELL-COO and JDS)", section
// "JDS format", variant paragraph). Sorted rows in sections of S; slot t of
// row j of section k at secPtr[k] + t*h_k + j. The main part takes the first
// kSellMainSlots slots of every row, either 4 consecutive sorted rows per
// thread with 16-byte loads (k_spmv_sell4: with S % 4 == 0 every section
// starts on a multiple of 4 slots, so a full section's 4 rows are one aligned
// load of columns and one of values per slot) or two rows per thread
// (k_spmv_sell1), chosen by the mean slots per row. Slots past
// kSellMainSlots of the wide sections (a prefix, the rows being sorted) are
// cut into SellItems of 32 rows handled by extra warps, one row per lane; the
// rows of those sections add into y with atomics.
// ---------------------------------------------------------------------------
// slots whose loads a thread issues together (as kJdsGroup)
template <class T>
constexpr int kSellGroup = sizeof(T) == 4 ? 8 : 5;
// mean slots per row above which the main part takes a row per thread (with
// 4-byte values)
constexpr int kSellRowsWide = 8;

// Sum over slots [t0, t1) of the row at position j of the section starting at
// base (height h): kSellGroup<T> slots' loads issued before their gathers;
// padding slots (column -1) add nothing.
template <class T>
__device__ __forceinline__ T sell_row_slots(const int* __restrict__ col, const T* __restrict__ val,
                                            const T* __restrict__ x, int base, int h, int j,
                                            int t0, int t1) {
  T acc = T(0);
  // offsets of loaded slots stay below the slot count (< 2^31); unsigned, as
  // the offset is advanced past the last slot and may then wrap
  unsigned o = (unsigned)base + (unsigned)t0 * (unsigned)h + (unsigned)j;
  for (int tg = t0; tg < t1; tg += kSellGroup<T>) {
    int c[kSellGroup<T>];
    T v[kSellGroup<T>];
#pragma unroll
    for (int g = 0; g < kSellGroup<T>; ++g) {
      c[g] = -1;
      v[g] = T(0);
      if (tg + g < t1) {
        c[g] = ld_stream(col + o);
        v[g] = ld_stream(val + o);
      }
      o += (unsigned)h;
    }
    T xg[kSellGroup<T>];
#pragma unroll
    for (int g = 0; g < kSellGroup<T>; ++g) xg[g] = c[g] >= 0 ? ld_x(x + c[g]) : T(0);
#pragma unroll
    for (int g = 0; g < kSellGroup<T>; ++g) acc = fma_t(v[g], xg[g], acc);
  }
  return acc;
}

// Sorted rows per thread of k_spmv_sell1 (two, 32 apart; cold L2 against
// one: 27-point stencil 152.3 -> 143.4 us, skewed rows 131.7 -> 127.0 us)
// and their slot groups.
constexpr int kSell1Rows = 2;
constexpr int kSell1Group = 4;
// Slots [0, n[q]) of Q rows (row q: section base[q], height h[q], row j[q]),
// kSell1Group slots of every row loaded before their gathers.
template <class T, int Q>
__device__ __forceinline__ void sell_rows_slots(const int* __restrict__ col,
                                                const T* __restrict__ val,
                                                const T* __restrict__ x, const int (&base)[Q],
                                                const int (&h)[Q], const int (&j)[Q],
                                                const int (&n)[Q], T (&acc)[Q]) {
  unsigned o[Q];
  int nmax = 0;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    acc[q] = T(0);
    o[q] = (unsigned)base[q] + (unsigned)j[q];  // unsigned: may wrap past the last slot
    nmax = max(nmax, n[q]);
  }
  for (int tg = 0; tg < nmax; tg += kSell1Group) {
    int c[Q][kSell1Group];
    T v[Q][kSell1Group];
#pragma unroll
    for (int g = 0; g < kSell1Group; ++g)
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        c[q][g] = -1;
        v[q][g] = T(0);
        if (tg + g < n[q]) {
          c[q][g] = ld_stream(col + o[q]);
          v[q][g] = ld_stream(val + o[q]);
        }
        o[q] += (unsigned)h[q];
      }
    T xg[Q][kSell1Group];
#pragma unroll
    for (int g = 0; g < kSell1Group; ++g)
#pragma unroll
      for (int q = 0; q < Q; ++q) xg[q][g] = c[q][g] >= 0 ? ld_x(x + c[q][g]) : T(0);
#pragma unroll
    for (int g = 0; g < kSell1Group; ++g)
#pragma unroll
      for (int q = 0; q < Q; ++q) acc[q] = fma_t(v[q][g], xg[q][g], acc[q]);
  }
}

// Tail item id (slots [t0, t1) of 32 rows of a wide section, one per lane),
// added into y atomically.
template <class T>
__device__ __forceinline__ void sell_tail_item(int R, int S, int slots, long long id,
                                               const int* __restrict__ secPtr,
                                               const int* __restrict__ perm,
                                               const int* __restrict__ col,
                                               const T* __restrict__ val,
                                               const SellItem* __restrict__ items,
                                               const T* __restrict__ x, T* __restrict__ y) {
  const SellItem it = items[id];
  const int k0 = it.k * S;
  const int h = min(S, R - k0);
  const int j = it.j0 + (threadIdx.x & 31);
  if (j >= h) return;
  const int base = __ldg(secPtr + it.k);
  const int end = __ldg(secPtr + it.k + 1);
  if (end > slots || it.t1 > (end - base) / h) return;  // item beyond its section
  const int r = __ldg(perm + k0 + j);
  atomicAdd(y + r, sell_row_slots(col, val, x, base, h, j, it.t0, it.t1));
}

// Main part, one sorted row per thread: a warp's rows are consecutive slots
// of a section, so every 4-byte load is coalesced and kSellGroup<T> slots'
// loads go out together. Chosen for more than kSellRowsWide slots per row on
// average (27-point stencil: 153.6 us against 160.4 with 4 rows per thread;
// the random-length workload 138 against 160).
template <class T>
__global__ void __launch_bounds__(256) k_spmv_sell1(int R, int S, int slots, int mainBlocks,
                                                   const int* __restrict__ secPtr,
                                                   const int* __restrict__ perm,
                                                   const int* __restrict__ col,
                                                   const T* __restrict__ val,
                                                   const SellItem* __restrict__ items,
                                                   int nItems, const T* __restrict__ x,
                                                   T* __restrict__ y) {
  if ((int)blockIdx.x < mainBlocks) {
    // kSell1Rows sorted rows per thread, 32 apart (a warp's loads stay 32
    // consecutive slots of one section row)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long first =
        ((long long)blockIdx.x * (blockDim.x >> 5) + warp) * (32LL * kSell1Rows) + lane;
    int base[kSell1Rows], h[kSell1Rows], j[kSell1Rows], n[kSell1Rows], r[kSell1Rows],
        w[kSell1Rows];
    T y0[kSell1Rows];
#pragma unroll
    for (int q = 0; q < kSell1Rows; ++q) {
      const long long s = first + 32LL * q;
      r[q] = -1;
      n[q] = 0;
      w[q] = 0;
      base[q] = 0;
      h[q] = 1;
      j[q] = 0;
      if (s < R) {
        const int k = (int)(s / S);
        const int k0 = k * S;
        h[q] = min(S, R - k0);
        j[q] = (int)(s - k0);
        // the loads that do not depend on each other first: section bounds,
        // the row's original index, then its y value
        base[q] = __ldg(secPtr + k);
        const int end = __ldg(secPtr + k + 1);
        r[q] = __ldg(perm + s);
        w[q] = end <= slots ? (end - base[q]) / h[q] : 0;  // never past the arrays
        n[q] = min(w[q], kSellMainSlots);
      }
    }
#pragma unroll
    for (int q = 0; q < kSell1Rows; ++q) y0[q] = r[q] >= 0 ? y[r[q]] : T(0);
    T acc[kSell1Rows];
    sell_rows_slots<T, kSell1Rows>(col, val, x, base, h, j, n, acc);
#pragma unroll
    for (int q = 0; q < kSell1Rows; ++q) {
      if (r[q] < 0) continue;
      if (w[q] > kSellMainSlots)
        atomicAdd(y + r[q], acc[q]);  // tail items add to this row too
      else
        y[r[q]] = y0[q] + acc[q];
    }
  } else {
    const long long id = (long long)(blockIdx.x - mainBlocks) * (blockDim.x >> 5) +
                         (threadIdx.x >> 5);
    if (id < nItems) sell_tail_item(R, S, slots, id, secPtr, perm, col, val, items, x, y);
  }
}

template <class T, bool VEC>
__device__ __forceinline__ void sell_rows(const int* __restrict__ col,
                                          const T* __restrict__ val,
                                          const T* __restrict__ x, long long base, int h,
                                          int j, int n, int t0, int t1, T acc[4]) {
  if (VEC && n == 4 && (h & 3) == 0) {
    const long long hq = h >> 2;
    const int4* c4 = reinterpret_cast<const int4*>(col + base + (long long)t0 * h + j);
    const T* v4 = val + base + (long long)t0 * h + j;  // 4 values per step of h
    int t = t0;
    for (; t + 4 <= t1; t += 4, c4 += 4 * hq, v4 += 4 * (size_t)h) {
      int4 c[4];
      Vec4<T> v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c[u] = ld_stream(c4 + u * hq);
        v[u] = ld4_stream(v4 + u * (size_t)h);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c[u].x >= 0) acc[0] = fma_t(v[u].x, ld_x(x + c[u].x), acc[0]);
        if (c[u].y >= 0) acc[1] = fma_t(v[u].y, ld_x(x + c[u].y), acc[1]);
        if (c[u].z >= 0) acc[2] = fma_t(v[u].z, ld_x(x + c[u].z), acc[2]);
        if (c[u].w >= 0) acc[3] = fma_t(v[u].w, ld_x(x + c[u].w), acc[3]);
      }
    }
    for (; t < t1; ++t, c4 += hq, v4 += h) {
      const int4 c = ld_stream(c4);
      const Vec4<T> v = ld4_stream(v4);
      if (c.x >= 0) acc[0] = fma_t(v.x, ld_x(x + c.x), acc[0]);
      if (c.y >= 0) acc[1] = fma_t(v.y, ld_x(x + c.y), acc[1]);
      if (c.z >= 0) acc[2] = fma_t(v.z, ld_x(x + c.z), acc[2]);
      if (c.w >= 0) acc[3] = fma_t(v.w, ld_x(x + c.w), acc[3]);
    }
  } else {
    // the last, partial section (h % 4 != 0), or S % 4 != 0
    for (int t = t0; t < t1; ++t) {
      const long long o = base + (long long)t * h + j;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (u < n) {
          const int c = ld_stream(col + o + u);
          const T v = ld_stream(val + o + u);
          if (c >= 0) acc[u] = fma_t(v, ld_x(x + c), acc[u]);
        }
      }
    }
  }
}

// perm[s0 .. s0+n-1] (one 16-byte load when n == 4: s0 is then a multiple of 4)
template <bool VEC>
__device__ __forceinline__ void sell_perm(const int* __restrict__ perm, int s0, int n, int r[4]) {
  if (VEC && n == 4) {
    const int4 p = __ldg(reinterpret_cast<const int4*>(perm + s0));
    r[0] = p.x; r[1] = p.y; r[2] = p.z; r[3] = p.w;
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u) r[u] = u < n ? __ldg(perm + s0 + u) : 0;
  }
}

// Main part, 4 consecutive sorted rows per thread (1 when S % 4 != 0) with
// 16-byte loads: the section bounds, perm and y are loaded once per 4 rows.
// Chosen for at most kSellRowsWide slots per row on average, where those
// loads weigh most (laplace2d: 48.3 us against 61.5 with a row per thread).
template <class T, bool VEC>
__global__ void __launch_bounds__(256, 4) k_spmv_sell4(int R, int S, int slots, int mainBlocks,
                                                       const int* __restrict__ secPtr,
                                                       const int* __restrict__ perm,
                                                       const int* __restrict__ col,
                                                       const T* __restrict__ val,
                                                       const SellItem* __restrict__ items,
                                                       int nItems, const T* __restrict__ x,
                                                       T* __restrict__ y) {
  constexpr int kRows = VEC ? 4 : 1;
  T acc[4] = {T(0), T(0), T(0), T(0)};
  int r[4];
  if ((int)blockIdx.x < mainBlocks) {
    const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (q * kRows >= R) return;
    const int s0 = (int)(q * kRows);
    const int k = s0 / S;
    const int k0 = k * S;
    const int h = min(S, R - k0);
    const int n = min(kRows, R - s0);
    // issue the loads that do not depend on each other before the slot loop:
    // section bounds, the rows' original indices, then their y values
    const int base = __ldg(secPtr + k);
    const int end = __ldg(secPtr + k + 1);
    sell_perm<VEC>(perm, s0, n, r);
    T y0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) y0[u] = u < n ? y[r[u]] : T(0);
    const int w = end <= slots ? (end - base) / h : 0;  // never past the arrays
    sell_rows<T, VEC>(col, val, x, base, h, s0 - k0, n, 0, min(w, kSellMainSlots), acc);
    const bool atomic = w > kSellMainSlots;  // tail items add to these rows too
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u < n) {
        if (atomic)
          atomicAdd(y + r[u], acc[u]);
        else
          y[r[u]] = y0[u] + acc[u];
      }
    }
  } else {
    const long long id = (long long)(blockIdx.x - mainBlocks) * (blockDim.x >> 5) +
                         (threadIdx.x >> 5);
    if (id < nItems) sell_tail_item(R, S, slots, id, secPtr, perm, col, val, items, x, y);
  }
}

template <class T>
cudaError_t launch_spmv_sell(int R, int S, int slots, const int* secPtr, const int* perm,
                             const int* sellCol, const T* sellVal, const SellItem* items,
                             int nItems, const T* x, T* y, cudaStream_t s) {
  if (R <= 0 || S <= 0) return cudaSuccess;
  constexpr int kSellWarps = kSellBlock / 32;
  // an item per warp
  const long long tailBlocks = ((long long)nItems + kSellWarps - 1) / kSellWarps;
  // 8-byte values keep 4 rows per thread (a row per thread measured 229 us
  // against 223 on the 27-point stencil)
  if (sizeof(T) == 4 && (long long)slots > (long long)kSellRowsWide * R) {
    // kSell1Rows sorted rows per thread
    constexpr long long rowsPerBlock = (long long)kSellBlock * kSell1Rows;
    const long long mainBlocks = ((long long)R + rowsPerBlock - 1) / rowsPerBlock;
    k_spmv_sell1<T><<<(unsigned)(mainBlocks + tailBlocks), kSellBlock, 0, s>>>(
        R, S, slots, (int)mainBlocks, secPtr, perm, sellCol, sellVal, items, nItems, x, y);
  } else {
    const bool vec = (S & 3) == 0;
    const long long threads = vec ? ((long long)R + 3) / 4 : R;
    const long long mainBlocks = (threads + kSellBlock - 1) / kSellBlock;
    if (vec)
      k_spmv_sell4<T, true><<<(unsigned)(mainBlocks + tailBlocks), kSellBlock, 0, s>>>(
          R, S, slots, (int)mainBlocks, secPtr, perm, sellCol, sellVal, items, nItems, x, y);
    else
      k_spmv_sell4<T, false><<<(unsigned)(mainBlocks + tailBlocks), kSellBlock, 0, s>>>(
          R, S, slots, (int)mainBlocks, secPtr, perm, sellCol, sellVal, items, nItems, x, y);
  }
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// x-blocked list ("Introduction to sparse computing and performance
// bottleneck location", section "Building the problem framework": a thread
// block handles only the nonzeros whose columns fall in one chunk of x, so
// the gather stays local). Persistent CTAs, one per SM: CTA b takes the b-th
// nnz-balanced slice of the chunk-ordered list; for every chunk its slice
// meets it stages that chunk of x (B floats) in shared memory, then each warp
// walks the slice kXbUnroll x 32 entries at a time, lane l taking entries l,
// l + 32, ... (every load coalesced, all of them issued before the first
// use), gathers from shared memory and adds into y with fire-and-forget
// atomics. Rows ascend inside a chunk, so equal rows of one instruction's 32
// entries sit in adjacent lanes: where any lane continues its neighbour's
// row (a 27-point stencil row keeps up to 27 entries in one chunk, the skewed
// matrix's long rows many more) the runs are summed by a segmented shuffle
// scan first, one reduction per run; where none does (scattered columns,
// about one entry per row in a chunk) each product goes to y by itself. The
// test costs one shuffle and one ballot per 32 entries. Cold L2: 27-point
// stencil 554.6 -> 262.1 us, skewed rows 115.3 -> 95.2 us (its long rows'
// reductions all fall on a few addresses), 5-point Laplacian (runs of 5)
// 65.5 -> 69.6 us. Taking the scan only where at least 28 of the 32 lanes
// continue a run kept the Laplacian at 67.6 us but left the skewed matrix
// at 108.6 us; a scan of only as many steps as the longest run needs (a
// runtime bound) measured 75.8 and 326 us. With 8-byte values every product
// goes to y by itself: the scan's fp64 adds cost more than the reductions.
// ---------------------------------------------------------------------------
constexpr int kXbUnroll = 8;

// THREADS = 1024 for the widest chunks (one CTA per SM); 512 when the chunk
// leaves shared memory for two or more CTAs per SM, so that one CTA stages
// its chunk while the others stream entries.
template <class T, int THREADS>
__global__ void __launch_bounds__(THREADS, 1) k_spmv_xb(int C, int B, int nch,
                                                           const int* __restrict__ chunkPtr,
                                                           const int* __restrict__ xbRow,
                                                           const unsigned short* __restrict__ xbCol,
                                                           const T* __restrict__ xbVal,
                                                           const T* __restrict__ x,
                                                           T* __restrict__ y) {
  extern __shared__ int4 sXraw[];
  T* sX = reinterpret_cast<T*>(sXraw);
  __shared__ int sFirst;
  const long long groups = (long long)__ldg(chunkPtr + nch) >> 2;  // slots are 4-aligned
  const long long lo = 4 * (groups * blockIdx.x / gridDim.x);
  const long long hi = 4 * (groups * (blockIdx.x + 1) / gridDim.x);
  if (lo >= hi) return;
  if (threadIdx.x == 0) {  // first chunk that ends after lo
    int a = 0, b = nch - 1;
    while (a < b) {
      const int m = (a + b) >> 1;
      if (__ldg(chunkPtr + m + 1) > lo) b = m; else a = m + 1;
    }
    sFirst = a;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nWarps = blockDim.x >> 5;
  constexpr int kStep = 32 * kXbUnroll;
  for (int c = sFirst; c < nch; ++c) {
    const long long cs = __ldg(chunkPtr + c);
    if (cs >= hi) break;
    const long long s0 = cs > lo ? cs : lo;
    const long long ce = __ldg(chunkPtr + c + 1);
    const long long s1 = ce < hi ? ce : hi;
    if (s0 >= s1) continue;
    // stage x[cB, cB + n) (the previous chunk's readers are past the barrier)
    const long long xb = (long long)c * B;
    const int n = (int)(C - xb < B ? C - xb : B);
    __syncthreads();
    const T* xs = x + xb;
    if ((reinterpret_cast<uintptr_t>(xs) & 15) == 0) {
      // 16-byte copies of the chunk's bytes, then the remaining elements
      constexpr int kPer16 = 16 / sizeof(T);
      const int4* x16 = reinterpret_cast<const int4*>(xs);
      for (int i = threadIdx.x; i < n / kPer16; i += blockDim.x) sXraw[i] = __ldg(x16 + i);
      for (int i = n / kPer16 * kPer16 + threadIdx.x; i < n; i += blockDim.x) sX[i] = __ldg(xs + i);
    } else {
      for (int i = threadIdx.x; i < n; i += blockDim.x) sX[i] = __ldg(xs + i);
    }
    __syncthreads();
    for (long long e0 = s0 + (long long)warp * kStep; e0 < s1; e0 += (long long)nWarps * kStep) {
      int row[kXbUnroll];
      T val[kXbUnroll];
      int col[kXbUnroll];
#pragma unroll
      for (int j = 0; j < kXbUnroll; ++j) {
        const long long e = e0 + 32 * j + lane;
        const bool in = e < s1;
        row[j] = in ? __ldcs(xbRow + e) : -1;
        val[j] = in ? __ldcs(xbVal + e) : T(0);
        col[j] = in ? (int)__ldcs(xbCol + e) : 0;
      }
#pragma unroll
      for (int j = 0; j < kXbUnroll; ++j) {
        // 32 consecutive entries, rows ascending: equal rows sit in adjacent
        // lanes. With no lane continuing its left neighbour's row (scattered
        // columns) each product goes to y by itself; otherwise each run of
        // equal row is summed by a segmented shuffle scan and its last lane
        // adds the sum, one reduction per run (padding: row -1, product 0)
        const T prod = row[j] >= 0 ? val[j] * sX[col[j]] : T(0);
        if constexpr (sizeof(T) == 8) {
          // 8-byte values: the fp64 adds of a scan would cost more than the
          // reductions they save (27-point stencil 432 -> 1292 us)
          if (row[j] >= 0) atomicAdd(y + row[j], prod);
          continue;
        }
        const int left = __shfl_up_sync(kFullMask, row[j], 1);
        const unsigned cont = __ballot_sync(kFullMask, lane > 0 && left == row[j]);
        if (cont == 0u) {  // warp-uniform
          if (row[j] >= 0) atomicAdd(y + row[j], prod);
        } else {
          const int segStart = 31 - __clz(~cont & (0xffffffffu >> (31 - lane)));
          T v = prod;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const T o = __shfl_up_sync(kFullMask, v, off);
            if (lane - off >= segStart) v += o;
          }
          const bool last = lane == 31 || ((cont >> (lane + 1)) & 1u) == 0u;
          if (last && row[j] >= 0) atomicAdd(y + row[j], v);
        }
      }
    }
  }
}

template <class T>
cudaError_t launch_spmv_xb(int C, int B, int nch, const int* chunkPtr, const int* xbRow,
                           const unsigned short* xbCol, const T* xbVal, const T* x,
                           T* y, cudaStream_t s) {
  if (nch <= 0) return cudaSuccess;
  const size_t smem = ((size_t)B * sizeof(T) + 15) / 16 * 16;
  const bool wide = smem > 100 * 1024;  // one CTA per SM
  // per device and variant: the dynamic shared-memory limit raised once,
  // and the blocks per SM for the last chunk size seen
  constexpr int kDevs = 64;
  static bool raised[2][kDevs] = {};
  static size_t lastSmem[2][kDevs] = {};
  static int lastPerSm[2][kDevs] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < kDevs;
  const int v = wide ? 1 : 0;
  const void* fn = wide ? reinterpret_cast<const void*>(k_spmv_xb<T, 1024>)
                        : reinterpret_cast<const void*>(k_spmv_xb<T, 512>);
  const int threads = wide ? 1024 : 512;
  if (!cache || !raised[v][dev]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kXbSmemBytes);
    if (e != cudaSuccess) return e;
    if (cache) raised[v][dev] = true;
  }
  int perSm = cache && lastSmem[v][dev] == smem ? lastPerSm[v][dev] : 0;
  if (perSm < 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&perSm, fn, threads, smem) !=
            cudaSuccess || perSm < 1) {
      cudaGetLastError();
      perSm = 1;
    }
    if (cache) {
      lastSmem[v][dev] = smem;
      lastPerSm[v][dev] = perSm;
    }
  }
  const unsigned grid = (unsigned)(perSm * num_sms());
  if (wide)
    k_spmv_xb<T, 1024><<<grid, 1024, smem, s>>>(C, B, nch, chunkPtr, xbRow, xbCol, xbVal, x, y);
  else
    k_spmv_xb<T, 512><<<grid, 512, smem, s>>>(C, B, nch, chunkPtr, xbRow, xbCol, xbVal, x, y);
  note_launches(1);
  return cudaGetLastError();
}

// the two value types
#define SPMV_INSTANTIATE(T)                                                                     \
  template cudaError_t launch_spmv_csr<T>(int, int, const int*, const int*, const T*,          \
                                          const CsrChunkDesc*, const T*, T*, cudaStream_t);    \
  template cudaError_t launch_spmv_coo<T>(int, const int*, const int*, const T*, const T*, T*, \
                                          bool, cudaStream_t);                                  \
  template cudaError_t launch_spmv_ell<T>(int, int, const int*, const T*, const T*, T*,        \
                                          cudaStream_t);                                        \
  template cudaError_t launch_spmv_jds<T>(int, int, int, int, const int*, const int*,          \
                                          const int*, const int*, const T*, const T*, T*,      \
                                          cudaStream_t);                                       \
  template cudaError_t launch_spmv_sell<T>(int, int, int, const int*, const int*, const int*,  \
                                           const T*, const SellItem*, int, const T*, T*,        \
                                           cudaStream_t);                                       \
  template cudaError_t launch_spmv_xb<T>(int, int, int, const int*, const int*,                \
                                         const unsigned short*, const T*, const T*, T*,         \
                                         cudaStream_t);
SPMV_INSTANTIATE(float)
SPMV_INSTANTIATE(double)
#undef SPMV_INSTANTIATE

}  // namespace spmv
