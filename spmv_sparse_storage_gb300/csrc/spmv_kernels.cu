// spmv_kernels.cu -- y <- A*x + y for each storage format.
//
// Operation: sparse matrix-vector multiplication and accumulation (PMPP
// notes, "Sparse Matrices and Basic Formats (COO and CSR)", section
// "Background & SpMV"). Every kernel is memory-bound: per nonzero it moves a
// 4-byte value and a 4-byte column index and does one multiply-add ("Regularized
// Formats (ELL, Hybrid ELL-COO and JDS)", section "Summary": 0.25 op/byte),
// so the designs below are about streaming those bytes at HBM speed, keeping
// the gathered x resident in L2, and balancing the work.
#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

// ===========================================================================
// CSR, nnz-balanced (merge path).
//
// The pages' kernels give a row to a thread ("CSR format and SpMV") or a warp
// ("[CUDA performance tuning] ...", section 2.2); both leave threads idle when
// row lengths differ ("Introduction to sparse computing ...", section
// "Building the problem framework": split work by nonzero count and split
// very long rows). Here each CTA owns an equal share of the merged sequence
// of row ends and nonzeros (kCsrTileItems items), located by a merge-path
// search done once at handle creation (tileRow). A CTA:
//   1. stages its slice of rowPtrs and the products value[k]*x[colIdx[k]] of
//      its nonzeros in shared memory (value/colIdx streamed with 16-byte
//      loads when aligned);
//   2. splits its items again, IPT per thread, by a merge-path search in
//      shared memory, and each thread sums its run of products, closing rows
//      as it meets their ends;
//   3. adds each row's sum into y: rows wholly inside the tile with a plain
//      read-modify-write (coalesced over consecutive rows), the first and last
//      row of the tile (possibly shared with a neighbour tile) atomically.
// ===========================================================================
template <int THREADS, int IPT, bool VEC>
__global__ void __launch_bounds__(THREADS, 4) k_spmv_csr(int R, int Z, const int* __restrict__ rowPtrs,
                                                      const int* __restrict__ colIdx,
                                                      const float* __restrict__ value,
                                                      const int* __restrict__ tileRow,
                                                      const float* __restrict__ x,
                                                      float* __restrict__ y) {
  constexpr int NT = THREADS * IPT;
  __shared__ float sProd[NT];
  __shared__ int sRp[NT + 1];
  __shared__ float sAcc[NT + 1];

  const int tile = blockIdx.x;
  const long long total = (long long)R + Z;
  const long long d0 = (long long)tile * NT;
  const long long d1 = d0 + NT < total ? d0 + NT : total;
  const int i0 = tileRow[tile];
  const int i1 = tileRow[tile + 1];
  const int j0 = (int)(d0 - i0);
  const int j1 = (int)(d1 - i1);
  const int nr = i1 - i0;  // rows whose end lies in this tile
  const int nn = j1 - j0;  // nonzeros of this tile

  // 1a. rowPtrs[i0 .. i1] (i1 <= R, so every entry exists)
  for (int q = threadIdx.x; q <= nr; q += THREADS) {
    sRp[q] = rowPtrs[i0 + q];
    sAcc[q] = 0.0f;
  }
  // 1b. products of nonzeros j0 .. j1-1
  if (VEC) {
    const int v0 = (j0 + 3) & ~3;          // first 16-byte aligned index
    const int v1 = j1 & ~3;                // end of the aligned body
    if (v0 < v1) {
      const int nvec = (v1 - v0) >> 2;
      const int4* c4 = reinterpret_cast<const int4*>(colIdx + v0);
      const float4* a4 = reinterpret_cast<const float4*>(value + v0);
      float* dst = sProd + (v0 - j0);
      for (int q = threadIdx.x; q < nvec; q += THREADS) {
        const int4 c = ld_stream(c4 + q);
        const float4 a = ld_stream(a4 + q);
        float4 p;
        p.x = a.x * ld_x(x + c.x);
        p.y = a.y * ld_x(x + c.y);
        p.z = a.z * ld_x(x + c.z);
        p.w = a.w * ld_x(x + c.w);
        dst[4 * q + 0] = p.x;
        dst[4 * q + 1] = p.y;
        dst[4 * q + 2] = p.z;
        dst[4 * q + 3] = p.w;
      }
      // unaligned head [j0, v0) and tail [v1, j1): at most 3 each
      const int t = threadIdx.x;
      if (t < v0 - j0) {
        const int k = j0 + t;
        sProd[k - j0] = ld_stream(value + k) * ld_x(x + ld_stream(colIdx + k));
      } else if (t >= 4 && t < 4 + (j1 - v1)) {
        const int k = v1 + (t - 4);
        sProd[k - j0] = ld_stream(value + k) * ld_x(x + ld_stream(colIdx + k));
      }
    } else {
      for (int k = j0 + threadIdx.x; k < j1; k += THREADS)
        sProd[k - j0] = ld_stream(value + k) * ld_x(x + ld_stream(colIdx + k));
    }
  } else {
    for (int k = j0 + threadIdx.x; k < j1; k += THREADS)
      sProd[k - j0] = ld_stream(value + k) * ld_x(x + ld_stream(colIdx + k));
  }
  __syncthreads();

  // 2. per-thread merge path over (row ends sRp[1..nr], nonzeros j0..j1-1)
  const int items = nr + nn;
  const int dt = threadIdx.x * IPT < items ? threadIdx.x * IPT : items;
  int lo = dt - nn > 0 ? dt - nn : 0;
  int hi = dt < nr ? dt : nr;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sRp[mid + 1] <= j0 + dt - 1 - mid)
      lo = mid + 1;
    else
      hi = mid;
  }
  int li = lo;         // local row
  int k = j0 + dt - lo;  // global nonzero index
  float acc = 0.0f;
  bool firstEnd = true;
  const int dEnd = dt + IPT < items ? dt + IPT : items;
#pragma unroll
  for (int it = 0; it < IPT; ++it) {
    if (dt + it < dEnd) {
      if (li < nr && sRp[li + 1] <= k) {
        // row i0 + li ends here
        if (firstEnd)
          atomicAdd(&sAcc[li], acc);  // may have started in an earlier thread
        else
          sAcc[li] = acc;  // started and ended inside this thread
        firstEnd = false;
        acc = 0.0f;
        ++li;
      } else {
        acc += sProd[k - j0];
        ++k;
      }
    }
  }
  if (acc != 0.0f) atomicAdd(&sAcc[li], acc);  // row continues in the next thread
  __syncthreads();

  // 3. write-out, coalesced over rows i0 .. i1
  for (int q = threadIdx.x; q <= nr; q += THREADS) {
    const int row = i0 + q;
    if (row >= R) break;
    const float v = sAcc[q];
    if (q == nr) {
      // row i1: its end is in a later tile; contribute only if it has
      // nonzeros here
      if (sRp[nr] < j1) atomicAdd(y + row, v);
    } else if (q == 0 && sRp[0] < j0) {
      atomicAdd(y + row, v);  // started in an earlier tile
    } else {
      y[row] += v;
    }
  }
}

// ===========================================================================
// ELL ("Regularized Formats ...", section "ELL format: padding +
// transposition"): thread per row, slot t of row r at t*numRows + r, so a
// warp reads consecutive slots (coalesced). The loop runs over all K slots;
// padding slots (column -1) skip the x gather and add nothing, so nnzPerRow
// is never read. VEC4: numRows % 4 == 0 and 16-byte aligned arrays, a thread
// handles 4 consecutive rows with 16-byte loads.
// ===========================================================================
template <bool VEC4>
__global__ void __launch_bounds__(256, 4) k_spmv_ell(int R, int K, const int* __restrict__ ellCol,
                                                  const float* __restrict__ ellVal,
                                                  const float* __restrict__ x,
                                                  float* __restrict__ y) {
  // let a programmatically dependent kernel (the COO part of HYB) start its
  // loads; it waits for this grid to finish before it writes y
  grid_dependency_trigger();
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (VEC4) {
    const long long ld = R >> 2;
    if (q >= ld) return;
    const int4* c4 = reinterpret_cast<const int4*>(ellCol);
    const float4* v4 = reinterpret_cast<const float4*>(ellVal);
    float4* y4 = reinterpret_cast<float4*>(y);
    const float4 y0 = y4[q];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int t = 0;
    for (; t + 4 <= K; t += 4) {
      int4 c[4];
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c[u] = ld_stream(c4 + (size_t)(t + u) * ld + q);
        v[u] = ld_stream(v4 + (size_t)(t + u) * ld + q);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c[u].x >= 0) acc.x = fmaf(v[u].x, ld_x(x + c[u].x), acc.x);
        if (c[u].y >= 0) acc.y = fmaf(v[u].y, ld_x(x + c[u].y), acc.y);
        if (c[u].z >= 0) acc.z = fmaf(v[u].z, ld_x(x + c[u].z), acc.z);
        if (c[u].w >= 0) acc.w = fmaf(v[u].w, ld_x(x + c[u].w), acc.w);
      }
    }
    for (; t < K; ++t) {
      const int4 c = ld_stream(c4 + (size_t)t * ld + q);
      const float4 v = ld_stream(v4 + (size_t)t * ld + q);
      if (c.x >= 0) acc.x = fmaf(v.x, ld_x(x + c.x), acc.x);
      if (c.y >= 0) acc.y = fmaf(v.y, ld_x(x + c.y), acc.y);
      if (c.z >= 0) acc.z = fmaf(v.z, ld_x(x + c.z), acc.z);
      if (c.w >= 0) acc.w = fmaf(v.w, ld_x(x + c.w), acc.w);
    }
    y4[q] = make_float4(y0.x + acc.x, y0.y + acc.y, y0.z + acc.z, y0.w + acc.w);
  } else {
    if (q >= R) return;
    const float y0 = y[q];
    float acc = 0.0f;
    int t = 0;
    for (; t + 4 <= K; t += 4) {
      int c[4];
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c[u] = ld_stream(ellCol + (size_t)(t + u) * R + q);
        v[u] = ld_stream(ellVal + (size_t)(t + u) * R + q);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c[u] >= 0) acc = fmaf(v[u], ld_x(x + c[u]), acc);
    }
    for (; t < K; ++t) {
      const int c = ld_stream(ellCol + (size_t)t * R + q);
      const float v = ld_stream(ellVal + (size_t)t * R + q);
      if (c >= 0) acc = fmaf(v, ld_x(x + c), acc);
    }
    y[q] = y0 + acc;
  }
}

// ===========================================================================
// COO ("Sparse Matrices and Basic Formats ...", section "COO format and
// SpMV" uses one atomicAdd per nonzero, and same-row nonzeros contend). Here
// a warp takes 128 consecutive entries, 4 per lane (16-byte loads when
// aligned), reduces runs of equal row index first inside each lane and then
// across lanes with a segmented shuffle scan, and issues ONE atomicAdd per
// run. Correct for any entry order (only adjacent equal rows merge); fastest
// when entries are grouped by row, as the converter produces them.
// `dependent`: the kernel was launched as a programmatic dependent of the
// ELL part of HYB; it computes everything before waiting for that kernel and
// only then touches y.
// ===========================================================================
template <bool VEC>
__global__ void __launch_bounds__(256) k_spmv_coo(int Z, const int* __restrict__ rowIdx,
                                                  const int* __restrict__ colIdx,
                                                  const float* __restrict__ value,
                                                  const float* __restrict__ x,
                                                  float* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long base = warp * 128 + 4 * lane;

  int row[4];
  float p[4];
  if (VEC && base + 4 <= Z) {
    const int4 r4 = ld_stream(reinterpret_cast<const int4*>(rowIdx + base));
    const int4 c4 = ld_stream(reinterpret_cast<const int4*>(colIdx + base));
    const float4 v4 = ld_stream(reinterpret_cast<const float4*>(value + base));
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
        p[e] = 0.0f;
      }
    }
  }
  // in-lane run sums: s[e] = sum of the run ending at e
  float s[4];
  s[0] = p[0];
#pragma unroll
  for (int e = 1; e < 4; ++e) s[e] = (row[e] == row[e - 1]) ? s[e - 1] + p[e] : p[e];
  const int hEnd = row[1] != row[0] ? 0 : row[2] != row[1] ? 1 : row[3] != row[2] ? 2 : 3;
  const bool single = (hEnd == 3);
  const int rh = row[0], rt = row[3];
  const float sh = s[hEnd], st = s[3];

  // across lanes: w = tail-run sum carried right while lanes are one run
  const int prevRt = __shfl_up_sync(kFullMask, rt, 1);
  const bool connected = lane > 0 && prevRt == rh;
  const unsigned heads = __ballot_sync(kFullMask, !(single && connected));
  const int segStart = 31 - __clz(heads & (0xffffffffu >> (31 - lane)));
  float w = st;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(kFullMask, w, off);
    if (lane - off >= segStart) w += o;
  }
  const float wPrev = __shfl_up_sync(kFullMask, w, 1);
  const float carryIn = connected ? wPrev : 0.0f;
  const int nextRh = __shfl_down_sync(kFullMask, rh, 1);
  const bool tailEnds = (lane == 31) || nextRh != rt;

  grid_dependency_wait();
  if (single) {
    if (tailEnds && rt >= 0) atomicAdd(y + rt, st + carryIn);
  } else {
    if (rh >= 0) atomicAdd(y + rh, sh + carryIn);
#pragma unroll
    for (int e = 1; e < 3; ++e)  // runs strictly inside the lane
      if (e > hEnd && row[e] != row[e + 1] && row[e] >= 0) atomicAdd(y + row[e], s[e]);
    if (tailEnds && rt >= 0) atomicAdd(y + rt, st);
  }
}

// ===========================================================================
// JDS ("Regularized Formats ...", section "JDS format": a thread takes a
// sorted row and walks the jagged diagonals from iterPtr; the page leaves the
// kernel as an exercise). Diagonal t holds one entry for every sorted row
// s < width(t), contiguous in s, so a warp's loads are coalesced. Widths only
// shrink with t; the first tSplit diagonals (those at least
// kJdsSplitMinWidth wide, at most kJdsSplitMaxDiag of them) run one thread
// per sorted row. The remaining diagonals belong to the few longest rows
// (s < wTail) and would serialise one thread over thousands of entries, so
// they are split into blocks of kJdsTailRows rows x kJdsTailDiags diagonals
// that run in parallel and add their partial sums atomically. The result of
// sorted row s goes straight to y[perm[s]] (the page permutes the result back
// with the row array).
// ===========================================================================
__global__ void __launch_bounds__(256) k_spmv_jds(int R, int maxLen, int tSplit, int wTail,
                                                  int nMainBlocks, int tailRowBlocks,
                                                  const int* __restrict__ iterPtr,
                                                  const int* __restrict__ perm,
                                                  const int* __restrict__ jdsCol,
                                                  const float* __restrict__ jdsVal,
                                                  const float* __restrict__ x,
                                                  float* __restrict__ y) {
  __shared__ int sIp[kJdsSplitMaxDiag + 1];
  if ((int)blockIdx.x < nMainBlocks) {
    for (int t = threadIdx.x; t <= tSplit; t += blockDim.x) sIp[t] = iterPtr[t];
    __syncthreads();
    const long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= R) return;
    // number of leading diagonals wider than s (binary search; widths shrink)
    int lo = 0, hi = tSplit;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sIp[mid + 1] - sIp[mid] > s)
        lo = mid + 1;
      else
        hi = mid;
    }
    const int n = lo;
    float acc = 0.0f;
    int t = 0;
    for (; t + 4 <= n; t += 4) {
      int c[4];
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const long long i = (long long)sIp[t + u] + s;
        c[u] = ld_stream(jdsCol + i);
        v[u] = ld_stream(jdsVal + i);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) acc = fmaf(v[u], ld_x(x + c[u]), acc);
    }
    for (; t < n; ++t) {
      const long long i = (long long)sIp[t] + s;
      acc = fmaf(ld_stream(jdsVal + i), ld_x(x + ld_stream(jdsCol + i)), acc);
    }
    const int r = perm[s];
    if (s < wTail)
      atomicAdd(y + r, acc);  // the tail blocks add to this row too
    else
      y[r] += acc;
  } else {
    const int b = blockIdx.x - nMainBlocks;
    const int rb = b % tailRowBlocks;
    const int tb = b / tailRowBlocks;
    const long long s = (long long)rb * kJdsTailRows + threadIdx.x;
    const int tBeg = tSplit + tb * kJdsTailDiags;
    const int tEnd = min(tBeg + kJdsTailDiags, maxLen);
    if (s >= wTail) return;
    float acc = 0.0f;
    bool any = false;
    for (int t = tBeg; t < tEnd; ++t) {
      const int a = __ldg(iterPtr + t);
      const int wdt = __ldg(iterPtr + t + 1) - a;
      if (s >= wdt) break;  // widths shrink: no later diagonal reaches s
      const long long i = (long long)a + s;
      acc = fmaf(ld_stream(jdsVal + i), ld_x(x + ld_stream(jdsCol + i)), acc);
      any = true;
    }
    if (any) atomicAdd(y + perm[s], acc);
  }
}

}  // namespace

cudaError_t launch_spmv_csr(int R, int Z, const int* rowPtrs, const int* colIdx,
                            const float* value, const int* tileRow, int nTiles, const float* x,
                            float* y, cudaStream_t s) {
  if (nTiles <= 0) return cudaSuccess;
  const bool vec = aligned16(colIdx) && aligned16(value);
  if (vec)
    k_spmv_csr<kCsrThreads, kCsrItemsPerThread, true>
        <<<nTiles, kCsrThreads, 0, s>>>(R, Z, rowPtrs, colIdx, value, tileRow, x, y);
  else
    k_spmv_csr<kCsrThreads, kCsrItemsPerThread, false>
        <<<nTiles, kCsrThreads, 0, s>>>(R, Z, rowPtrs, colIdx, value, tileRow, x, y);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_spmv_coo(int Z, const int* rowIdx, const int* colIdx, const float* value,
                            const float* x, float* y, bool dependent, cudaStream_t s) {
  if (Z <= 0) return cudaSuccess;
  const long long warps = ((long long)Z + 127) / 128;
  const long long blocks = (warps * 32 + 255) / 256;
  const bool vec = aligned16(rowIdx) && aligned16(colIdx) && aligned16(value);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  cudaError_t err;
  if (vec)
    err = cudaLaunchKernelEx(&cfg, k_spmv_coo<true>, Z, rowIdx, colIdx, value, x, y);
  else
    err = cudaLaunchKernelEx(&cfg, k_spmv_coo<false>, Z, rowIdx, colIdx, value, x, y);
  note_launches(1);
  return err;
}

cudaError_t launch_spmv_ell(int R, int K, const int* ellCol, const float* ellVal,
                            const float* x, float* y, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const bool vec4 = (R % 4 == 0) && aligned16(ellCol) && aligned16(ellVal) && aligned16(y);
  const long long threads = vec4 ? R / 4 : R;
  const long long blocks = (threads + 255) / 256;
  if (vec4)
    k_spmv_ell<true><<<(unsigned)blocks, 256, 0, s>>>(R, K, ellCol, ellVal, x, y);
  else
    k_spmv_ell<false><<<(unsigned)blocks, 256, 0, s>>>(R, K, ellCol, ellVal, x, y);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_spmv_jds(int R, int maxLen, int tSplit, int wTail, const int* iterPtr,
                            const int* perm, const int* jdsCol, const float* jdsVal,
                            const float* x, float* y, cudaStream_t s) {
  if (R <= 0 || maxLen <= 0) return cudaSuccess;
  const long long mainBlocks = ((long long)R + 255) / 256;
  long long tailBlocks = 0;
  int tailRowBlocks = 1;
  if (tSplit < maxLen && wTail > 0) {
    tailRowBlocks = (wTail + kJdsTailRows - 1) / kJdsTailRows;
    const long long diagBlocks = ((long long)(maxLen - tSplit) + kJdsTailDiags - 1) / kJdsTailDiags;
    tailBlocks = (long long)tailRowBlocks * diagBlocks;
  }
  k_spmv_jds<<<(unsigned)(mainBlocks + tailBlocks), 256, 0, s>>>(
      R, maxLen, tSplit, wTail, (int)mainBlocks, tailRowBlocks, iterPtr, perm, jdsCol, jdsVal, x,
      y);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace spmv
