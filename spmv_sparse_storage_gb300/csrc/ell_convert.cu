// ell_convert.cu -- CSR -> ELL ("Regularized Formats (ELL, Hybrid ELL-COO and
// JDS)", section "ELL format: padding + transposition"): every row padded to
// the width K and stored column-major, slot t*numRows + row. Also builds the
// ELL part of HYB (section "Hybrid ELL-COO format": the first K entries of
// each row; the rest goes to the COO part, convert.cu).
#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

// Thread per row, writes coalesced across rows (slot t of consecutive rows
// is one store per warp for every t). Padding slots get column -1 and value
// +0.0f; nnzPerRow[r] = min(len(r), K). This direct form reads a row's t-th
// entry straight from global memory: a warp's load then touches a sector per
// lane (the rows are one row length apart), and ncu shows the L1 pipeline as
// the bound on a 27-point stencil (lg_throttle stalls; L2-to-L1 reads 2.6
// times the entries). It serves widths outside [kStageMinK, kStageMaxK];
// k_csr_to_ell_staged serves the rest.
template <class T>
__global__ void __launch_bounds__(256) k_csr_to_ell(int R, int K, const int* __restrict__ rowPtrs,
                                                    const int* __restrict__ colIdx,
                                                    const T* __restrict__ value,
                                                    int* __restrict__ ellCol,
                                                    T* __restrict__ ellVal,
                                                    int* __restrict__ nnzPerRow) {
  const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int a = rowPtrs[r];
  const int len = rowPtrs[r + 1] - a;
  const int kept = len < K ? len : K;
  nnzPerRow[r] = kept;
  for (int t = 0; t < K; ++t) {
    const size_t i = (size_t)t * (size_t)R + (size_t)r;
    int c = -1;
    T v = T(0);
    if (t < kept) {
      c = colIdx[a + t];
      v = value[a + t];
    }
    __stcs(ellCol + i, c);
    __stcs(ellVal + i, v);
  }
}

// Warp-staged form for widths in [kStageMinK, kStageMaxK]: a warp's 32 consecutive rows
// hold at most 32 * K entries, contiguous in CSR. The warp copies them into
// its own part of shared memory (warp_stage_entries: asynchronous 16-byte
// copies, all in flight before one wait), then each lane writes its row's K
// slots from there (one coalesced store per warp for every t). ncu on a
// 27-point stencil: 267 us against 333 for the direct form, DRAM at 82 % with
// exactly the algorithmic bytes, no lg_throttle stalls (the 16-byte copies
// bypass L1, so L2 serves each 32-byte sector as two requests).
// Measured alternatives, slower than the direct form in the bench step
// (5-point Laplacian / 27-point stencil, against 60.4 / 334 us): staging
// with plain loads, whose stores to shared memory waited on each load in
// turn, 89.1 / 359 us (the same with 128 rows per block and a block barrier,
// 117.8 / 350 us); a row's loads issued 8 at a time before its stores, 68.4 /
// 344 us. A warp whose rows hold more than 32 * K entries (rows longer than a
// HYB part's K) reads directly. Shared memory per warp: 32 * K + 8 entries,
// sized by the launch.
template <class T, bool VEC>
__global__ void __launch_bounds__(32 * kStageWarps) k_csr_to_ell_staged(
    int R, int K, const int* __restrict__ rowPtrs, const int* __restrict__ colIdx,
    const T* __restrict__ value, int* __restrict__ ellCol, T* __restrict__ ellVal,
    int* __restrict__ nnzPerRow) {
  extern __shared__ int4 sRaw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = 32 * K + 8;  // a multiple of 4: every warp's buffers start 16-byte aligned
  int* sCol = reinterpret_cast<int*>(sRaw) + warp * cap;
  T* sVal = reinterpret_cast<T*>(reinterpret_cast<int*>(sRaw) + kStageWarps * cap) + warp * cap;
  const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long w0 = r - lane;  // the warp's first row
  if (w0 >= R) return;            // warp-uniform
  const long long wEnd = w0 + 32 < R ? w0 + 32 : R;
  const int a0 = __ldg(rowPtrs + w0);
  const int a1 = __ldg(rowPtrs + wEnd);
  int a = 0, len = 0;
  if (r < R) {
    a = __ldg(rowPtrs + r);
    len = __ldg(rowPtrs + r + 1) - a;
  }
  const int kept = len < K ? len : K;
  if (r < R) nnzPerRow[r] = kept;
  const bool staged = (long long)a1 - a0 <= 32LL * K;  // warp-uniform
  if (staged) warp_stage_entries<T, VEC>(colIdx, value, a0, a1, lane, sCol, sVal);
  __syncwarp();
  if (r >= R) return;
  const int off = (int)(a - (a0 & ~3LL));
  for (int t = 0; t < K; ++t) {
    const size_t i = (size_t)t * (size_t)R + (size_t)r;
    int c = -1;
    T v = T(0);
    if (t < kept) {
      c = staged ? sCol[off + t] : colIdx[a + t];
      v = staged ? sVal[off + t] : value[a + t];
    }
    __stcs(ellCol + i, c);
    __stcs(ellVal + i, v);
  }
}

}  // namespace

// Threads per block of the direct form (128 and 64 measured slower: CSR ->
// ELL on the 27-point stencil 325 / 338 / 332 us with 256 / 128 / 64 threads).
constexpr int kCsrToEllBlock = 256;

template <class T>
cudaError_t launch_csr_to_ell(int R, int K, const int* rowPtrs, const int* colIdx,
                              const T* value, int* ellCol, T* ellVal, int* nnzPerRow,
                              cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  if (K >= kStageMinK && K <= kStageMaxK<T>) {
    constexpr int threads = 32 * kStageWarps;
    const unsigned blocks = (unsigned)(((long long)R + threads - 1) / threads);
    const size_t smem = warp_stage_smem<T>(K);
    if (aligned16(colIdx) && aligned16(value))
      k_csr_to_ell_staged<T, true><<<blocks, threads, smem, s>>>(R, K, rowPtrs, colIdx, value,
                                                                 ellCol, ellVal, nnzPerRow);
    else
      k_csr_to_ell_staged<T, false><<<blocks, threads, smem, s>>>(R, K, rowPtrs, colIdx, value,
                                                                  ellCol, ellVal, nnzPerRow);
    note_launches(1);
    return cudaGetLastError();
  }
  const unsigned blocks = (unsigned)(((long long)R + kCsrToEllBlock - 1) / kCsrToEllBlock);
  k_csr_to_ell<T><<<blocks, kCsrToEllBlock, 0, s>>>(R, K, rowPtrs, colIdx, value, ellCol, ellVal,
                                                    nnzPerRow);
  note_launches(1);
  return cudaGetLastError();
}

template cudaError_t launch_csr_to_ell<float>(int, int, const int*, const int*, const float*, int*,
                                              float*, int*, cudaStream_t);
template cudaError_t launch_csr_to_ell<double>(int, int, const int*, const int*, const double*,
                                               int*, double*, int*, cudaStream_t);

}  // namespace spmv
