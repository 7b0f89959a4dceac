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
// +0.0f; nnzPerRow[r] = min(len(r), K). A warp's load of the rows' t-th
// entries touches a sector per lane (the rows are one row length apart), and
// ncu shows the L1 pipeline as the bound on a 27-point stencil (lg_throttle
// stalls; L2-to-L1 reads 2.6 times the entries), while DRAM moves exactly
// the algorithmic bytes. Measured alternatives, all slower in the bench step
// (5-point Laplacian / 27-point stencil, against 60.4 / 334 us): a row's
// loads issued 8 at a time before its stores, 68.4 / 344 us; the block's CSR
// entries staged in shared memory with coalesced 16-byte loads, 128 rows per
// block, 117.8 / 350 us; each warp's entries staged in its own shared memory
// sized to the width, 89.1 / 359 us.
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

}  // namespace

// Threads per block (128 and 64 measured slower: CSR -> ELL on the 27-point
// stencil 325 / 338 / 332 us with 256 / 128 / 64 threads).
constexpr int kCsrToEllBlock = 256;

template <class T>
cudaError_t launch_csr_to_ell(int R, int K, const int* rowPtrs, const int* colIdx,
                              const T* value, int* ellCol, T* ellVal, int* nnzPerRow,
                              cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
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
