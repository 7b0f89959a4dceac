// noalloc.cu -- a one-shot CSR SpMV that allocates nothing.
//
// Some callers cannot call cudaMalloc: processes whose device memory is
// fully reserved by another allocator or a fixed pool, and real-time loops
// whose rules forbid allocation (and the device synchronisation that
// cudaMalloc and cudaFree may bring) after start-up. spmv_run_csr_noalloc serves them: it runs
// y <- A*x + y from the caller's CSR arrays without a handle, keeping the
// per-chunk row index the CSR kernel needs in a fixed array in device global
// memory that the library reserves for the life of the process.
#include <mutex>

#include "device_util.cuh"
#include "internal.h"

namespace spmv {
namespace {

// Shared scratch: one record per kCsrChunk nonzeros, at most
// kNoAllocMaxChunks of them (1 MiB per GPU that loads the library). Every
// call overwrites what it uses; calls that overlap on the GPU race on it.
// Under CUDA's lazy module loading the array (and the kernels) take their
// device memory when this module is first loaded on a device, i.e. at the
// first call with nnz > 0 there (cudaGetSymbolAddress below), not when the
// library is loaded.
constexpr int kNoAllocMaxChunks = 32768;  // nnz <= 4,194,304
static __device__ __align__(256) CsrChunkDesc g_noallocDesc[kNoAllocMaxChunks];

constexpr int kMaxDevices = 64;
std::mutex g_setupMu;
CsrChunkDesc* g_descPtr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the host-side symbol is a stand-in, not a device address).
cudaError_t scratch_for_device(int dev, CsrChunkDesc** desc) {
  std::lock_guard<std::mutex> lk(g_setupMu);
  if (!g_descPtr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noallocDesc);
    if (e != cudaSuccess) return e;
    g_descPtr[dev] = static_cast<CsrChunkDesc*>(p);
  }
  *desc = g_descPtr[dev];
  return cudaSuccess;
}

// desc[c].lo = the row holding nonzero c*kCsrChunk: a row writes the records
// of the chunks that start inside it (bounds-checked).
__global__ void k_noalloc_chunk_lo(int R, int Z, const int* __restrict__ rowPtrs, int nChunks,
                                   CsrChunkDesc* __restrict__ desc) {
  const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int a = rowPtrs[r];
  const int b = rowPtrs[r + 1];
  if (a < 0 || b > Z || b <= a) return;
  const int c0 = (a + kCsrChunk - 1) / kCsrChunk;
  const int c1 = min((b - 1) / kCsrChunk, nChunks - 1);
  for (int c = c0; c <= c1; ++c) desc[c].lo = (int)r;
}

}  // namespace
}  // namespace spmv

extern "C" int spmv_run_csr_noalloc(int32_t numRows, int32_t numCols, int32_t nnz,
                                    const int32_t* d_rowPtrs, const int32_t* d_colIdx,
                                    const float* d_value, const float* d_x, float* d_y,
                                    void* stream) {
  using namespace spmv;
  if (numRows < 0 || numCols < 0 || nnz < 0) return SPMV_ERR_INVALID_ARG;
  if (numRows > 0 && (!d_rowPtrs || !d_y)) return SPMV_ERR_INVALID_ARG;
  if (nnz > 0 && (!d_colIdx || !d_value || !d_x)) return SPMV_ERR_INVALID_ARG;
  const long long nChunks = ((long long)nnz + kCsrChunk - 1) / kCsrChunk;
  if (nChunks > kNoAllocMaxChunks) return SPMV_ERR_TOO_LARGE;
  if (numRows == 0 || nnz == 0) return SPMV_OK;
  // every CUDA failure goes through record_cuda, so that spmv_last_cuda_error()
  // names it
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return SPMV_ERR_INVALID_ARG;
  CsrChunkDesc* desc = nullptr;
  e = scratch_for_device(dev, &desc);
  if (e != cudaSuccess) return record_cuda(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_noalloc_chunk_lo<<<(unsigned)(((long long)numRows + 255) / 256), 256, 0, s>>>(
      numRows, nnz, d_rowPtrs, (int)nChunks, desc);
  note_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda(e);
  e = launch_csr_chunk_masks(numRows, nnz, d_rowPtrs, (int)nChunks, desc, s);
  if (e != cudaSuccess) return record_cuda(e);
  return record_cuda(
      launch_spmv_csr(numRows, nnz, d_rowPtrs, d_colIdx, d_value, desc, d_x, d_y, s));
}
