// internal.h -- declarations shared by the library's translation units.
// Not installed; the public ABI is include/spmv.h.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/spmv.h"

namespace spmv {

// ---------------------------------------------------------------------------
// Row statistics and validation results, written by the stats kernels.
// ---------------------------------------------------------------------------
constexpr int kExactLenBins = 1024;  // exact row-length histogram for len < 1024

enum : unsigned {
  kErrRowPtrStart = 1u,     // rowPtrs[0] != 0
  kErrRowPtrDecrease = 2u,  // rowPtrs[r+1] < rowPtrs[r]
  kErrRowPtrEnd = 4u,       // rowPtrs[numRows] != nnz
  kErrColRange = 8u,        // colIdx outside [0, numCols)
};

// Results of the statistics pass, accumulated by every block with atomics
// into a zeroed record (no fold at the end). Minima are kept as maxima of
// INT_MAX - v, so that 0 means "none".
struct DevStats {
  unsigned int err;      // kErrRowPtrStart | kErrRowPtrEnd (the others: stats_errors)
  int badRowKey;         // max over decreasing rows r of INT_MAX - r
  int badNnzKey;         // max over out-of-range positions k of INT_MAX - k
  int maxLen;
  int minLenKey;         // max over rows of INT_MAX - len
  int emptyRows;
  int maxWarpNnz;
  int pad0;
  unsigned long long sumSq;
  unsigned long long gatherLines;   // sampled: distinct 128-byte x lines per gather set
  unsigned long long gatherSets;    // sampled: number of 32-lane gather sets
  unsigned long long histLog2[33];  // rows with len >= kExactLenBins only
  unsigned int histExact[kExactLenBins];
};

// Every validation error bit of a finished record.
inline unsigned stats_errors(const DevStats& d) {
  return d.err | (d.badRowKey ? kErrRowPtrDecrease : 0u) | (d.badNnzKey ? kErrColRange : 0u);
}
// Shortest row (INT_MAX when there is no row).
inline int stats_min_len(const DevStats& d) { return 2147483647 - d.minLenKey; }

// Work area of the statistics pass: the DevStats record (read back by the
// host), a multiple of 256 bytes, zeroed before launch_stats.
size_t stats_work_bytes(int R, int Z, const int* colIdx);

// ---------------------------------------------------------------------------
// CSR work split: the nonzeros in chunks of kCsrChunk, each described by a
// 32-byte record built at handle creation.
// ---------------------------------------------------------------------------
constexpr int kCsrChunk = 128;
struct __align__(16) CsrChunkDesc {
  int lo;      // row holding the chunk's first nonzero
  int hi;      // row holding the next chunk's first nonzero (numRows-1 for the last)
  int flags;   // kCsrChunkHasEmptyRow: an empty row lies inside the chunk
  int pad0;
  uint4 mask;  // bit p: a row other than lo starts at position p of the chunk
};
constexpr int kCsrChunkHasEmptyRow = 1;
constexpr int kGatherSampleBlocks = 64;  // blocks of the column check that sample gathers

constexpr int kJdsSplitMinWidth = 8192;  // diagonals at least this wide run thread-per-row
constexpr int kJdsSplitMaxDiag = 1024;   // at most this many diagonals in the row-parallel part
constexpr int kJdsTailRows = 256;        // tail blocks: sorted rows per block
constexpr int kJdsTailDiags = 64;        // tail blocks: diagonals per block

// ---------------------------------------------------------------------------
// Launch accounting (every launcher reports its kernels).
// ---------------------------------------------------------------------------
void note_launches(int n);
int num_sms();
// A CUDA result as a library status: cudaSuccess -> SPMV_OK; otherwise the
// error is kept for spmv_last_cuda_error() on this thread and mapped to
// SPMV_ERR_ALLOC (out of memory) or SPMV_ERR_CUDA.
int record_cuda(cudaError_t e);

// ---------------------------------------------------------------------------
// Launchers. Each returns the cudaError_t of its launches.
// ---------------------------------------------------------------------------
// stats.cu: one launch; also writes the CSR chunk records into zeroed desc
cudaError_t launch_stats(int R, int C, int Z, const int* rowPtrs, const int* colIdx, void* work,
                         int nChunks, CsrChunkDesc* desc, cudaStream_t s);

// convert.cu
// CSR -> COO rowIdx from the CSR chunk records (spmv_kernels.cu)
cudaError_t launch_expand_rows(int R, int Z, const int* rowPtrs, const CsrChunkDesc* desc,
                               int* rowIdx, cudaStream_t s);
template <class T>
cudaError_t launch_csr_to_ell(int R, int K, const int* rowPtrs, const int* colIdx,
                              const T* value, int* ellCol, T* ellVal, int* nnzPerRow,
                              cudaStream_t s);
// Exclusive scan of max(0, len(r) - K) over rows into tailPtr[0..R].
cudaError_t launch_tail_scan(int R, int K, const int* rowPtrs, int* tailPtr, int* scratch,
                             cudaStream_t s);
size_t scan_scratch_ints(long long n);
template <class T>
cudaError_t launch_hyb_tail_copy(int R, int K, const int* rowPtrs, const int* colIdx,
                                 const T* value, const int* tailPtr, int* cooRow,
                                 int* cooCol, T* cooVal, cudaStream_t s);
// JDS: stable sort of rows by length (longest first), iterPtr, jagged scatter.
size_t jds_sort_scratch_bytes(int R, int maxLen);
// hostIterPtr: iterPtr computed on the host (nullptr: computed on the device);
// wLong: the number of rows longer than kJdsCoop (their entries past kJdsCoop
// are copied by extra warps)
constexpr int kJdsCoop = 64;
template <class T>
cudaError_t launch_jds_build(int R, int maxLen, int wLong, const int* rowPtrs,
                             const int* colIdx, const T* value, int* perm, int* iterPtr,
                             int* jdsCol, T* jdsVal, void* scratch, const int* hostIterPtr,
                             cudaStream_t s);
constexpr int kJdsPad = 8;  // extra elements after the JDS arrays (aligned vector reads)
// Sectioned ELL (the JDS variant): sort, section widths (for a read-back when
// the host cannot derive them), scatter; secPtr is int32 (slots < 2^31).
constexpr int kSellDefaultRows = 128;  // default section height
constexpr int kSellMainSlots = 64;     // slots per row done by the row-parallel part
constexpr int kSellTailSlots = 64;     // slots per row of one tail work item
// One tail work item of a section wider than kSellMainSlots: slots [t0, t1) of
// rows j0 .. j0 + 31 of section k (one row per lane).
struct SellItem {
  int k, t0, t1, j0;
};
size_t sell_scratch_bytes(int R, int maxLen, long long nsec);
// secPtr (nsec + 1 entries) by a device scan of the section sizes; the caller
// guarantees that the total fits in int32
cudaError_t launch_sell_offsets(int R, int S, int maxLen, long long nsec, const int* rowPtrs,
                                const int* perm, int* secPtr, void* scratch, cudaStream_t s);
cudaError_t launch_sell_sort(int R, int maxLen, const int* rowPtrs, int* perm, void* scratch,
                             cudaStream_t s);
cudaError_t launch_sell_widths(int R, int S, int nsec, const int* rowPtrs, const int* perm,
                               int* widths, cudaStream_t s);
// maxLen: the longest row (rows of kStageMinK to kStageMaxK entries are staged)
template <class T>
cudaError_t launch_sell_scatter(int R, int S, int maxLen, const int* rowPtrs, const int* colIdx,
                                const T* value, const void* scratch, const int* secPtr,
                                int slots, int* sellCol, T* sellVal, cudaStream_t s);

// spmv_kernels.cu
// fills hi, flags and mask of every chunk record; runs after the stats pass
cudaError_t launch_csr_chunk_masks(int R, int Z, const int* rowPtrs, int nChunks,
                                   CsrChunkDesc* desc, cudaStream_t s);
template <class T>
cudaError_t launch_spmv_csr(int R, int Z, const int* rowPtrs, const int* colIdx,
                            const T* value, const CsrChunkDesc* desc, const T* x,
                            T* y, cudaStream_t s);
template <class T>
cudaError_t launch_spmv_coo(int Z, const int* rowIdx, const int* colIdx, const T* value,
                            const T* x, T* y, bool dependent, cudaStream_t s);
template <class T>
cudaError_t launch_spmv_ell(int R, int K, const int* ellCol, const T* ellVal,
                            const T* x, T* y, cudaStream_t s);
// x-blocked list: nonzeros grouped by column chunk of B columns (CSR order in
// a chunk), 16-bit local columns, chunks padded to 4 entries (row -1).
constexpr int kXbSmemBytes = 196608;    // x staged per CTA: 192 KiB
constexpr int kXbDefaultChunk = 49152;  // columns per chunk with 4-byte values (24576 with 8)
constexpr int kXbMaxChunks = 65536;     // chunk ids sorted in at most two radix passes
// up to this many chunks the build sorts tiles of nonzeros by chunk in shared
// memory and decodes rows from the CSR chunk records (rowIdx unused;
// scattered: the columns are scattered, many chunks among 32 consecutive
// nonzeros); more chunks take a radix sort of all nonzeros and need rowIdx
constexpr int kXbTileChunks = 256;
size_t xb_scratch_bytes(int Z, int nch);
template <class T>
cudaError_t launch_xb_build(int Z, int B, int nch, const int* rowPtrs, const CsrChunkDesc* desc,
                            const int* colIdx, const T* value, const int* rowIdx, bool scattered,
                            int* chunkPtr, int* xbRow, unsigned short* xbCol, T* xbVal,
                            void* scratch, cudaStream_t s);
template <class T>
cudaError_t launch_spmv_xb(int C, int B, int nch, const int* chunkPtr, const int* xbRow,
                           const unsigned short* xbCol, const T* xbVal, const T* x,
                           T* y, cudaStream_t s);

// Conjugate gradient for A·X + Y = 0: device state shared by the kernels of
// one solve (zeroed before the first). status: kCgRunning until the stop test
// passes (kCgConverged) or d'Ad <= 0 (kCgBreakdown).
constexpr int kCgRunning = -1;
constexpr int kCgConverged = 0;
constexpr int kCgMaxIter = 1;
constexpr int kCgBreakdown = 2;
struct CgState {
  double gg;      // g'g of the current gradient
  double alpha, beta;
  double stop;    // tol * |Y|
  double gnorm;   // |g| after the last iteration
  double ynorm;   // |Y|
  int iter;       // iterations done
  int status;
  unsigned ticket;
  unsigned pad;
};
// per-block partial sums of the CG kernels (floats, in the work buffer)
size_t cg_partials_floats();
cudaError_t launch_cg_start(int R, const float* g, const float* Y, double tol, float* partials,
                            CgState* st, cudaStream_t s);
// generic format path: d = -g + beta d; (q = A d by spmv); d'q
cudaError_t launch_cg_direction(int R, const float* g, float* d, const CgState* st,
                                cudaStream_t s);
cudaError_t launch_cg_dot(int R, const float* d, const float* q, float* partials, CgState* st,
                          cudaStream_t s);
// ELL path: dNew = -g + beta dOld, q = A dNew, dNew'q in one kernel
cudaError_t launch_cg_ell_q(int R, int K, const int* ellCol, const float* ellVal, const float* g,
                            const float* dOld, float* dNew, float* q, float* partials,
                            CgState* st, cudaStream_t s);
cudaError_t launch_cg_update(int R, float* X, float* g, const float* d, const float* q,
                             float* partials, CgState* st, cudaStream_t s);

// items: tail work of the sections wider than kSellMainSlots (nItems of them)
template <class T>
cudaError_t launch_spmv_sell(int R, int S, int slots, const int* secPtr, const int* perm,
                             const int* sellCol, const T* sellVal, const SellItem* items,
                             int nItems, const T* x, T* y, cudaStream_t s);
// hostIterPtr: iterPtr[0 .. tSplit] on the host (or nullptr); with tSplit <=
// kJdsParamDiags the kernel takes them as a launch parameter
constexpr int kJdsParamDiags = 64;
template <class T>
cudaError_t launch_spmv_jds(int R, int maxLen, int tSplit, int wTail, const int* iterPtr,
                            const int* hostIterPtr, const int* perm, const int* jdsCol,
                            const T* jdsVal, const T* x, T* y, cudaStream_t s);

}  // namespace spmv
