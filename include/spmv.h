/*
 * spmv.h -- C ABI of the GB300 (sm_103a) sparse matrix-vector library.
 *
 * Operation (PMPP notes, "Sparse Matrices and Basic Formats (COO and CSR)",
 * section "Background & SpMV"): sparse matrix-vector multiplication AND
 * ACCUMULATION, y <- A*x + y, with A sparse and x, y dense fp32 vectors.
 *
 * The matrix enters in CSR form (same page, section "CSR format and SpMV":
 * rowPtrs[numRows+1] with rowPtrs[0] = 0 and rowPtrs[numRows] = nnz, colIdx
 * and value grouped by row; columns inside a row need not be sorted). The
 * library converts it ON THE DEVICE into the pages' other storage formats
 * and runs a hand-written kernel per format:
 *   COO  -- "Sparse Matrices and Basic Formats (COO and CSR)", section
 *           "COO format and SpMV": value/colIdx/rowIdx per nonzero.
 *   ELL  -- "Regularized Formats (ELL, Hybrid ELL-COO and JDS)", section
 *           "ELL format: padding + transposition": rows padded to the longest
 *           row, stored column-major, slot i = t*numRows + row.
 *   HYB  -- same page, section "Hybrid ELL-COO format": an ELL part of width
 *           K plus a COO part holding each row's entries beyond K.
 *   JDS  -- same page, section "JDS format": rows sorted by length (longest
 *           first, stable), a row permutation, and jagged diagonals starting
 *           at iterPtr[t].
 *   SELL -- same page, same section, the variant it describes: the sorted
 *           rows cut into sections of S rows, each section an ELL padded to
 *           its own longest row (sectioned / sliced ELL).
 *   XBLOCK -- "Introduction to sparse computing and performance bottleneck
 *           location", section "Building the problem framework": x split
 *           into chunks of B columns, the nonzeros grouped by the chunk their
 *           column falls in, so that one thread block gathers from one chunk.
 *
 * Conventions for every function:
 *   - Every function returns an int status (spmv_status); nothing throws or
 *     aborts across this ABI. spmv_status_string() names a status.
 *   - "device pointer" means memory of the CURRENT CUDA device, allocated by
 *     the caller (cudaMalloc, a torch tensor, ...). Handles are bound to the
 *     device current at spmv_create_csr and must be used with it current.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued on it asynchronously unless stated.
 *   - Index type is int32 (signed; negatives are rejected), values are fp32.
 *   - Ownership: the caller owns the CSR arrays, x and y. The handle BORROWS
 *     the CSR arrays (it reads them again in spmv_run(SPMV_CSR) and the
 *     COO format reuses colIdx/value), so they must stay alive and unchanged
 *     until spmv_destroy. The handle OWNS every converted array; they are
 *     allocated from a library-private stream-ordered pool on the stream of
 *     the call that creates them and released by spmv_destroy.
 *   - Thread safety: distinct handles may be used from distinct threads; one
 *     handle must not be used by two threads at once.
 */
#ifndef SPMV_GB300_H
#define SPMV_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spmv_handle_s *spmv_handle; /* opaque */

typedef enum {
  SPMV_COO = 0,
  SPMV_CSR = 1,
  SPMV_ELL = 2,
  SPMV_HYB = 3,
  SPMV_JDS = 4,
  SPMV_AUTO = 5, /* spmv_run: the format spmv_select would choose */
  SPMV_SELL = 6,  /* sectioned ELL over the JDS row order */
  SPMV_XBLOCK = 7 /* nonzeros grouped by column chunk of x */
} spmv_format;

typedef enum {
  SPMV_OK = 0,
  SPMV_ERR_INVALID_ARG = -1,      /* null/negative/inconsistent argument */
  SPMV_ERR_BAD_ROWPTRS = -2,      /* rowPtrs[0] != 0, decreasing, or rowPtrs[numRows] != nnz */
  SPMV_ERR_COL_OUT_OF_RANGE = -3, /* some colIdx < 0 or >= numCols */
  SPMV_ERR_TOO_LARGE = -4,        /* ELL/HYB/SELL slot count beyond int32 or the padding budget */
  SPMV_ERR_NOT_CONVERTED = -5,    /* spmv_run/export of a format not converted yet */
  SPMV_ERR_CUDA = -6,             /* a CUDA runtime call failed (see spmv_last_cuda_error) */
  SPMV_ERR_ALLOC = -7,            /* device allocation failed or exceeded the set limit */
  SPMV_ERR_TIMEOUT = -8           /* reserved (no kernel of this library waits on another) */
} spmv_status;

/* Row-length statistics computed on the device by spmv_create_csr
 * ("[CUDA performance tuning] SpMV storage format selection and performance
 * comparison", section 4.1: nonzero distribution histogram and row-length
 * variance; "Introduction to sparse computing and performance bottleneck
 * location", section "Building the problem framework": max/mean load ratio). */
typedef struct {
  int64_t num_rows, num_cols, nnz;
  int64_t max_len;          /* longest row */
  int64_t min_len;          /* shortest row (0 if numRows == 0) */
  int64_t empty_rows;       /* rows with no entry */
  int64_t sum_sq_len;       /* sum over rows of len^2 (exact) */
  double mean_len;          /* nnz / numRows */
  double var_len;           /* population variance of the row lengths */
  int64_t hist_log2[33];    /* bin 0: len 0; bin b >= 1: len in [2^(b-1), 2^b) */
  double imbalance_thread;  /* max_len / mean_len: one row per thread */
  double imbalance_warp;    /* max over groups of 32 consecutive rows of their nnz,
                               divided by the mean group nnz: one group per warp */
  int32_t auto_format;      /* spmv_format chosen by spmv_select */
  int32_t auto_hyb_width;   /* HYB width used when spmv_convert_hyb gets 0 */
  double gather_lines;      /* x locality, sampled: distinct 128-byte lines of x touched
                               by 32 gathers of consecutive nonzeros (1 = all in one line,
                               32 = all in different lines); 0 when not sampled */
} spmv_stats;

/* Read-only view of one converted format (device pointers owned by the
 * handle, valid until spmv_destroy or until the format is converted again).
 * Unused fields are NULL / 0. */
typedef struct {
  int32_t format;           /* spmv_format */
  int64_t num_rows, num_cols, nnz;
  int32_t width;            /* ELL and HYB: K (slots per row); JDS: longest row;
                               SELL: width of the widest (first) section */
  int64_t ell_slots;        /* ELL/HYB: num_rows * width; SELL, XBLOCK: total slots */
  int64_t coo_nnz;          /* COO: nnz; HYB: entries of the COO part */
  const int32_t *row_ptrs;  /* CSR: numRows + 1 (the caller's array) */
  const int32_t *row_idx;   /* COO: nnz;  HYB: coo_nnz;  XBLOCK: ell_slots (padding = -1) */
  const int32_t *col_idx;   /* CSR/COO: nnz; ELL/HYB/SELL: ell_slots (padding = -1); JDS: nnz */
  const float *value;       /* as col_idx (padding = +0.0f) */
  const int32_t *nnz_per_row;  /* ELL/HYB: entries of each row held in the ELL slots */
  const int32_t *coo_col_idx;  /* HYB: coo_nnz */
  const float *coo_value;      /* HYB: coo_nnz */
  const int32_t *perm;      /* JDS/SELL: perm[s] = original row of sorted row s (numRows) */
  const int32_t *iter_ptr;  /* JDS: width + 1 entries, iter_ptr[width] = nnz */
  const int32_t *sec_ptr;   /* SELL: ceil(numRows/S) + 1 entries, first slot of each
                               section, sec_ptr[last] = ell_slots */
  int32_t section_rows;     /* SELL: S, rows per section (the last may be shorter) */
  const int32_t *chunk_ptr; /* XBLOCK: num_chunks + 1 entries, first slot of each chunk
                               (multiples of 4); chunk_ptr[num_chunks] = ell_slots */
  const uint16_t *col16;    /* XBLOCK: ell_slots local columns (column - chunk * chunk_cols) */
  int32_t chunk_cols;       /* XBLOCK: B, columns per chunk */
  int32_t num_chunks;       /* XBLOCK: ceil(numCols / B) */
  int32_t value_bytes;      /* 4 (handle from spmv_create_csr) or 8 (spmv_create_csr_f64) */
  const double *value_f64;     /* 8-byte handles: the value array (value is then NULL) */
  const double *coo_value_f64; /* 8-byte handles: HYB's COO values (coo_value is then NULL) */
} spmv_arrays;

/* Create a handle over a CSR matrix that lives on the current device.
 *   numRows, numCols >= 0; nnz >= 0; d_rowPtrs: numRows+1 ints; d_colIdx and
 *   d_value: nnz entries (may be NULL when nnz == 0).
 * Validates the input on the device by the sanity rules of "Sparse matrix
 * multiplication acceleration techniques", section 5.3 (rowPtrs monotone,
 * every column below numCols, nnz consistent with rowPtrs[numRows]),
 * computes the row statistics and the nnz-balanced CSR partition, then
 * SYNCHRONISES `stream` once to read the result. On any error *out is set to
 * NULL and nothing stays allocated. Returns SPMV_ERR_BAD_ROWPTRS before
 * SPMV_ERR_COL_OUT_OF_RANGE when both apply. */
int spmv_create_csr(spmv_handle *out, int32_t numRows, int32_t numCols, int32_t nnz,
                    const int32_t *d_rowPtrs, const int32_t *d_colIdx,
                    const float *d_value, void *stream);

/* As spmv_create_csr with 8-byte values ("Introduction to sparse computing
 * and performance bottleneck location", section "Building the problem
 * framework": a value and an x entry take 4 or 8 bytes). Every conversion
 * keeps the values in 8 bytes; the handle is run with spmv_run_f64 on
 * double x and y (spmv_run and spmv_cg_solve answer SPMV_ERR_INVALID_ARG).
 * XBLOCK chunks hold at most 24576 columns (chunkCols 0 picks 24576). */
int spmv_create_csr_f64(spmv_handle *out, int32_t numRows, int32_t numCols, int32_t nnz,
                        const int32_t *d_rowPtrs, const int32_t *d_colIdx,
                        const double *d_value, void *stream);

/* CSR -> COO ("COO format and SpMV"): expands rowPtrs into rowIdx[nnz]
 * (rowIdx[k] = r for rowPtrs[r] <= k < rowPtrs[r+1]). colIdx and value are
 * unchanged, so the COO view shares the caller's two arrays. Asynchronous. */
int spmv_convert_coo(spmv_handle h, void *stream);

/* CSR -> ELL ("ELL format: padding + transposition"): K = longest row;
 * slot t*numRows + r holds the t-th entry of row r, or value +0.0f and
 * column -1 when row r has fewer than t+1 entries; nnzPerRow[r] = len(r).
 * Returns SPMV_ERR_TOO_LARGE (nothing allocated) when numRows*K exceeds
 * INT32_MAX or the padding budget numRows*K <= 4*nnz + numRows. Async. */
int spmv_convert_ell(spmv_handle h, void *stream);

/* CSR -> HYB ("Hybrid ELL-COO format"): an ELL part of width K with the first
 * min(len, K) entries of each row, and a COO part with every row's remaining
 * entries in row order, then in-row order. ellWidth = 0 picks K as the
 * smallest L such that 99% of the rows have length <= L; ellWidth > 0 is used
 * as given (capped at the longest row). Same size limits as ELL.
 * Asynchronous when K < 1024: the COO part's size then follows from the
 * exact row-length histogram taken by spmv_create_csr. With K >= 1024 the
 * size is computed on the device and read back, which SYNCHRONISES `stream`
 * once. */
int spmv_convert_hyb(spmv_handle h, int32_t ellWidth, void *stream);

/* CSR -> JDS ("JDS format", steps 1-4): perm sorts the rows by length,
 * longest first, equal lengths in original order; iterPtr[t] is where
 * jagged diagonal t starts (iterPtr[maxLen] = nnz); entry iterPtr[t] + s is
 * the t-th entry of sorted row s. Asynchronous. */
int spmv_convert_jds(spmv_handle h, void *stream);

/* CSR -> SELL, the sectioned variant of JDS ("Regularized Formats (ELL,
 * Hybrid ELL-COO and JDS)", section "JDS format", last paragraph): rows
 * sorted as for JDS (perm), sorted row s in section k = s / S; a section
 * holds h_k = min(S, numRows - k*S) rows and is padded to w_k, the length of
 * its first (longest) row; slot t of the j-th row of section k is at
 * sec_ptr[k] + t*h_k + j (column-major inside the section), padding as ELL
 * (column -1, value +0.0f). sectionRows = 0 picks S = 128; sectionRows < 0 is
 * SPMV_ERR_INVALID_ARG. Returns SPMV_ERR_TOO_LARGE (nothing kept) when the
 * slot count exceeds INT32_MAX or 4*nnz + numRows. Asynchronous when every
 * row has fewer than 1024 entries (the section widths then follow from the
 * exact row-length histogram). Otherwise the widths are computed on the
 * device after the sort and read back, which SYNCHRONISES `stream` once. */
int spmv_convert_sell(spmv_handle h, int32_t sectionRows, void *stream);

/* CSR -> XBLOCK ("Introduction to sparse computing and performance bottleneck
 * location", section "Building the problem framework": split x into chunks
 * and let a thread block process only the nonzeros whose columns fall in one
 * chunk, localising the random gather). Chunk c covers columns
 * [c*B, min(numCols, (c+1)*B)); its entries are the nonzeros with a column
 * there, in CSR order (by row, then position in the row), from chunk_ptr[c]:
 * row_idx (int32), col16 = column - c*B (uint16), value; each chunk padded
 * to a multiple of 4 entries with row -1, col16 0, value +0.0f.
 *   chunkCols: B in [1, 49152] (the SpMV stages B floats of x in 192 KiB of
 *   shared memory; [1, 24576] for 8-byte values), 0 picks the largest;
 *   else SPMV_ERR_INVALID_ARG. More than 65536
 *   chunks, or nnz + 3*chunks above INT32_MAX: SPMV_ERR_TOO_LARGE.
 *   Asynchronous. The slot count stays on the device; spmv_export of XBLOCK
 *   reads it (one synchronisation, the first time). */
int spmv_convert_xblock(spmv_handle h, int32_t chunkCols, void *stream);

/* y <- A*x + y with the given format (SPMV_AUTO = spmv_select's choice).
 * d_x: numCols floats, d_y: numRows floats, both on the handle's device;
 * x and y must not overlap (SPMV_ERR_INVALID_ARG). The format must have been
 * converted (SPMV_CSR always is), else SPMV_ERR_NOT_CONVERTED; nothing is
 * converted implicitly. Allocates nothing and never synchronises, so it can
 * be captured into a CUDA graph (after one call outside capture for each
 * format on each device, which sets kernel attributes once) and replayed.
 * Asynchronous on `stream`; launches 1 kernel
 * (CSR, COO, ELL, JDS, SELL, XBLOCK) or 2 (HYB: ELL part, then the COO part with a
 * programmatic dependent launch). Floating-point rounding differs from a
 * sequential sum (tree and atomic reductions); per row the result is within
 * 1e-5 * (sum_j |a_ij x_j| + |y_i|) of the exact value for rows up to
 * several thousand entries. */
int spmv_run(spmv_handle h, spmv_format format, const float *d_x, float *d_y, void *stream);

/* y <- A*x + y for a handle made by spmv_create_csr_f64: double x (numCols)
 * and y (numRows), every product and sum in fp64; otherwise as spmv_run
 * (SPMV_ERR_INVALID_ARG for a 4-byte handle). Per row the result is within
 * (len + 2) * 2^-52 * (sum_j |a_ij x_j| + |y_i|) of the exact value. */
int spmv_run_f64(spmv_handle h, spmv_format format, const double *d_x, double *d_y,
                 void *stream);

/* Result of spmv_cg_solve. */
typedef struct {
  int32_t iterations;     /* iterations done */
  int32_t status;         /* 0: |A·X + Y| <= tol*|Y| reached; 1: maxIter iterations done first;
                             2: stopped because d'Ad <= 0 (A is not positive definite) */
  double residual_norm;   /* |g| = |A·X + Y| after the last iteration (recurrence value) */
  double y_norm;          /* |Y| */
} spmv_cg_info;

/* Solve A·X + Y = 0 for X by conjugate gradients ("Sparse Matrices and
 * Basic Formats (COO and CSR)", section "Background & SpMV": the iterative
 * method for positive-definite A that guesses X, forms A·X + Y -- this
 * library's SpMV -- and corrects X along the gradient). Textbook CG
 * (Hestenes-Stiefel) in gradient form: g = A·X + Y, d = -g; per iteration
 * q = A d, alpha = g'g/d'q, X += alpha d, g += alpha q, stop when
 * |g| <= tol*|Y|, beta = g'g(new)/g'g(old), d = -g + beta d.
 *   A must be square (numRows == numCols) and symmetric positive definite
 *   (symmetry is not checked; a non-positive curvature stops with status 2).
 *   format: any converted format or SPMV_AUTO; SPMV_ELL runs a fused
 *   q = A d + d'q kernel, the others their spmv_run kernel plus a dot.
 *   d_y: numRows floats (Y, read only); d_x: numRows floats, the starting
 *   guess on entry and the solution on return; x and y must not overlap.
 *   maxIter >= 0, tol >= 0 (tol = 0: run maxIter iterations unless g
 *   becomes exactly 0). fp32 vectors; inner products summed in fp32 within
 *   a block and fp64 across blocks.
 *   Allocates 3*numRows floats of work from the library pool for the call.
 *   SYNCHRONISES `stream`: after 1, 2, 4, ..., 64 iterations, then every
 *   64, and at the end, to read the device's stop decision into *info.
 * Returns SPMV_ERR_NOT_CONVERTED for a format not converted yet. */
int spmv_cg_solve(spmv_handle h, spmv_format format, const float *d_y, float *d_x,
                  int32_t maxIter, double tol, spmv_cg_info *info, void *stream);

/* Format choice from the statistics of spmv_create_csr ("[CUDA performance
 * tuning] SpMV storage format selection and performance comparison", section
 * 4.3; its comparison operators are lost in the page, the reading is):
 * longest <= 2*mean -> ELL; else mean < 10 -> COO; else HYB when
 * longest > 5*mean, otherwise CSR. Two rules of this library come around it:
 * compulsory SpMV bytes (8 per nonzero + 12 per row + 4 per column) below
 * 4 MiB -> CSR, checked first (a matrix that small is bound by memory round
 * trips, not bandwidth); and in the HYB case, scattered columns
 * (stats.gather_lines >= 16) -> XBLOCK, the x-blocked list. The chosen format
 * must be converted before spmv_run(SPMV_AUTO). *ellWidth gets the automatic
 * HYB width. Host-only; either output pointer may be NULL. */
int spmv_select(spmv_handle h, spmv_format *format, int32_t *ellWidth);

/* Format choice by timing ("[CUDA performance tuning] SpMV storage format
 * selection and performance comparison", end of section 4.3: run every
 * format on the matrix and keep the fastest). Runs y <- A*x + y in every
 * format converted so far (CSR always; COO, ELL, HYB, JDS, SELL, XBLOCK
 * when converted): one untimed run, then `reps` runs each timed with CUDA
 * events on `stream` (back to back, L2 as the previous run left it), and
 * takes each format's median.
 *   d_x: numCols floats; d_y: numRows floats of SCRATCH, overwritten (it
 *   accumulates every run). reps in [1, 1000]. 4-byte handles only
 *   (SPMV_ERR_INVALID_ARG for a handle from spmv_create_csr_f64).
 *   *best: the fastest format. From then on spmv_select, spmv_get_stats'
 *   auto_format and spmv_run(SPMV_AUTO) use it (it is converted by
 *   construction). times_ms (optional, NULL allowed): 8 floats indexed by
 *   spmv_format, the median ms of each timed format, -1 for formats not
 *   timed (not converted, and SPMV_AUTO).
 *   SYNCHRONISES `stream` after every timed run. */
int spmv_autotune(spmv_handle h, const float *d_x, float *d_y, int32_t reps,
                  spmv_format *best, float *times_ms, void *stream);

/* Copy the statistics computed at creation into *out (host). */
int spmv_get_stats(spmv_handle h, spmv_stats *out);

/* Describe the device arrays of a converted format (SPMV_NOT_CONVERTED if
 * absent). The pointers are read-only views owned by the handle. */
int spmv_export(spmv_handle h, spmv_format format, spmv_arrays *out);

/* Release every array the handle owns, in stream order on the stream of the
 * handle's most recent call, and free the handle. Work on other streams that
 * uses the handle must be complete. NULL is accepted. */
int spmv_destroy(spmv_handle h);

/* y <- A*x + y straight from CSR arrays, with no handle and no allocation.
 * (The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory -- processes whose device memory is fully
 * reserved by another allocator or pool, real-time loops that forbid
 * allocation and the synchronisation it may bring.)
 *   Arguments as spmv_create_csr plus d_x (numCols floats) and d_y (numRows
 *   floats); all device pointers on the current device, x and y not
 *   overlapping. The CSR input is NOT validated: pass arrays that
 *   spmv_create_csr would accept.
 *   Scratch: the per-chunk row index lives in a fixed array of device global
 *   memory reserved by the library (1 MiB on every GPU that loads it, held
 *   until the process exits), so nnz is limited to 4,194,304 (32768 chunks of
 *   128); a larger nnz returns SPMV_ERR_TOO_LARGE and does nothing.
 *   Set-up: the first call with nnz > 0 on a device (with that device
 *   current) looks up the array's device address. That is also when the
 *   array and the kernels this call launches take their device memory (CUDA
 *   loads a module on its first use), so a caller whose other allocator
 *   reserves the device should make one such call at start-up, before that
 *   reservation (any small valid matrix will do), and before any stream
 *   capture. Later calls neither allocate nor free memory. A CUDA failure
 *   returns SPMV_ERR_CUDA (SPMV_ERR_ALLOC when it is an out-of-memory error),
 *   with the cudaError_t in spmv_last_cuda_error().
 *   Concurrency: every call reuses the same array, so calls that overlap on
 *   the GPU (different streams, no ordering between them) race and give
 *   wrong results; calls ordered on one stream are fine.
 *   Asynchronous on `stream`; launches 3 kernels. */
int spmv_run_csr_noalloc(int32_t numRows, int32_t numCols, int32_t nnz,
                         const int32_t *d_rowPtrs, const int32_t *d_colIdx,
                         const float *d_value, const float *d_x, float *d_y, void *stream);

/* Static English text for a status code. */
const char *spmv_status_string(int status);

/* The last cudaError_t the library saw on this thread (0 if none). */
int spmv_last_cuda_error(void);

/* Number of kernels this process has launched through the library. */
uint64_t spmv_launch_count(void);

/* Cap (bytes) on device memory the library may hold in total; a request
 * beyond it fails with SPMV_ERR_ALLOC. A negative value removes the cap. */
int spmv_set_memory_limit(int64_t bytes);

/* Library version, major*10000 + minor*100 + patch. */
int spmv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPMV_GB300_H */
