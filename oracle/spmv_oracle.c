/*
 * spmv_oracle.c -- plain, slow, single-threaded CPU oracle for sparse
 * matrix-vector multiply-and-accumulate y = A*x + y and for the storage
 * formats COO, CSR, ELL, hybrid ELL+COO and JDS.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the bench's CPU
 * baseline do. It shares no code, header, table or helper with the CUDA path.
 *
 * Also: the conjugate-gradient loop that the first page names as the main
 * user of the SpMV (or_cg_csr, at the end of this file).
 *
 * Sources (web pages, cited by title and section):
 *   [P1] PMPP notes, "Sparse Matrices and Basic Formats (COO and CSR)":
 *        "Background & SpMV", Fig. 14.1, "COO format and SpMV",
 *        "CSR format and SpMV".
 *   [P2] PMPP notes, "Regularized Formats (ELL, Hybrid ELL-COO and JDS)":
 *        "ELL format: padding + transposition", "Hybrid ELL-COO format",
 *        "JDS format", "Summary: data-dependent performance and OP/B".
 *   [P3] "[CUDA performance tuning] SpMV storage format selection and
 *        performance comparison": section 4.1 (matrix feature analysis),
 *        section 4.3 (automatic format selection).
 *   [P5] "Sparse matrix multiplication acceleration techniques", section 5.3
 *        (common problems: input sanity checks).
 *
 * Readings where the pages are open (each is also listed in the design notes):
 *   - SpMV accumulates: y_i <- y_i + sum_k a_k x_col(k)   ([P1] Background).
 *   - ELL padding slot: value +0.0f ([P2] ELL step 1 says the padding value
 *     is 0) and column index -1 (the page prints '*' and leaves it open).
 *   - ELL width K = the longest row; an all-empty matrix has K = 0.
 *   - JDS: rows sorted by length, longest first, ties kept in original row
 *     order (the worked example puts r0 before r2); zero-length rows last.
 *   - HYB: the first min(len, K) entries of a row (in CSR order) stay in the
 *     ELL part, the rest go to the COO part in row order.
 *   - Sectioned ELL (the JDS variant): section height S is a parameter (the
 *     page leaves it open); sections are column-major with their own height,
 *     so the last section may be shorter; padding as in ELL.
 *   - Accumulation in the oracle is fp64, summed in CSR order.
 *
 * Parity status: every function here is pinned by tests (worked example of
 * Fig. 14.1 and the ELL/JDS figures, dense brute force, closed forms, round
 * trips, invariants), except or_select, whose comparison operators are
 * stripped in the source page: "parity unpinned" for its thresholds (its
 * outcome on the page's own described cases is still tested).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* Status values of the oracle (its own names; tests map them). */
#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_ROWPTRS 2
#define OR_COL_RANGE 3
#define OR_NO_MEMORY 4

/* Input sanity rules of [P5] section 5.3: row_ptr monotone non-decreasing,
 * every column index below the column count, value length = nnz (here:
 * rowPtrs[0] = 0 and rowPtrs[numRows] = nnz). Row-pointer errors are
 * reported before column errors. */
int or_validate_csr(int64_t R, int64_t C, int64_t Z, const int32_t *rowPtrs,
                    const int32_t *colIdx) {
    if (R < 0 || C < 0 || Z < 0) return OR_BAD_ARG;
    if (rowPtrs[0] != 0) return OR_BAD_ROWPTRS;
    for (int64_t r = 0; r < R; ++r)
        if (rowPtrs[r + 1] < rowPtrs[r]) return OR_BAD_ROWPTRS;
    if ((int64_t)rowPtrs[R] != Z) return OR_BAD_ROWPTRS;
    for (int64_t k = 0; k < Z; ++k)
        if (colIdx[k] < 0 || (int64_t)colIdx[k] >= C) return OR_COL_RANGE;
    return OR_OK;
}

/* Row-length statistics of [P3] section 4.1 (distribution histogram and
 * row-length variance): longest row, mean, population variance (two-pass,
 * fp64) and a log2 histogram with bin 0 = empty rows and bin b >= 1 holding
 * lengths in [2^(b-1), 2^b). */
void or_row_stats(int64_t R, const int32_t *rowPtrs, int64_t *maxLen,
                  double *mean, double *var, int64_t hist33[33]) {
    int64_t mx = 0;
    double sum = 0.0;
    for (int b = 0; b < 33; ++b) hist33[b] = 0;
    for (int64_t r = 0; r < R; ++r) {
        int64_t len = (int64_t)rowPtrs[r + 1] - rowPtrs[r];
        if (len > mx) mx = len;
        sum += (double)len;
        int b = 0;
        while (b < 32 && ((int64_t)1 << b) <= len) ++b;
        hist33[b] += 1;
    }
    double m = R > 0 ? sum / (double)R : 0.0;
    double ss = 0.0;
    for (int64_t r = 0; r < R; ++r) {
        double d = (double)((int64_t)rowPtrs[r + 1] - rowPtrs[r]) - m;
        ss += d * d;
    }
    *maxLen = mx;
    *mean = m;
    *var = R > 0 ? ss / (double)R : 0.0;
}

/* SpMV over CSR, [P1] "CSR format and SpMV": for each row, walk
 * value/colIdx from rowPtrs[row] to rowPtrs[row+1] and add the dot product
 * to y[row]. fp64 accumulation; also returns the per-row magnitude
 * sum_k |a_k x_col(k)| + |y0_row| used by the tolerance. */
void or_spmv_csr(int64_t R, const int32_t *rowPtrs, const int32_t *colIdx,
                 const float *value, const float *x, const float *y0,
                 double *y, double *mag) {
    for (int64_t r = 0; r < R; ++r) {
        double s = 0.0, a = 0.0;
        for (int64_t k = rowPtrs[r]; k < rowPtrs[r + 1]; ++k) {
            double p = (double)value[k] * (double)x[colIdx[k]];
            s += p;
            a += fabs(p);
        }
        y[r] = (double)y0[r] + s;
        if (mag) mag[r] = a + fabs((double)y0[r]);
    }
}

/* The same definition for a subset of rows (sampled checks at full size). */
void or_spmv_csr_rows(int64_t nrows, const int64_t *rows, const int32_t *rowPtrs,
                      const int32_t *colIdx, const float *value, const float *x,
                      const float *y0, double *y, double *mag) {
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        double s = 0.0, a = 0.0;
        for (int64_t k = rowPtrs[r]; k < rowPtrs[r + 1]; ++k) {
            double p = (double)value[k] * (double)x[colIdx[k]];
            s += p;
            a += fabs(p);
        }
        y[i] = (double)y0[r] + s;
        mag[i] = a + fabs((double)y0[r]);
    }
}

/* Dense row-major matrix to CSR, [P1] "CSR format and SpMV": nonzeros grouped
 * by row, ascending column inside a row, rowPtrs[numRows] = nnz. Returns nnz;
 * pass NULL outputs to count only. */
int64_t or_dense_to_csr(int64_t R, int64_t C, const float *A, int32_t *rowPtrs,
                        int32_t *colIdx, float *value) {
    int64_t z = 0;
    if (rowPtrs) rowPtrs[0] = 0;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t c = 0; c < C; ++c) {
            float a = A[r * C + c];
            if (a != 0.0f) {
                if (colIdx) { colIdx[z] = (int32_t)c; value[z] = a; }
                ++z;
            }
        }
        if (rowPtrs) rowPtrs[r + 1] = (int32_t)z;
    }
    return z;
}

/* CSR -> COO, [P1] "COO format and SpMV": every nonzero keeps its value and
 * column and gains its row index; order is unchanged (grouped by row). */
void or_csr_to_coo(int64_t R, const int32_t *rowPtrs, const int32_t *colIdx,
                   const float *value, int32_t *rowIdx, int32_t *cooCol,
                   float *cooVal) {
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = rowPtrs[r]; k < rowPtrs[r + 1]; ++k) {
            rowIdx[k] = (int32_t)r;
            cooCol[k] = colIdx[k];
            cooVal[k] = value[k];
        }
}

/* COO (grouped by row) -> CSR: count entries per row, prefix them. */
void or_coo_to_csr(int64_t R, int64_t Z, const int32_t *rowIdx, int32_t *rowPtrs) {
    for (int64_t r = 0; r <= R; ++r) rowPtrs[r] = 0;
    for (int64_t k = 0; k < Z; ++k) rowPtrs[rowIdx[k] + 1] += 1;
    for (int64_t r = 0; r < R; ++r) rowPtrs[r + 1] += rowPtrs[r];
}

/* CSR -> ELL, [P2] "ELL format": (1) pad every row to the longest row's
 * length, (2) lay the padded rectangle out column-major, so the t-th slot of
 * row r sits at i = t*numRows + r. nnzPerRow[r] keeps the true length.
 * ellCol/ellVal must hold R*K entries, K = longest row. */
void or_csr_to_ell(int64_t R, int64_t K, const int32_t *rowPtrs,
                   const int32_t *colIdx, const float *value, int32_t *nnzPerRow,
                   int32_t *ellCol, float *ellVal) {
    for (int64_t r = 0; r < R; ++r) {
        int64_t len = (int64_t)rowPtrs[r + 1] - rowPtrs[r];
        nnzPerRow[r] = (int32_t)len;
        for (int64_t t = 0; t < K; ++t) {
            int64_t i = t * R + r;
            if (t < len) {
                ellCol[i] = colIdx[rowPtrs[r] + t];
                ellVal[i] = value[rowPtrs[r] + t];
            } else {
                ellCol[i] = -1;
                ellVal[i] = 0.0f;
            }
        }
    }
}

/* ELL -> CSR: row r's entries are its first nnzPerRow[r] slots. */
void or_ell_to_csr(int64_t R, int64_t K, const int32_t *nnzPerRow,
                   const int32_t *ellCol, const float *ellVal, int32_t *rowPtrs,
                   int32_t *colIdx, float *value) {
    int64_t z = 0;
    rowPtrs[0] = 0;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < nnzPerRow[r]; ++t) {
            colIdx[z] = ellCol[t * R + r];
            value[z] = ellVal[t * R + r];
            ++z;
        }
        rowPtrs[r + 1] = (int32_t)z;
    }
    (void)K;
}

/* CSR -> hybrid ELL+COO, [P2] "Hybrid ELL-COO format": before the ELL step
 * the surplus entries of each row beyond width K are moved to a separate COO
 * part; the rest is an ELL of width K. Returns the number of COO entries;
 * pass NULL COO outputs to count only. */
int64_t or_csr_to_hyb(int64_t R, int64_t K, const int32_t *rowPtrs,
                      const int32_t *colIdx, const float *value,
                      int32_t *nnzPerRow, int32_t *ellCol, float *ellVal,
                      int32_t *cooRow, int32_t *cooCol, float *cooVal) {
    int64_t nc = 0;
    for (int64_t r = 0; r < R; ++r) {
        int64_t len = (int64_t)rowPtrs[r + 1] - rowPtrs[r];
        int64_t inEll = len < K ? len : K;
        if (nnzPerRow) {
            nnzPerRow[r] = (int32_t)inEll;
            for (int64_t t = 0; t < K; ++t) {
                int64_t i = t * R + r;
                if (t < inEll) {
                    ellCol[i] = colIdx[rowPtrs[r] + t];
                    ellVal[i] = value[rowPtrs[r] + t];
                } else {
                    ellCol[i] = -1;
                    ellVal[i] = 0.0f;
                }
            }
        }
        for (int64_t t = inEll; t < len; ++t) {
            if (cooRow) {
                cooRow[nc] = (int32_t)r;
                cooCol[nc] = colIdx[rowPtrs[r] + t];
                cooVal[nc] = value[rowPtrs[r] + t];
            }
            ++nc;
        }
    }
    return nc;
}

/* Hybrid -> CSR: row r = its ELL slots followed by its COO entries. */
void or_hyb_to_csr(int64_t R, int64_t K, const int32_t *nnzPerRow,
                   const int32_t *ellCol, const float *ellVal, int64_t nc,
                   const int32_t *cooRow, const int32_t *cooCol,
                   const float *cooVal, int32_t *rowPtrs, int32_t *colIdx,
                   float *value) {
    int64_t z = 0, c = 0;
    rowPtrs[0] = 0;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < nnzPerRow[r]; ++t) {
            colIdx[z] = ellCol[t * R + r];
            value[z] = ellVal[t * R + r];
            ++z;
        }
        while (c < nc && cooRow[c] == r) {
            colIdx[z] = cooCol[c];
            value[z] = cooVal[c];
            ++z;
            ++c;
        }
        rowPtrs[r + 1] = (int32_t)z;
    }
    (void)K;
}

/* CSR -> JDS, [P2] "JDS format", steps (1)-(4): (1) group by row as in CSR;
 * (2) sort the rows by their nonzero count, longest first, recording the
 * original row index of sorted row s in perm[s] (stable: equal lengths keep
 * original order); (3) store column-major: the t-th nonzero of every sorted
 * row that has one forms jagged diagonal t, sorted rows in order; (4)
 * iterPtr[t] = where diagonal t starts, iterPtr[maxLen] = nnz.
 * perm has R entries, iterPtr maxLen+1, jdsCol/jdsVal nnz. */
int or_csr_to_jds(int64_t R, int64_t maxLen, const int32_t *rowPtrs,
                  const int32_t *colIdx, const float *value, int32_t *perm,
                  int32_t *iterPtr, int32_t *jdsCol, float *jdsVal) {
    /* Stable counting sort by length, longest first. */
    int64_t *count = (int64_t *)calloc((size_t)maxLen + 2, sizeof(int64_t));
    if (!count) return OR_NO_MEMORY;
    for (int64_t r = 0; r < R; ++r) count[rowPtrs[r + 1] - rowPtrs[r]] += 1;
    /* first[len] = number of rows strictly longer than len */
    int64_t *first = (int64_t *)calloc((size_t)maxLen + 2, sizeof(int64_t));
    if (!first) { free(count); return OR_NO_MEMORY; }
    int64_t acc = 0;
    for (int64_t len = maxLen; len >= 0; --len) {
        first[len] = acc;
        acc += count[len];
    }
    for (int64_t r = 0; r < R; ++r) {
        int64_t len = rowPtrs[r + 1] - rowPtrs[r];
        perm[first[len]] = (int32_t)r;
        first[len] += 1;
    }
    /* iterPtr: diagonal t holds one entry per sorted row longer than t. */
    iterPtr[0] = 0;
    int64_t longer = R - count[0];
    for (int64_t t = 0; t < maxLen; ++t) {
        iterPtr[t + 1] = (int32_t)(iterPtr[t] + longer);
        longer -= count[t + 1];
    }
    for (int64_t s = 0; s < R; ++s) {
        int64_t r = perm[s];
        int64_t len = rowPtrs[r + 1] - rowPtrs[r];
        for (int64_t t = 0; t < len; ++t) {
            int64_t i = (int64_t)iterPtr[t] + s;
            jdsCol[i] = colIdx[rowPtrs[r] + t];
            jdsVal[i] = value[rowPtrs[r] + t];
        }
    }
    free(count);
    free(first);
    return OR_OK;
}

/* JDS -> CSR: sorted row s owns entry iterPtr[t] + s of every diagonal t
 * that is wider than s; put them back under row perm[s]. */
void or_jds_to_csr(int64_t R, int64_t maxLen, const int32_t *perm,
                   const int32_t *iterPtr, const int32_t *jdsCol,
                   const float *jdsVal, int32_t *rowPtrs, int32_t *colIdx,
                   float *value) {
    int32_t *lens = (int32_t *)calloc((size_t)R + 1, sizeof(int32_t));
    for (int64_t s = 0; s < R; ++s) {
        int64_t len = 0;
        while (len < maxLen && iterPtr[len] + s < iterPtr[len + 1]) ++len;
        lens[perm[s]] = (int32_t)len;
    }
    rowPtrs[0] = 0;
    for (int64_t r = 0; r < R; ++r) rowPtrs[r + 1] = rowPtrs[r] + lens[r];
    for (int64_t s = 0; s < R; ++s) {
        int64_t r = perm[s];
        for (int64_t t = 0; t < lens[r]; ++t) {
            colIdx[rowPtrs[r] + t] = jdsCol[iterPtr[t] + s];
            value[rowPtrs[r] + t] = jdsVal[iterPtr[t] + s];
        }
    }
    free(lens);
}

/* SpMV walking each format's own layout, fp64. */

/* [P1] "COO format and SpMV": one contribution per stored nonzero. */
void or_spmv_coo(int64_t R, int64_t Z, const int32_t *rowIdx, const int32_t *colIdx,
                 const float *value, const float *x, const float *y0, double *y) {
    for (int64_t r = 0; r < R; ++r) y[r] = (double)y0[r];
    for (int64_t k = 0; k < Z; ++k)
        y[rowIdx[k]] += (double)value[k] * (double)x[colIdx[k]];
}

/* [P2] "ELL format": row r reads slot t*numRows + r for t < nnzPerRow[r]. */
void or_spmv_ell(int64_t R, int64_t K, const int32_t *nnzPerRow,
                 const int32_t *ellCol, const float *ellVal, const float *x,
                 const float *y0, double *y) {
    for (int64_t r = 0; r < R; ++r) {
        double s = 0.0;
        for (int64_t t = 0; t < nnzPerRow[r]; ++t) {
            int64_t i = t * R + r;
            s += (double)ellVal[i] * (double)x[ellCol[i]];
        }
        y[r] = (double)y0[r] + s;
    }
    (void)K;
}

/* [P2] "Hybrid ELL-COO format": ELL part plus COO part, added into y. */
void or_spmv_hyb(int64_t R, int64_t K, const int32_t *nnzPerRow,
                 const int32_t *ellCol, const float *ellVal, int64_t nc,
                 const int32_t *cooRow, const int32_t *cooCol,
                 const float *cooVal, const float *x, const float *y0, double *y) {
    or_spmv_ell(R, K, nnzPerRow, ellCol, ellVal, x, y0, y);
    for (int64_t k = 0; k < nc; ++k)
        y[cooRow[k]] += (double)cooVal[k] * (double)x[cooCol[k]];
}

/* [P2] "JDS format": sorted row s walks diagonal t at iterPtr[t] + s while
 * that diagonal is wider than s; the sum goes back to row perm[s]. */
void or_spmv_jds(int64_t R, int64_t maxLen, const int32_t *perm,
                 const int32_t *iterPtr, const int32_t *jdsCol,
                 const float *jdsVal, const float *x, const float *y0, double *y) {
    for (int64_t r = 0; r < R; ++r) y[r] = (double)y0[r];
    for (int64_t s = 0; s < R; ++s) {
        double acc = 0.0;
        for (int64_t t = 0; t < maxLen && iterPtr[t] + s < iterPtr[t + 1]; ++t) {
            int64_t i = (int64_t)iterPtr[t] + s;
            acc += (double)jdsVal[i] * (double)x[jdsCol[i]];
        }
        y[perm[s]] += acc;
    }
}

/* Format selection, [P3] section 4.3. The page's comparison operators are
 * lost in extraction; the reading used here is: longest row <= 2 x mean ->
 * ELL; else mean < 10 -> COO; else HYB when longest > 5 x mean, otherwise
 * CSR. Two rules of ours come around it: a matrix whose compulsory SpMV
 * bytes (8 per nonzero, 12 per row, 4 per column) are below 4 MiB -> CSR
 * (too small to be bound by bandwidth: the format with the fewest dependent
 * memory round trips), checked first; and in the HYB case, columns that are
 * scattered (gatherLines, the sampled number of distinct 128-byte lines of x
 * among 32 consecutive nonzeros, at least 16) -> the x-blocked list of
 * "Introduction to sparse computing and performance bottleneck location".
 * (parity unpinned: the thresholds and their directions are a reading.)
 * Format codes as the library's: 0 COO, 1 CSR, 2 ELL, 3 HYB, 7 XBLOCK. */
int or_select(int64_t R, int64_t C, int64_t Z, int64_t maxLen, double gatherLines) {
    double mean = R > 0 ? (double)Z / (double)R : 0.0;
    if (8.0 * (double)Z + 12.0 * (double)R + 4.0 * (double)C < 4194304.0) return 1;
    if ((double)maxLen <= 2.0 * mean) return 2;
    if (mean < 10.0) return 0;
    if ((double)maxLen > 5.0 * mean) return gatherLines >= 16.0 ? 7 : 3;
    return 1;
}

/* Automatic HYB width: the smallest L such that at least 99% of the rows
 * have length <= L, i.e. 100 * #{len <= L} >= 99 * R ([P3] section 4.1's
 * example keeps the 99% of rows of length 10-20 whole in an ELL part of
 * width 20 and sends the few very long rows' surplus to COO). */
int64_t or_hyb_auto_width(int64_t R, const int32_t *rowPtrs, int64_t maxLen) {
    if (R == 0) return 0;
    int64_t *count = (int64_t *)calloc((size_t)maxLen + 1, sizeof(int64_t));
    for (int64_t r = 0; r < R; ++r) count[rowPtrs[r + 1] - rowPtrs[r]] += 1;
    int64_t cum = 0, L = 0;
    for (L = 0; L <= maxLen; ++L) {
        cum += count[L];
        if (100 * cum >= 99 * R) break;
    }
    free(count);
    return L;
}

/* CSR -> sectioned ELL, [P2] "JDS format", the variant paragraph: after the
 * rows are sorted by length (longest first, stable, as for JDS) they are cut
 * into sections of S consecutive sorted rows (the last section may be
 * shorter); each section is an ELL of its own, padded only to the length of
 * its longest (first) row and laid out column-major: slot t of the j-th row of
 * section k sits at secPtr[k] + t*h_k + j, h_k the section's row count.
 * secPtr[k] marks where section k starts (it replaces iterPtr); padding slots
 * hold column -1 and value +0.0f as in ELL. perm[s] = original row of sorted
 * row s. Returns the total slot count; pass NULL outputs to count only.
 * S < 1 is treated as 1. */
int64_t or_csr_to_sell(int64_t R, int64_t S, const int32_t *rowPtrs,
                       const int32_t *colIdx, const float *value, int32_t *perm,
                       int64_t *secPtr, int32_t *sellCol, float *sellVal) {
    if (S < 1) S = 1;
    int64_t maxLen = 0;
    for (int64_t r = 0; r < R; ++r)
        if (rowPtrs[r + 1] - rowPtrs[r] > maxLen) maxLen = rowPtrs[r + 1] - rowPtrs[r];
    /* stable counting sort by length, longest first */
    int64_t *first = (int64_t *)calloc((size_t)maxLen + 2, sizeof(int64_t));
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    for (int64_t r = 0; r < R; ++r) first[rowPtrs[r + 1] - rowPtrs[r]] += 1;
    int64_t acc = 0;
    for (int64_t len = maxLen; len >= 0; --len) {
        int64_t c = first[len];
        first[len] = acc;
        acc += c;
    }
    for (int64_t r = 0; r < R; ++r) order[first[rowPtrs[r + 1] - rowPtrs[r]]++] = (int32_t)r;
    int64_t nsec = (R + S - 1) / S, slots = 0;
    for (int64_t k = 0; k < nsec; ++k) {
        int64_t s0 = k * S, h = R - s0 < S ? R - s0 : S;
        int64_t w = rowPtrs[order[s0] + 1] - rowPtrs[order[s0]];
        if (secPtr) secPtr[k] = slots;
        if (sellCol) {
            for (int64_t j = 0; j < h; ++j) {
                int64_t r = order[s0 + j];
                int64_t len = rowPtrs[r + 1] - rowPtrs[r];
                for (int64_t t = 0; t < w; ++t) {
                    int64_t i = slots + t * h + j;
                    if (t < len) {
                        sellCol[i] = colIdx[rowPtrs[r] + t];
                        sellVal[i] = value[rowPtrs[r] + t];
                    } else {
                        sellCol[i] = -1;
                        sellVal[i] = 0.0f;
                    }
                }
            }
        }
        slots += h * w;
    }
    if (secPtr) secPtr[nsec] = slots;
    if (perm)
        for (int64_t s = 0; s < R; ++s) perm[s] = order[s];
    free(first);
    free(order);
    return slots;
}

/* Sectioned ELL -> CSR: a row's entries are its leading non-padding slots. */
void or_sell_to_csr(int64_t R, int64_t S, const int32_t *perm, const int64_t *secPtr,
                    const int32_t *sellCol, const float *sellVal, int32_t *rowPtrs,
                    int32_t *colIdx, float *value) {
    if (S < 1) S = 1;
    int64_t nsec = (R + S - 1) / S;
    int32_t *lens = (int32_t *)calloc((size_t)R + 1, sizeof(int32_t));
    for (int64_t k = 0; k < nsec; ++k) {
        int64_t s0 = k * S, h = R - s0 < S ? R - s0 : S;
        int64_t w = h > 0 ? (secPtr[k + 1] - secPtr[k]) / h : 0;
        for (int64_t j = 0; j < h; ++j) {
            int64_t len = 0;
            while (len < w && sellCol[secPtr[k] + len * h + j] >= 0) ++len;
            lens[perm[s0 + j]] = (int32_t)len;
        }
    }
    rowPtrs[0] = 0;
    for (int64_t r = 0; r < R; ++r) rowPtrs[r + 1] = rowPtrs[r] + lens[r];
    for (int64_t k = 0; k < nsec; ++k) {
        int64_t s0 = k * S, h = R - s0 < S ? R - s0 : S;
        for (int64_t j = 0; j < h; ++j) {
            int64_t r = perm[s0 + j];
            for (int64_t t = 0; t < lens[r]; ++t) {
                colIdx[rowPtrs[r] + t] = sellCol[secPtr[k] + t * h + j];
                value[rowPtrs[r] + t] = sellVal[secPtr[k] + t * h + j];
            }
        }
    }
    free(lens);
}

/* SpMV over the sectioned ELL: sorted row s (section k, position j) sums
 * its non-padding slots and adds the result to y[perm[s]]. fp64. */
void or_spmv_sell(int64_t R, int64_t S, const int32_t *perm, const int64_t *secPtr,
                  const int32_t *sellCol, const float *sellVal, const float *x,
                  const float *y0, double *y) {
    if (S < 1) S = 1;
    for (int64_t r = 0; r < R; ++r) y[r] = (double)y0[r];
    int64_t nsec = (R + S - 1) / S;
    for (int64_t k = 0; k < nsec; ++k) {
        int64_t s0 = k * S, h = R - s0 < S ? R - s0 : S;
        int64_t w = h > 0 ? (secPtr[k + 1] - secPtr[k]) / h : 0;
        for (int64_t j = 0; j < h; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < w; ++t) {
                int64_t i = secPtr[k] + t * h + j;
                if (sellCol[i] >= 0) acc += (double)sellVal[i] * (double)x[sellCol[i]];
            }
            y[perm[s0 + j]] += acc;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Conjugate gradient around the SpMV ([P1] "Background & SpMV": for a
 * positive-definite A the system A·X + Y = 0 is solved iteratively -- take a
 * guess X, form A·X + Y, stop when it is close to zero, otherwise correct X
 * along a direction built from the gradient). A·X + Y is the gradient of
 * f(X) = X'AX/2 + Y'X, so this is the textbook method of Hestenes and
 * Stiefel (1952) for A X = -Y, written with the gradient g = A·X + Y:
 *   g_0 = A·X_0 + Y,  d_0 = -g_0
 *   iteration k:  q = A d_k,  alpha = (g_k'g_k) / (d_k'q)
 *                 X_{k+1} = X_k + alpha d_k,  g_{k+1} = g_k + alpha q
 *                 stop when |g_{k+1}| <= tol |Y|
 *                 beta = (g_{k+1}'g_{k+1}) / (g_k'g_k),  d_{k+1} = -g_{k+1} + beta d_k
 * fp64 throughout. X (R doubles) gets the last iterate. gnorm, when not NULL
 * (maxIter + 1 doubles), gets |g_k| for k = 0 .. iterations. *status: 0 =
 * stopped by the tolerance (or g = 0 exactly), 1 = maxIter reached, 2 = the
 * curvature d'q was not positive (A not positive definite). Returns the
 * number of iterations done.
 * ------------------------------------------------------------------------- */
static void csr_apply_f64(int64_t R, const int32_t *rowPtrs, const int32_t *colIdx,
                          const float *value, const double *v, double *out) {
    for (int64_t r = 0; r < R; ++r) {
        double s = 0.0;
        for (int64_t k = rowPtrs[r]; k < rowPtrs[r + 1]; ++k)
            s += (double)value[k] * v[colIdx[k]];
        out[r] = s;
    }
}

static double dot_f64(int64_t n, const double *a, const double *b) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

int64_t or_cg_csr(int64_t R, const int32_t *rowPtrs, const int32_t *colIdx,
                  const float *value, const float *Y, const float *X0, int64_t maxIter,
                  double tol, double *X, double *gnorm, int32_t *status) {
    size_t n = (size_t)(R > 0 ? R : 1);
    double *g = (double *)malloc(sizeof(double) * n);
    double *d = (double *)malloc(sizeof(double) * n);
    double *q = (double *)malloc(sizeof(double) * n);
    for (int64_t i = 0; i < R; ++i) X[i] = X0 ? (double)X0[i] : 0.0;
    /* g_0 = A·X_0 + Y */
    csr_apply_f64(R, rowPtrs, colIdx, value, X, g);
    double yy = 0.0;
    for (int64_t i = 0; i < R; ++i) {
        g[i] += (double)Y[i];
        yy += (double)Y[i] * (double)Y[i];
        d[i] = -g[i];
    }
    double gg = dot_f64(R, g, g);
    const double stop = tol * sqrt(yy);
    if (gnorm) gnorm[0] = sqrt(gg);
    int64_t k = 0;
    *status = 1;
    if (sqrt(gg) <= stop || gg == 0.0) *status = 0;
    while (*status == 1 && k < maxIter) {
        csr_apply_f64(R, rowPtrs, colIdx, value, d, q);
        double dq = dot_f64(R, d, q);
        if (!(dq > 0.0)) {
            *status = 2;
            break;
        }
        double alpha = gg / dq;
        for (int64_t i = 0; i < R; ++i) {
            X[i] += alpha * d[i];
            g[i] += alpha * q[i];
        }
        double ggNew = dot_f64(R, g, g);
        ++k;
        if (gnorm) gnorm[k] = sqrt(ggNew);
        if (sqrt(ggNew) <= stop || ggNew == 0.0) {
            *status = 0;
            break;
        }
        double beta = ggNew / gg;
        for (int64_t i = 0; i < R; ++i) d[i] = -g[i] + beta * d[i];
        gg = ggNew;
    }
    free(g);
    free(d);
    free(q);
    return k;
}

/* ---------------------------------------------------------------------------
 * x-blocked list ([P4] "Building the problem framework", memory efficiency:
 * with random columns, split x into chunks and let a thread block handle
 * only the nonzeros whose columns fall in one chunk, so that the gather stays
 * local -- "blocking + reordering"). Chunk c covers the columns
 * [c*B, min(C, (c+1)*B)); its entries are the nonzeros whose column falls in
 * it, in CSR order (by row, then by position in the row), stored from
 * chunkPtr[c]: row index, local column col - c*B (16 bits, B <= 65536) and
 * value. Each chunk is padded to a multiple of 4 entries with (row -1, local
 * column 0, value +0.0f). Returns the slot count chunkPtr[nChunks]; the
 * arrays may be NULL to only count.
 * ------------------------------------------------------------------------- */
int64_t or_csr_to_xblock(int64_t R, int64_t C, int64_t B, const int32_t *rowPtrs,
                         const int32_t *colIdx, const float *value, int64_t *chunkPtr,
                         int32_t *xbRow, uint16_t *xbCol, float *xbVal) {
    if (B < 1) B = 1;
    int64_t nch = (C + B - 1) / B;
    int64_t *cnt = (int64_t *)calloc((size_t)(nch > 0 ? nch : 1), sizeof(int64_t));
    int64_t *cur = (int64_t *)calloc((size_t)(nch > 0 ? nch : 1), sizeof(int64_t));
    int64_t Z = R > 0 ? rowPtrs[R] : 0;
    for (int64_t k = 0; k < Z; ++k) cnt[colIdx[k] / B] += 1;
    int64_t slots = 0;
    for (int64_t c = 0; c < nch; ++c) {
        if (chunkPtr) chunkPtr[c] = slots;
        cur[c] = slots;
        slots += (cnt[c] + 3) / 4 * 4;
    }
    if (chunkPtr) chunkPtr[nch] = slots;
    if (xbRow) {
        for (int64_t r = 0; r < R; ++r)
            for (int64_t k = rowPtrs[r]; k < rowPtrs[r + 1]; ++k) {
                int64_t c = colIdx[k] / B, i = cur[c]++;
                xbRow[i] = (int32_t)r;
                xbCol[i] = (uint16_t)(colIdx[k] - c * B);
                xbVal[i] = value[k];
            }
        for (int64_t c = 0; c < nch; ++c)
            for (int64_t i = cur[c]; i < (cur[c] + 3) / 4 * 4; ++i) {  /* to the padded end */
                xbRow[i] = -1;
                xbCol[i] = 0;
                xbVal[i] = 0.0f;
            }
    }
    free(cnt);
    free(cur);
    return slots;
}

/* x-blocked list -> CSR: each row's entries in chunk order, then in stored
 * order (the original order when every row's columns ascend). */
void or_xblock_to_csr(int64_t R, int64_t B, int64_t nch, const int64_t *chunkPtr,
                      const int32_t *xbRow, const uint16_t *xbCol, const float *xbVal,
                      int32_t *rowPtrs, int32_t *colIdx, float *value) {
    if (B < 1) B = 1;
    int64_t slots = chunkPtr[nch];
    for (int64_t r = 0; r <= R; ++r) rowPtrs[r] = 0;
    for (int64_t i = 0; i < slots; ++i)
        if (xbRow[i] >= 0) rowPtrs[xbRow[i] + 1] += 1;
    for (int64_t r = 0; r < R; ++r) rowPtrs[r + 1] += rowPtrs[r];
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(R > 0 ? R : 1));
    for (int64_t r = 0; r < R; ++r) pos[r] = rowPtrs[r];
    for (int64_t c = 0; c < nch; ++c)
        for (int64_t i = chunkPtr[c]; i < chunkPtr[c + 1]; ++i) {
            if (xbRow[i] < 0) continue;
            int64_t k = pos[xbRow[i]]++;
            colIdx[k] = (int32_t)(c * B + xbCol[i]);
            value[k] = xbVal[i];
        }
    free(pos);
}

/* SpMV over the x-blocked list: every non-padding entry adds val*x[c*B +
 * local column] to its row, rows summed in fp64 in storage order. */
void or_spmv_xblock(int64_t R, int64_t B, int64_t nch, const int64_t *chunkPtr,
                    const int32_t *xbRow, const uint16_t *xbCol, const float *xbVal,
                    const float *x, const float *y0, double *y) {
    if (B < 1) B = 1;
    for (int64_t r = 0; r < R; ++r) y[r] = (double)y0[r];
    for (int64_t c = 0; c < nch; ++c)
        for (int64_t i = chunkPtr[c]; i < chunkPtr[c + 1]; ++i)
            if (xbRow[i] >= 0)
                y[xbRow[i]] += (double)xbVal[i] * (double)x[c * B + xbCol[i]];
}

/* ---------------------------------------------------------------------------
 * SpMV with 8-byte values ([P4] "Building the problem framework": a
 * nonzero's value and an x entry take 4 or 8 bytes; [P1] "Background &
 * SpMV": y <- A*x + y). fp64 inputs; every product is split exactly into
 * p + e (p = a*x rounded, e = fma(a, x, -p)), and the row is summed with
 * Neumaier's compensated summation, so y_i is within about one rounding of
 * the exact value whatever the order in which the code under test adds.
 * mag_i = |y0_i| + sum_k |a_k x_col(k)|.
 * ------------------------------------------------------------------------- */
static void neumaier_add(double *s, double *c, double t) {
    double u = *s + t;
    if (fabs(*s) >= fabs(t))
        *c += (*s - u) + t;
    else
        *c += (t - u) + *s;
    *s = u;
}

void or_spmv_csr_f64(int64_t R, const int32_t *rowPtrs, const int32_t *colIdx,
                     const double *value, const double *x, const double *y0, double *y,
                     double *mag) {
    for (int64_t r = 0; r < R; ++r) {
        double s = y0[r], c = 0.0, a = fabs(y0[r]);
        for (int64_t k = rowPtrs[r]; k < rowPtrs[r + 1]; ++k) {
            double p = value[k] * x[colIdx[k]];
            double e = fma(value[k], x[colIdx[k]], -p);
            neumaier_add(&s, &c, p);
            c += e;
            a += fabs(p);
        }
        y[r] = s + c;
        if (mag) mag[r] = a;
    }
}
