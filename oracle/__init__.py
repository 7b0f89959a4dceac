"""NumPy front end of the C oracle (``spmv_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check in
``__graft_entry__`` and by the CPU-baseline leg of ``bench.py``. The product
library never imports it, and it imports nothing from the product.

Every function follows the pages cited in ``spmv_oracle.c``; all sums are
fp64 in CSR order. Parity status per function:

* validate, row stats, SpMV (every format), CSR<->COO/ELL/HYB/JDS: pinned by
  the worked examples of Fig. 14.1 and the ELL/JDS figures, dense brute force,
  closed forms, round trips and invariants (``tests/test_oracle_*.py``).
* ``cg`` (conjugate gradient for A·X + Y = 0): pinned by closed-form
  eigenpairs of the Dirichlet Laplacian (one-step convergence), finite
  termination on matrices with few distinct eigenvalues, a dense direct
  solve, and the monotone decrease of the A-norm error
  (``tests/test_oracle_cg.py``).
* x-blocked list (CSR<->XBLOCK, its SpMV): pinned by hand-worked Fig. 14.1
  chunkings, reduction to the oracle's COO when one chunk holds every
  column, dense brute force, round trips and layout invariants
  (``tests/test_oracle_xblock.py``).
* ``spmv_csr_f64`` (8-byte values): pinned by exact rational arithmetic
  (``fractions``), Fig. 14.1, sums that need 8-byte values, and a
  cancellation that only compensated summation gets right
  (``tests/test_oracle_f64.py``).
* ``select``: parity unpinned (the page's comparison operators are stripped);
  only its outcome on the cases the page describes in words is checked.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_i64 = C.c_int64
_p = C.c_void_p

_SIGS = {
    "or_validate_csr": (C.c_int, [_i64, _i64, _i64, _p, _p]),
    "or_row_stats": (None, [_i64, _p, _p, _p, _p, _p]),
    "or_spmv_csr": (None, [_i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_spmv_csr_rows": (None, [_i64, _p, _p, _p, _p, _p, _p, _p, _p]),
    "or_dense_to_csr": (_i64, [_i64, _i64, _p, _p, _p, _p]),
    "or_csr_to_coo": (None, [_i64, _p, _p, _p, _p, _p, _p]),
    "or_coo_to_csr": (None, [_i64, _i64, _p, _p]),
    "or_csr_to_ell": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p]),
    "or_ell_to_csr": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p]),
    "or_csr_to_hyb": (_i64, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p, _p, _p]),
    "or_hyb_to_csr": (None, [_i64, _i64, _p, _p, _p, _i64, _p, _p, _p, _p, _p, _p]),
    "or_csr_to_jds": (C.c_int, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_jds_to_csr": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_spmv_coo": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p]),
    "or_spmv_ell": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p]),
    "or_spmv_hyb": (None, [_i64, _i64, _p, _p, _p, _i64, _p, _p, _p, _p, _p, _p]),
    "or_spmv_jds": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_csr_to_sell": (_i64, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_sell_to_csr": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_spmv_sell": (None, [_i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_csr_to_xblock": (_i64, [_i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_xblock_to_csr": (None, [_i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_spmv_xblock": (None, [_i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_spmv_csr_f64": (None, [_i64, _p, _p, _p, _p, _p, _p, _p]),
    "or_cg_csr": (_i64, [_i64, _p, _p, _p, _p, _p, _i64, C.c_double, _p, _p, _p]),
    "or_select": (C.c_int, [_i64, _i64, _i64, _i64, C.c_double]),
    "or_hyb_auto_width": (_i64, [_i64, _p, _i64]),
}

OK, BAD_ARG, BAD_ROWPTRS, COL_RANGE, NO_MEMORY = 0, 1, 2, 3, 4
FORMAT_NAMES = {0: "COO", 1: "CSR", 2: "ELL", 3: "HYB", 7: "XBLOCK"}

_lib = None


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        lib = C.CDLL(path)
    else:
        if _lib is not None:
            return _lib
        lib = C.CDLL(_build.build())
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p) if a.size else None


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """Bound view of one oracle library (the default build or a variant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # --- checks and statistics -------------------------------------------
    def validate(self, num_rows, num_cols, row_ptrs, col_idx):
        rp, ci = _i32(row_ptrs), _i32(col_idx)
        if rp.shape[0] != num_rows + 1:
            return BAD_ROWPTRS
        return self.lib.or_validate_csr(num_rows, num_cols, ci.shape[0], _ptr(rp), _ptr(ci))

    def row_stats(self, row_ptrs):
        rp = _i32(row_ptrs)
        R = rp.shape[0] - 1
        mx = np.zeros(1, np.int64)
        mean = np.zeros(1, np.float64)
        var = np.zeros(1, np.float64)
        hist = np.zeros(33, np.int64)
        self.lib.or_row_stats(R, _ptr(rp), _ptr(mx), _ptr(mean), _ptr(var), _ptr(hist))
        return {"max_len": int(mx[0]), "mean": float(mean[0]), "var": float(var[0]),
                "hist_log2": hist}

    # --- SpMV --------------------------------------------------------------
    def spmv_csr(self, row_ptrs, col_idx, value, x, y0):
        """y = A x + y0 in fp64 and the per-row magnitude sum |a x| + |y0|."""
        rp, ci, v, xx, yy = _i32(row_ptrs), _i32(col_idx), _f32(value), _f32(x), _f32(y0)
        R = rp.shape[0] - 1
        y = np.zeros(R, np.float64)
        mag = np.zeros(R, np.float64)
        self.lib.or_spmv_csr(R, _ptr(rp), _ptr(ci), _ptr(v), _ptr(xx), _ptr(yy), _ptr(y), _ptr(mag))
        return y, mag

    def spmv_csr_rows(self, rows, row_ptrs, col_idx, value, x, y0):
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp, ci, v, xx, yy = _i32(row_ptrs), _i32(col_idx), _f32(value), _f32(x), _f32(y0)
        y = np.zeros(rows.shape[0], np.float64)
        mag = np.zeros(rows.shape[0], np.float64)
        self.lib.or_spmv_csr_rows(rows.shape[0], _ptr(rows), _ptr(rp), _ptr(ci), _ptr(v),
                                  _ptr(xx), _ptr(yy), _ptr(y), _ptr(mag))
        return y, mag

    def spmv_coo(self, num_rows, row_idx, col_idx, value, x, y0):
        ri, ci, v, xx, yy = _i32(row_idx), _i32(col_idx), _f32(value), _f32(x), _f32(y0)
        y = np.zeros(num_rows, np.float64)
        self.lib.or_spmv_coo(num_rows, ri.shape[0], _ptr(ri), _ptr(ci), _ptr(v), _ptr(xx),
                             _ptr(yy), _ptr(y))
        return y

    def spmv_ell(self, ell, x, y0):
        R = ell["num_rows"]
        y = np.zeros(R, np.float64)
        self.lib.or_spmv_ell(R, ell["width"], _ptr(ell["nnz_per_row"]), _ptr(ell["col_idx"]),
                             _ptr(ell["value"]), _ptr(_f32(x)), _ptr(_f32(y0)), _ptr(y))
        return y

    def spmv_hyb(self, hyb, x, y0):
        R = hyb["num_rows"]
        y = np.zeros(R, np.float64)
        self.lib.or_spmv_hyb(R, hyb["width"], _ptr(hyb["nnz_per_row"]), _ptr(hyb["col_idx"]),
                             _ptr(hyb["value"]), hyb["coo_row_idx"].shape[0],
                             _ptr(hyb["coo_row_idx"]), _ptr(hyb["coo_col_idx"]),
                             _ptr(hyb["coo_value"]), _ptr(_f32(x)), _ptr(_f32(y0)), _ptr(y))
        return y

    def spmv_jds(self, jds, x, y0):
        R = jds["num_rows"]
        y = np.zeros(R, np.float64)
        self.lib.or_spmv_jds(R, jds["max_len"], _ptr(jds["perm"]), _ptr(jds["iter_ptr"]),
                             _ptr(jds["col_idx"]), _ptr(jds["value"]), _ptr(_f32(x)),
                             _ptr(_f32(y0)), _ptr(y))
        return y

    # --- conversions -------------------------------------------------------
    def dense_to_csr(self, A):
        A = np.ascontiguousarray(A, dtype=np.float32)
        R, Cc = A.shape
        z = self.lib.or_dense_to_csr(R, Cc, _ptr(A), None, None, None)
        rp = np.zeros(R + 1, np.int32)
        ci = np.zeros(z, np.int32)
        v = np.zeros(z, np.float32)
        self.lib.or_dense_to_csr(R, Cc, _ptr(A), _ptr(rp), _ptr(ci), _ptr(v))
        return rp, ci, v

    def csr_to_coo(self, row_ptrs, col_idx, value):
        rp, ci, v = _i32(row_ptrs), _i32(col_idx), _f32(value)
        R, Z = rp.shape[0] - 1, ci.shape[0]
        ri = np.zeros(Z, np.int32)
        co = np.zeros(Z, np.int32)
        vo = np.zeros(Z, np.float32)
        self.lib.or_csr_to_coo(R, _ptr(rp), _ptr(ci), _ptr(v), _ptr(ri), _ptr(co), _ptr(vo))
        return {"row_idx": ri, "col_idx": co, "value": vo}

    def coo_to_csr(self, num_rows, row_idx):
        ri = _i32(row_idx)
        rp = np.zeros(num_rows + 1, np.int32)
        self.lib.or_coo_to_csr(num_rows, ri.shape[0], _ptr(ri), _ptr(rp))
        return rp

    def csr_to_ell(self, row_ptrs, col_idx, value, width=None):
        rp, ci, v = _i32(row_ptrs), _i32(col_idx), _f32(value)
        R = rp.shape[0] - 1
        K = int(np.diff(rp.astype(np.int64)).max()) if R and width is None else (width or 0)
        npr = np.zeros(R, np.int32)
        ec = np.zeros(R * K, np.int32)
        ev = np.zeros(R * K, np.float32)
        self.lib.or_csr_to_ell(R, K, _ptr(rp), _ptr(ci), _ptr(v), _ptr(npr), _ptr(ec), _ptr(ev))
        return {"num_rows": R, "width": K, "nnz_per_row": npr, "col_idx": ec, "value": ev}

    def ell_to_csr(self, ell):
        R, K = ell["num_rows"], ell["width"]
        Z = int(ell["nnz_per_row"].astype(np.int64).sum())
        rp = np.zeros(R + 1, np.int32)
        ci = np.zeros(Z, np.int32)
        v = np.zeros(Z, np.float32)
        self.lib.or_ell_to_csr(R, K, _ptr(ell["nnz_per_row"]), _ptr(ell["col_idx"]),
                               _ptr(ell["value"]), _ptr(rp), _ptr(ci), _ptr(v))
        return rp, ci, v

    def csr_to_hyb(self, row_ptrs, col_idx, value, width):
        rp, ci, v = _i32(row_ptrs), _i32(col_idx), _f32(value)
        R, K = rp.shape[0] - 1, int(width)
        nc = self.lib.or_csr_to_hyb(R, K, _ptr(rp), _ptr(ci), _ptr(v), None, None, None,
                                    None, None, None)
        npr = np.zeros(R, np.int32)
        ec = np.zeros(R * K, np.int32)
        ev = np.zeros(R * K, np.float32)
        cr = np.zeros(nc, np.int32)
        cc = np.zeros(nc, np.int32)
        cv = np.zeros(nc, np.float32)
        self.lib.or_csr_to_hyb(R, K, _ptr(rp), _ptr(ci), _ptr(v), _ptr(npr), _ptr(ec), _ptr(ev),
                               _ptr(cr), _ptr(cc), _ptr(cv))
        return {"num_rows": R, "width": K, "nnz_per_row": npr, "col_idx": ec, "value": ev,
                "coo_row_idx": cr, "coo_col_idx": cc, "coo_value": cv}

    def hyb_to_csr(self, hyb):
        R, K = hyb["num_rows"], hyb["width"]
        nc = hyb["coo_row_idx"].shape[0]
        Z = int(hyb["nnz_per_row"].astype(np.int64).sum()) + nc
        rp = np.zeros(R + 1, np.int32)
        ci = np.zeros(Z, np.int32)
        v = np.zeros(Z, np.float32)
        self.lib.or_hyb_to_csr(R, K, _ptr(hyb["nnz_per_row"]), _ptr(hyb["col_idx"]),
                               _ptr(hyb["value"]), nc, _ptr(hyb["coo_row_idx"]),
                               _ptr(hyb["coo_col_idx"]), _ptr(hyb["coo_value"]), _ptr(rp),
                               _ptr(ci), _ptr(v))
        return rp, ci, v

    def csr_to_jds(self, row_ptrs, col_idx, value):
        rp, ci, v = _i32(row_ptrs), _i32(col_idx), _f32(value)
        R, Z = rp.shape[0] - 1, ci.shape[0]
        L = int(np.diff(rp.astype(np.int64)).max()) if R else 0
        perm = np.zeros(R, np.int32)
        ip = np.zeros(L + 1, np.int32)
        jc = np.zeros(Z, np.int32)
        jv = np.zeros(Z, np.float32)
        st = self.lib.or_csr_to_jds(R, L, _ptr(rp), _ptr(ci), _ptr(v), _ptr(perm), _ptr(ip),
                                    _ptr(jc), _ptr(jv))
        if st != OK:
            raise MemoryError("oracle JDS conversion ran out of memory")
        return {"num_rows": R, "max_len": L, "perm": perm, "iter_ptr": ip, "col_idx": jc,
                "value": jv}

    def jds_to_csr(self, jds):
        R, L = jds["num_rows"], jds["max_len"]
        Z = jds["col_idx"].shape[0]
        rp = np.zeros(R + 1, np.int32)
        ci = np.zeros(Z, np.int32)
        v = np.zeros(Z, np.float32)
        self.lib.or_jds_to_csr(R, L, _ptr(jds["perm"]), _ptr(jds["iter_ptr"]),
                               _ptr(jds["col_idx"]), _ptr(jds["value"]), _ptr(rp), _ptr(ci),
                               _ptr(v))
        return rp, ci, v

    def csr_to_sell(self, row_ptrs, col_idx, value, section_rows):
        rp, ci, v = _i32(row_ptrs), _i32(col_idx), _f32(value)
        R, S = rp.shape[0] - 1, int(section_rows)
        n = self.lib.or_csr_to_sell(R, S, _ptr(rp), _ptr(ci), _ptr(v), None, None, None, None)
        Se = max(S, 1)
        nsec = (R + Se - 1) // Se
        perm = np.zeros(R, np.int32)
        sp = np.zeros(nsec + 1, np.int64)
        sc = np.zeros(n, np.int32)
        sv = np.zeros(n, np.float32)
        self.lib.or_csr_to_sell(R, S, _ptr(rp), _ptr(ci), _ptr(v), _ptr(perm), _ptr(sp),
                                _ptr(sc), _ptr(sv))
        return {"num_rows": R, "section_rows": Se, "perm": perm, "sec_ptr": sp,
                "col_idx": sc, "value": sv}

    def sell_to_csr(self, sell):
        R, S = sell["num_rows"], sell["section_rows"]
        Z = int((sell["col_idx"] >= 0).sum())
        rp = np.zeros(R + 1, np.int32)
        ci = np.zeros(Z, np.int32)
        v = np.zeros(Z, np.float32)
        self.lib.or_sell_to_csr(R, S, _ptr(sell["perm"]), _ptr(sell["sec_ptr"]),
                                _ptr(sell["col_idx"]), _ptr(sell["value"]), _ptr(rp), _ptr(ci),
                                _ptr(v))
        return rp, ci, v

    def spmv_csr_f64(self, row_ptrs, col_idx, value, x, y0):
        """y = A x + y0 with 8-byte values and vectors (compensated fp64 sums);
        returns (y, mag) with mag = |y0| + sum |a x| per row."""
        rp, ci = _i32(row_ptrs), _i32(col_idx)
        v = np.ascontiguousarray(value, np.float64)
        xx = np.ascontiguousarray(x, np.float64)
        yy = np.ascontiguousarray(y0, np.float64)
        R = rp.shape[0] - 1
        y = np.zeros(max(R, 1), np.float64)
        mag = np.zeros(max(R, 1), np.float64)
        self.lib.or_spmv_csr_f64(R, _ptr(rp), _ptr(ci), _ptr(v), _ptr(xx), _ptr(yy), _ptr(y),
                                 _ptr(mag))
        return y[:R], mag[:R]

    def csr_to_xblock(self, row_ptrs, col_idx, value, num_cols, chunk_cols):
        """x-blocked list: {num_rows, chunk_cols, num_chunks, chunk_ptr (int64),
        row_idx (int32, -1 padding), col16 (uint16 local column), value}."""
        rp, ci, v = _i32(row_ptrs), _i32(col_idx), _f32(value)
        R, C, B = rp.shape[0] - 1, int(num_cols), int(chunk_cols)
        Be = max(B, 1)
        nch = (C + Be - 1) // Be
        n = self.lib.or_csr_to_xblock(R, C, B, _ptr(rp), _ptr(ci), _ptr(v), None, None, None,
                                      None)
        cp = np.zeros(nch + 1, np.int64)
        rows = np.zeros(n, np.int32)
        cols = np.zeros(n, np.uint16)
        vals = np.zeros(n, np.float32)
        self.lib.or_csr_to_xblock(R, C, B, _ptr(rp), _ptr(ci), _ptr(v), _ptr(cp), _ptr(rows),
                                  _ptr(cols), _ptr(vals))
        return {"num_rows": R, "chunk_cols": Be, "num_chunks": nch, "chunk_ptr": cp,
                "row_idx": rows, "col16": cols, "value": vals}

    def xblock_to_csr(self, xb):
        R = xb["num_rows"]
        Z = int((xb["row_idx"] >= 0).sum())
        rp = np.zeros(R + 1, np.int32)
        ci = np.zeros(Z, np.int32)
        v = np.zeros(Z, np.float32)
        self.lib.or_xblock_to_csr(R, xb["chunk_cols"], xb["num_chunks"], _ptr(xb["chunk_ptr"]),
                                  _ptr(xb["row_idx"]), _ptr(xb["col16"]), _ptr(xb["value"]),
                                  _ptr(rp), _ptr(ci), _ptr(v))
        return rp, ci, v

    def spmv_xblock(self, xb, x, y0):
        R = xb["num_rows"]
        y = np.zeros(max(R, 1), np.float64)
        self.lib.or_spmv_xblock(R, xb["chunk_cols"], xb["num_chunks"], _ptr(xb["chunk_ptr"]),
                                _ptr(xb["row_idx"]), _ptr(xb["col16"]), _ptr(xb["value"]),
                                _ptr(_f32(x)), _ptr(_f32(y0)), _ptr(y))
        return y[:R]

    def cg(self, row_ptrs, col_idx, value, Y, X0=None, max_iter=1000, tol=1e-6):
        """Conjugate gradient for A·X + Y = 0 (A symmetric positive definite).
        Returns {"x": fp64 X, "iterations", "status" (0 tolerance, 1 max_iter,
        2 non-positive curvature), "gnorm": |A·X_k + Y| for k = 0..iterations}."""
        rp, ci, v, y = _i32(row_ptrs), _i32(col_idx), _f32(value), _f32(Y)
        R = rp.shape[0] - 1
        x0 = None if X0 is None else _f32(X0)
        x = np.zeros(max(R, 1), np.float64)
        gn = np.zeros(int(max_iter) + 1, np.float64)
        st = np.zeros(1, np.int32)
        k = self.lib.or_cg_csr(R, _ptr(rp), _ptr(ci), _ptr(v), _ptr(y),
                               None if x0 is None else _ptr(x0), int(max_iter), float(tol),
                               _ptr(x), _ptr(gn), _ptr(st))
        return {"x": x[:R], "iterations": int(k), "status": int(st[0]), "gnorm": gn[:k + 1]}

    def spmv_sell(self, sell, x, y0):
        R = sell["num_rows"]
        y = np.zeros(R, np.float64)
        self.lib.or_spmv_sell(R, sell["section_rows"], _ptr(sell["perm"]), _ptr(sell["sec_ptr"]),
                              _ptr(sell["col_idx"]), _ptr(sell["value"]), _ptr(_f32(x)),
                              _ptr(_f32(y0)), _ptr(y))
        return y

    # --- selection -----------------------------------------------------------
    def select(self, num_rows, num_cols, nnz, max_len, gather_lines):
        return FORMAT_NAMES[self.lib.or_select(num_rows, num_cols, nnz, max_len,
                                               float(gather_lines))]

    def hyb_auto_width(self, row_ptrs):
        rp = _i32(row_ptrs)
        R = rp.shape[0] - 1
        L = int(np.diff(rp.astype(np.int64)).max()) if R else 0
        return int(self.lib.or_hyb_auto_width(R, _ptr(rp), L))


_default = None


def get() -> Oracle:
    """The oracle bound to the default build."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def within_tolerance(y_test, y_ref, mag, rel=1e-5, abs_floor=1e-30):
    """Per-row check |y_test - y_ref| <= rel * (sum_j |a_ij x_j| + |y0_i|) + abs_floor.
    Returns (ok, worst ratio of error to bound)."""
    y_test = np.asarray(y_test, dtype=np.float64)
    err = np.abs(y_test - y_ref)
    bound = rel * mag + abs_floor
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(np.all(err <= bound)), worst


__all__ = ["Oracle", "get", "load", "within_tolerance", "OK", "BAD_ARG", "BAD_ROWPTRS",
           "COL_RANGE", "FORMAT_NAMES"]
