"""Python binding of the GB300 SpMV library (``include/spmv.h``).

Argument marshalling only: every function here calls the C function of the
same name in ``_lib/libspmv_gb300.so`` and raises :class:`SpmvError` on a
non-OK status. Arrays are passed as torch CUDA tensors (or raw integer device
pointers); PyTorch serves only for device memory and streams. There is no
fallback: importing this package fails when the compiled library is absent.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libspmv_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing; build it with "
        "`python spmv_sparse_storage_gb300/_build.py`")

_lib = C.CDLL(LIB_PATH)

# --- enums -----------------------------------------------------------------
SPMV_COO, SPMV_CSR, SPMV_ELL, SPMV_HYB, SPMV_JDS, SPMV_AUTO, SPMV_SELL, SPMV_XBLOCK = range(8)
FORMATS = {"COO": SPMV_COO, "CSR": SPMV_CSR, "ELL": SPMV_ELL, "HYB": SPMV_HYB,
           "JDS": SPMV_JDS, "AUTO": SPMV_AUTO, "SELL": SPMV_SELL, "XBLOCK": SPMV_XBLOCK}
FORMAT_NAMES = {v: k for k, v in FORMATS.items()}

SPMV_OK = 0
SPMV_ERR_INVALID_ARG = -1
SPMV_ERR_BAD_ROWPTRS = -2
SPMV_ERR_COL_OUT_OF_RANGE = -3
SPMV_ERR_TOO_LARGE = -4
SPMV_ERR_NOT_CONVERTED = -5
SPMV_ERR_CUDA = -6
SPMV_ERR_ALLOC = -7
SPMV_ERR_TIMEOUT = -8


class spmv_stats(C.Structure):
    _fields_ = [("num_rows", C.c_int64), ("num_cols", C.c_int64), ("nnz", C.c_int64),
                ("max_len", C.c_int64), ("min_len", C.c_int64), ("empty_rows", C.c_int64),
                ("sum_sq_len", C.c_int64), ("mean_len", C.c_double), ("var_len", C.c_double),
                ("hist_log2", C.c_int64 * 33), ("imbalance_thread", C.c_double),
                ("imbalance_warp", C.c_double), ("auto_format", C.c_int32),
                ("auto_hyb_width", C.c_int32), ("gather_lines", C.c_double)]


class spmv_arrays(C.Structure):
    _fields_ = [("format", C.c_int32), ("num_rows", C.c_int64), ("num_cols", C.c_int64),
                ("nnz", C.c_int64), ("width", C.c_int32), ("ell_slots", C.c_int64),
                ("coo_nnz", C.c_int64), ("row_ptrs", C.c_void_p), ("row_idx", C.c_void_p),
                ("col_idx", C.c_void_p), ("value", C.c_void_p), ("nnz_per_row", C.c_void_p),
                ("coo_col_idx", C.c_void_p), ("coo_value", C.c_void_p), ("perm", C.c_void_p),
                ("iter_ptr", C.c_void_p), ("sec_ptr", C.c_void_p),
                ("section_rows", C.c_int32), ("chunk_ptr", C.c_void_p), ("col16", C.c_void_p),
                ("chunk_cols", C.c_int32), ("num_chunks", C.c_int32),
                ("value_bytes", C.c_int32), ("value_f64", C.c_void_p),
                ("coo_value_f64", C.c_void_p)]


class spmv_cg_info(C.Structure):
    _fields_ = [("iterations", C.c_int32), ("status", C.c_int32),
                ("residual_norm", C.c_double), ("y_norm", C.c_double)]


_H = C.c_void_p
_P = C.c_void_p
_SIGS = {
    "spmv_create_csr": (C.c_int, [C.POINTER(_H), C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P]),
    "spmv_create_csr_f64": (C.c_int, [C.POINTER(_H), C.c_int32, C.c_int32, C.c_int32, _P, _P, _P,
                                      _P]),
    "spmv_convert_coo": (C.c_int, [_H, _P]),
    "spmv_convert_ell": (C.c_int, [_H, _P]),
    "spmv_convert_hyb": (C.c_int, [_H, C.c_int32, _P]),
    "spmv_convert_jds": (C.c_int, [_H, _P]),
    "spmv_convert_sell": (C.c_int, [_H, C.c_int32, _P]),
    "spmv_convert_xblock": (C.c_int, [_H, C.c_int32, _P]),
    "spmv_run": (C.c_int, [_H, C.c_int, _P, _P, _P]),
    "spmv_run_f64": (C.c_int, [_H, C.c_int, _P, _P, _P]),
    "spmv_cg_solve": (C.c_int, [_H, C.c_int, _P, _P, C.c_int32, C.c_double,
                                C.POINTER(spmv_cg_info), _P]),
    "spmv_select": (C.c_int, [_H, C.POINTER(C.c_int), C.POINTER(C.c_int32)]),
    "spmv_autotune": (C.c_int, [_H, _P, _P, C.c_int32, C.POINTER(C.c_int),
                                C.POINTER(C.c_float), _P]),
    "spmv_get_stats": (C.c_int, [_H, C.POINTER(spmv_stats)]),
    "spmv_export": (C.c_int, [_H, C.c_int, C.POINTER(spmv_arrays)]),
    "spmv_destroy": (C.c_int, [_H]),
    "spmv_run_csr_noalloc": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P]),
    "spmv_status_string": (C.c_char_p, [C.c_int]),
    "spmv_last_cuda_error": (C.c_int, []),
    "spmv_launch_count": (C.c_uint64, []),
    "spmv_set_memory_limit": (C.c_int, [C.c_int64]),
    "spmv_version": (C.c_int, []),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class SpmvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.spmv_status_string(code).decode()
        if code == SPMV_ERR_CUDA:
            msg += f" (cudaError {_lib.spmv_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")


def _check(code: int, where: str):
    if code != SPMV_OK:
        raise SpmvError(code, where)


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, torch.Tensor):
        if not a.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if not a.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        return a.data_ptr() if a.numel() else None
    raise TypeError(f"expected a torch CUDA tensor or a device pointer, got {type(a)}")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _fmt(f):
    return FORMATS[f.upper()] if isinstance(f, str) else int(f)


# --- the C functions, same names ---------------------------------------------
def spmv_create_csr(num_rows, num_cols, nnz, row_ptrs, col_idx, value, stream=None):
    """Returns an opaque handle (int). See spmv.h for the contract."""
    h = _H()
    _check(_lib.spmv_create_csr(C.byref(h), num_rows, num_cols, nnz, _ptr(row_ptrs),
                                _ptr(col_idx), _ptr(value), _stream(stream)), "spmv_create_csr")
    return h.value


def spmv_create_csr_f64(num_rows, num_cols, nnz, row_ptrs, col_idx, value, stream=None):
    """As spmv_create_csr with float64 values (a torch.float64 tensor)."""
    h = _H()
    _check(_lib.spmv_create_csr_f64(C.byref(h), num_rows, num_cols, nnz, _ptr(row_ptrs),
                                    _ptr(col_idx), _ptr(value), _stream(stream)),
           "spmv_create_csr_f64")
    return h.value


def spmv_convert_coo(h, stream=None):
    _check(_lib.spmv_convert_coo(h, _stream(stream)), "spmv_convert_coo")


def spmv_convert_ell(h, stream=None):
    _check(_lib.spmv_convert_ell(h, _stream(stream)), "spmv_convert_ell")


def spmv_convert_hyb(h, ell_width=0, stream=None):
    _check(_lib.spmv_convert_hyb(h, ell_width, _stream(stream)), "spmv_convert_hyb")


def spmv_convert_jds(h, stream=None):
    _check(_lib.spmv_convert_jds(h, _stream(stream)), "spmv_convert_jds")


def spmv_convert_sell(h, section_rows=0, stream=None):
    _check(_lib.spmv_convert_sell(h, section_rows, _stream(stream)), "spmv_convert_sell")


def spmv_run_f64(h, fmt, x, y, stream=None):
    """y <- A x + y for a float64 handle (x, y float64)."""
    _check(_lib.spmv_run_f64(h, _fmt(fmt), _ptr(x), _ptr(y), _stream(stream)), "spmv_run_f64")


def spmv_convert_xblock(h, chunk_cols=0, stream=None):
    _check(_lib.spmv_convert_xblock(h, chunk_cols, _stream(stream)), "spmv_convert_xblock")


def spmv_run(h, fmt, x, y, stream=None):
    """y <- A x + y in the given format (name or code)."""
    _check(_lib.spmv_run(h, _fmt(fmt), _ptr(x), _ptr(y), _stream(stream)), "spmv_run")


def spmv_cg_solve(h, fmt, y, x, max_iter, tol, stream=None):
    """Solve A·X + Y = 0 by conjugate gradients; ``x`` holds the starting
    guess and receives the solution. Returns the spmv_cg_info fields."""
    info = spmv_cg_info()
    _check(_lib.spmv_cg_solve(h, _fmt(fmt), _ptr(y), _ptr(x), int(max_iter), float(tol),
                              C.byref(info), _stream(stream)), "spmv_cg_solve")
    return {name: getattr(info, name) for name, _ in spmv_cg_info._fields_}


def spmv_select(h):
    f = C.c_int()
    w = C.c_int32()
    _check(_lib.spmv_select(h, C.byref(f), C.byref(w)), "spmv_select")
    return FORMAT_NAMES[f.value], w.value


def spmv_autotune(h, x, y, reps=5, stream=None):
    """Time every converted format's SpMV (``y`` is scratch, overwritten) and
    make the fastest the handle's automatic choice. Returns (format name,
    {format name: median ms} for the timed formats)."""
    best = C.c_int()
    times = (C.c_float * 8)()
    _check(_lib.spmv_autotune(h, _ptr(x), _ptr(y), int(reps), C.byref(best), times,
                              _stream(stream)), "spmv_autotune")
    timed = {FORMAT_NAMES[f]: float(times[f]) for f in range(8)
             if f in FORMAT_NAMES and times[f] >= 0.0}
    return FORMAT_NAMES[best.value], timed


def spmv_get_stats(h):
    s = spmv_stats()
    _check(_lib.spmv_get_stats(h, C.byref(s)), "spmv_get_stats")
    d = {name: getattr(s, name) for name, _ in spmv_stats._fields_}
    d["hist_log2"] = list(s.hist_log2)
    d["auto_format"] = FORMAT_NAMES[s.auto_format]
    return d


def spmv_export(h, fmt):
    """Raw view of a converted format: dict of sizes and device pointers."""
    a = spmv_arrays()
    _check(_lib.spmv_export(h, _fmt(fmt), C.byref(a)), "spmv_export")
    return {name: getattr(a, name) for name, _ in spmv_arrays._fields_}


def spmv_destroy(h):
    _check(_lib.spmv_destroy(h), "spmv_destroy")


def spmv_run_csr_noalloc(num_rows, num_cols, nnz, row_ptrs, col_idx, value, x, y,
                         stream=None):
    """y <- A x + y from CSR arrays without a handle or any allocation (see
    spmv.h: nnz <= 4,194,304; first call on a device before stream capture;
    calls that overlap on the GPU race)."""
    _check(_lib.spmv_run_csr_noalloc(num_rows, num_cols, nnz, _ptr(row_ptrs), _ptr(col_idx),
                                     _ptr(value), _ptr(x), _ptr(y), _stream(stream)),
           "spmv_run_csr_noalloc")


def spmv_status_string(code):
    return _lib.spmv_status_string(code).decode()


def spmv_last_cuda_error():
    return _lib.spmv_last_cuda_error()


def spmv_launch_count():
    return _lib.spmv_launch_count()


def spmv_set_memory_limit(nbytes):
    _check(_lib.spmv_set_memory_limit(-1 if nbytes is None else int(nbytes)),
           "spmv_set_memory_limit")


def spmv_version():
    return _lib.spmv_version()


# --- conveniences built only from the calls above ------------------------------
class _DeviceView:
    """Zero-copy torch view of a device array owned by the library."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (int(n),), "typestr": typestr,
                                         "data": (int(ptr or 0), False), "version": 3}


def device_view(ptr, n, dtype):
    """torch tensor aliasing ``n`` elements at device pointer ``ptr`` (no copy;
    valid while the owning handle and format live)."""
    if n == 0 or not ptr:
        return torch.empty(0, dtype=dtype, device="cuda")
    typestr = {torch.int32: "<i4", torch.float32: "<f4", torch.int16: "<i2",
               torch.float64: "<f8"}[dtype]
    return torch.as_tensor(_DeviceView(ptr, n, typestr), device="cuda")


def export_tensors(h, fmt):
    """Copies (host numpy arrays) of a converted format's arrays, for checks."""
    a = spmv_export(h, fmt)
    R, Z = a["num_rows"], a["nnz"]
    i32, f32 = torch.int32, torch.float32

    def get(ptr, n, dt):
        return device_view(ptr, n, dt).cpu().numpy().copy()

    f = FORMAT_NAMES[a["format"]]
    out = {"format": f, "num_rows": R, "nnz": Z, "width": a["width"]}
    if a["value_bytes"] == 8:  # 8-byte values: read the f64 fields under the usual names
        f32 = torch.float64
        a["value"], a["coo_value"] = a["value_f64"], a["coo_value_f64"]
    if f == "CSR":
        out.update(row_ptrs=get(a["row_ptrs"], R + 1, i32), col_idx=get(a["col_idx"], Z, i32),
                   value=get(a["value"], Z, f32))
    elif f == "COO":
        out.update(row_idx=get(a["row_idx"], Z, i32), col_idx=get(a["col_idx"], Z, i32),
                   value=get(a["value"], Z, f32))
    elif f in ("ELL", "HYB"):
        S = a["ell_slots"]
        out.update(col_idx=get(a["col_idx"], S, i32), value=get(a["value"], S, f32),
                   nnz_per_row=get(a["nnz_per_row"], R, i32))
        if f == "HYB":
            n = a["coo_nnz"]
            out.update(coo_row_idx=get(a["row_idx"], n, i32),
                       coo_col_idx=get(a["coo_col_idx"], n, i32),
                       coo_value=get(a["coo_value"], n, f32))
    elif f == "JDS":
        out.update(perm=get(a["perm"], R, i32), iter_ptr=get(a["iter_ptr"], a["width"] + 1, i32),
                   col_idx=get(a["col_idx"], Z, i32), value=get(a["value"], Z, f32))
    elif f == "XBLOCK":
        n, nch = a["ell_slots"], a["num_chunks"]
        out.update(chunk_cols=a["chunk_cols"], num_chunks=nch,
                   chunk_ptr=get(a["chunk_ptr"], nch + 1, i32),
                   row_idx=get(a["row_idx"], n, i32),
                   col16=get(a["col16"], n, torch.int16).view("u2"),
                   value=get(a["value"], n, f32))
    elif f == "SELL":
        S, n = a["section_rows"], a["ell_slots"]
        out.update(section_rows=S, perm=get(a["perm"], R, i32),
                   sec_ptr=get(a["sec_ptr"], (R + S - 1) // S + 1, i32),
                   col_idx=get(a["col_idx"], n, i32), value=get(a["value"], n, f32))
    return out


class SparseMatrix:
    """Owns a handle and keeps the borrowed CSR tensors alive until close().
    A float64 ``value`` tensor makes an 8-byte handle (run on float64 x, y)."""

    def __init__(self, num_rows, num_cols, row_ptrs, col_idx, value, stream=None):
        self._keep = (row_ptrs, col_idx, value)
        self.num_rows, self.num_cols = int(num_rows), int(num_cols)
        self.nnz = int(col_idx.numel())
        self.f64 = isinstance(value, torch.Tensor) and value.dtype == torch.float64
        create = spmv_create_csr_f64 if self.f64 else spmv_create_csr
        self.handle = create(self.num_rows, self.num_cols, self.nnz, row_ptrs, col_idx, value,
                             stream)

    def convert(self, fmt, ell_width=0, stream=None, section_rows=0, chunk_cols=0):
        f = FORMAT_NAMES[_fmt(fmt)]
        if f == "COO":
            spmv_convert_coo(self.handle, stream)
        elif f == "ELL":
            spmv_convert_ell(self.handle, stream)
        elif f == "HYB":
            spmv_convert_hyb(self.handle, ell_width, stream)
        elif f == "JDS":
            spmv_convert_jds(self.handle, stream)
        elif f == "SELL":
            spmv_convert_sell(self.handle, section_rows, stream)
        elif f == "XBLOCK":
            spmv_convert_xblock(self.handle, chunk_cols, stream)
        elif f != "CSR":
            raise ValueError(f"cannot convert to {f}")

    def run(self, fmt, x, y, stream=None):
        (spmv_run_f64 if self.f64 else spmv_run)(self.handle, fmt, x, y, stream)

    def cg_solve(self, fmt, y, x, max_iter=1000, tol=1e-6, stream=None):
        return spmv_cg_solve(self.handle, fmt, y, x, max_iter, tol, stream)

    def select(self):
        return spmv_select(self.handle)

    def autotune(self, x, y, reps=5, stream=None):
        return spmv_autotune(self.handle, x, y, reps, stream)

    def stats(self):
        return spmv_get_stats(self.handle)

    def export(self, fmt):
        return export_tensors(self.handle, fmt)

    def close(self):
        if self.handle:
            spmv_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


__all__ = [n for n in list(globals()) if n.startswith("spmv_") or n.startswith("SPMV_")] + [
    "SpmvError", "SparseMatrix", "export_tensors", "device_view", "FORMATS", "FORMAT_NAMES",
    "LIB_PATH"]
