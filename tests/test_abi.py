"""The C ABI library loads and exports every function include/spmv.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


def header_functions():
    src = open(os.path.join(ROOT, "include", "spmv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spmv_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def sp():
    from conftest import build_library
    build_library()
    import spmv_sparse_storage_gb300 as sp
    return sp


def test_header_lists_the_boundary():
    fns = header_functions()
    for name in ["spmv_create_csr", "spmv_convert_coo", "spmv_convert_ell", "spmv_convert_hyb",
                 "spmv_convert_jds", "spmv_convert_sell", "spmv_run", "spmv_select", "spmv_get_stats",
                 "spmv_export", "spmv_destroy", "spmv_status_string"]:
        assert name in fns


def test_library_exports_every_declared_symbol(sp):
    lib = ctypes.CDLL(sp.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in spmv.h but not exported"


def test_binding_has_same_names(sp):
    for name in header_functions():
        assert callable(getattr(sp, name)), name


def test_status_strings(sp):
    for code in range(-8, 1):
        assert sp.spmv_status_string(code) not in ("", "unknown status")
    assert sp.spmv_status_string(5) == "unknown status"


def test_host_argument_checks_without_gpu(sp):
    lib = sp._lib
    h = ctypes.c_void_p()
    # null out-pointer, negative sizes, null arrays: rejected before any CUDA call
    assert lib.spmv_create_csr(None, 1, 1, 0, None, None, None, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_create_csr(ctypes.byref(h), -1, 1, 0, 8, None, None, None) == \
        sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_create_csr(ctypes.byref(h), 1, 1, 0, None, None, None, None) == \
        sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_create_csr(ctypes.byref(h), 1, 1, 3, 8, None, None, None) == \
        sp.SPMV_ERR_INVALID_ARG
    assert h.value is None
    for fn in ("spmv_convert_coo", "spmv_convert_ell", "spmv_convert_jds"):
        assert getattr(lib, fn)(None, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_convert_hyb(None, 0, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_convert_sell(None, 0, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_run(None, 0, None, None, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_select(None, None, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_get_stats(None, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_export(None, 0, None) == sp.SPMV_ERR_INVALID_ARG
    assert lib.spmv_destroy(None) == sp.SPMV_OK


def test_misc_calls(sp):
    assert sp.spmv_version() >= 10000
    assert sp.spmv_launch_count() >= 0
    sp.spmv_set_memory_limit(1 << 20)
    sp.spmv_set_memory_limit(None)
    assert sp.spmv_last_cuda_error() >= 0


def test_binding_rejects_host_tensors(sp):
    import torch
    with pytest.raises(ValueError):
        sp.spmv_create_csr(1, 1, 0, torch.zeros(2, dtype=torch.int32), None, None, stream=0)


def test_product_does_not_import_oracle():
    """The product package never imports or reads the test oracle."""
    pkg = os.path.join(ROOT, "spmv_sparse_storage_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"


def test_oracle_does_not_import_product():
    d = os.path.join(ROOT, "oracle")
    for f in os.listdir(d):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(d, f)).read()
            assert "spmv_sparse_storage_gb300" not in text
            assert "spmv.h" not in text
