"""spmv_run_csr_noalloc: the entry point for callers that cannot allocate
device memory (memory fully reserved by another allocator, loops whose rules
forbid allocation after start-up).
It keeps its per-chunk row index in a fixed device array instead of memory
it would allocate. Checked against the handle-based spmv_run(SPMV_CSR) on the
same inputs, within the parity tolerance, on two calls in a row. Collected
last so that a run stopping at the first failure has run everything else."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

MAX_NNZ = 4_194_304


@pytest.fixture(scope="module")
def sp():
    from conftest import build_library
    build_library()
    import spmv_sparse_storage_gb300 as sp
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    return sp


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


CASES = {
    "laplace": lambda: synth.laplace2d(700),                     # 2.45M nnz, banded
    "irregular": lambda: synth.random_csr(12, 50_000, 40_000, mean_len=9, empty_frac=0.2,
                                          long_rows=3, long_len=20_000),
    "at_limit": lambda: synth.uniform_rows("at_limit", MAX_NNZ // 8, 8),  # exactly the max
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_handle_path(sp, orc, name):
    inp = CASES[name]()
    assert inp.nnz <= MAX_NNZ
    rp, ci, va, x = dev(inp.row_ptrs), dev(inp.col_idx), dev(inp.value), dev(inp.x)
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, rp, ci, va) as m:
        y_handle = dev(inp.y0)
        m.run("CSR", x, y_handle)
    torch.cuda.synchronize()
    y_h = y_handle.cpu().numpy()
    for call in range(2):  # two calls in a row reuse the same scratch array
        y = dev(inp.y0)
        sp.spmv_run_csr_noalloc(inp.num_rows, inp.num_cols, inp.nnz, rp, ci, va, x, y)
        torch.cuda.synchronize()
        y_n = y.cpu().numpy()
        ok, worst = oracle.within_tolerance(y_n, y_h.astype(np.float64), 2 * mag)
        assert ok, (name, call, worst)
        ok, worst = oracle.within_tolerance(y_n, yref, mag)
        assert ok, (name, call, worst)


def test_noalloc_rejects_too_large(sp):
    lib = sp._lib
    st = lib.spmv_run_csr_noalloc(1, 1, MAX_NNZ + 1, ctypes.c_void_p(8), ctypes.c_void_p(8),
                                  ctypes.c_void_p(8), ctypes.c_void_p(8), ctypes.c_void_p(8),
                                  None)
    assert st == sp.SPMV_ERR_TOO_LARGE
