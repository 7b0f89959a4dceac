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


def chunk_edge_matrix():
    """A matrix whose empty rows sit exactly at 128-entry chunk starts and
    inside chunks, with rows that end on a chunk boundary and rows longer
    than a chunk."""
    rng = np.random.default_rng(21)
    lens = [128, 0, 0, 127, 1, 0, 128, 0, 300, 0, 0, 0, 5, 123, 0, 0]
    lens += list(rng.choice([0, 0, 1, 3, 64, 127, 128, 129], size=4000))
    lens = np.array(lens, np.int64)
    R, C = lens.size, 3000
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Z = int(rp[-1])
    ci = rng.integers(0, C, size=Z).astype(np.int32)
    va = rng.uniform(-1, 1, size=Z).astype(np.float32)
    x = rng.uniform(-1, 1, size=C).astype(np.float32)
    y0 = rng.uniform(-1, 1, size=R).astype(np.float32)
    return synth.CSRInput("chunk_edges", R, C, rp, ci, va, x, y0)


def test_noalloc_smaller_matrix_after_larger(sp, orc):
    """A call on a smaller, irregular matrix issued right after one on the
    largest matrix, on the same stream with no synchronisation between them,
    must not see the first call's records; each call launches 3 kernels."""
    big = CASES["at_limit"]()
    small = chunk_edge_matrix()
    assert small.nnz < big.nnz
    rows_at_chunk_start = np.isin(small.row_ptrs[:-1], np.arange(0, small.nnz, 128)) & (
        np.diff(small.row_ptrs) == 0)
    assert rows_at_chunk_start.any()  # the case this test is about
    db = [dev(a) for a in (big.row_ptrs, big.col_idx, big.value, big.x)]
    ds = [dev(a) for a in (small.row_ptrs, small.col_idx, small.value, small.x)]
    yb, ys = dev(big.y0), dev(small.y0)
    torch.cuda.synchronize()
    n0 = sp.spmv_launch_count()
    sp.spmv_run_csr_noalloc(big.num_rows, big.num_cols, big.nnz, *db, yb)
    n1 = sp.spmv_launch_count()
    sp.spmv_run_csr_noalloc(small.num_rows, small.num_cols, small.nnz, *ds, ys)
    n2 = sp.spmv_launch_count()
    torch.cuda.synchronize()
    assert n1 - n0 == 3 and n2 - n1 == 3
    for inp, y in ((big, yb), (small, ys)):
        want, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
        ok, worst = oracle.within_tolerance(y.cpu().numpy(), want, mag)
        assert ok, (inp.name, worst)
