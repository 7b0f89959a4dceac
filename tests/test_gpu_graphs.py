"""The SpMV calls are stream-ordered, allocate nothing and never synchronise,
so they can be captured into a CUDA graph and replayed: y <- A x + y for
every format, captured once and replayed three times, gives y0 + 3 A x
within three times the parity tolerance. Conversions allocate (from the
library's stream-ordered pool) and are run before capture."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

FORMATS = ("CSR", "COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK")


@pytest.fixture(scope="module")
def sp():
    from conftest import build_library
    build_library()
    import spmv_sparse_storage_gb300 as sp
    torch.cuda.set_device(0)
    return sp


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("name", ["irregular", "laplace"])
def test_spmv_replays_from_a_cuda_graph(sp, orc, name):
    inp = (synth.random_csr(61, 20_000, 18_000, mean_len=7, empty_frac=0.1, long_rows=4,
                            long_len=25, name=name)
           if name == "irregular" else synth.laplace2d(300))
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    ax = yref - inp.y0.astype(np.float64)
    x = dev(inp.x)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        for f in FORMATS[1:]:
            m.convert(f)
        for f in FORMATS:
            y = dev(inp.y0)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # first launch of each kernel outside capture
                m.run(f, x, y)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            y.copy_(dev(inp.y0))
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                m.run(f, x, y)
            torch.cuda.synchronize()
            assert np.array_equal(y.cpu().numpy(), inp.y0), f  # capture does not run
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            ok, worst = oracle.within_tolerance(y.cpu().numpy(), inp.y0 + 3 * ax, 3 * mag)
            assert ok, (name, f, worst)
