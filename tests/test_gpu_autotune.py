"""spmv_autotune: the format chosen by timing (the format-selection page,
end of section 4.3: run every format on the matrix and keep the fastest)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


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


def test_autotune_times_the_converted_formats_and_sets_auto(sp, orc):
    inp = synth.laplace2d(300)
    R = inp.num_rows
    with sp.SparseMatrix(R, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        for f in ("COO", "ELL", "JDS"):
            m.convert(f)
        x = dev(inp.x)
        scratch = torch.empty(R, dtype=torch.float32, device="cuda")
        best, times = m.autotune(x, scratch, reps=3)
        assert set(times) == {"CSR", "COO", "ELL", "JDS"}  # every converted format, no other
        assert all(t > 0 for t in times.values())
        assert best == min(times, key=times.get)
        assert m.select()[0] == best
        assert m.stats()["auto_format"] == best
        # SPMV_AUTO now runs the timed choice
        y = dev(inp.y0)
        m.run("AUTO", x, y)
        torch.cuda.synchronize()
        want, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
        ok, worst = oracle.within_tolerance(y.cpu().numpy(), want, mag)
        assert ok, worst
        # more formats converted later: a second call times them too
        m.convert("HYB")
        best2, times2 = m.autotune(x, scratch, reps=2)
        assert set(times2) == {"CSR", "COO", "ELL", "JDS", "HYB"}
        assert best2 == min(times2, key=times2.get) == m.select()[0]


def test_autotune_rejects_bad_arguments(sp):
    inp = synth.random_csr(3, 200, 150, mean_len=5)
    x = dev(inp.x)
    y = torch.empty(inp.num_rows, dtype=torch.float32, device="cuda")
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        for reps in (0, 1001):
            with pytest.raises(sp.SpmvError) as ei:
                m.autotune(x, y, reps=reps)
            assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        with pytest.raises(sp.SpmvError) as ei:  # x and y overlap
            m.autotune(y, y, reps=1)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value.astype(np.float64))) as m64:
        with pytest.raises(sp.SpmvError) as ei:  # 8-byte handles are not timed
            m64.autotune(x, y, reps=1)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
