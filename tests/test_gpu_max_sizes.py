"""Near the int32 index limits: nnz = 2,147,483,639 (126,322,567 rows of 17
entries, 2^31 - 9), ~17 GB of CSR. Every offset computation of the library
that would overflow 32 bits shows up here. Checked on sampled rows (the first
and last rows, and random ones) against the oracle, whose row sample is
rebuilt from the closed-form generator; XBLOCK must refuse (its padding
pushes the slot count past int32)."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

PER_ROW = 17
R = (2**31 - 1) // PER_ROW          # 126,322,567
Z = R * PER_ROW                     # 2,147,483,639
C = R


@pytest.fixture(scope="module")
def sp():
    from conftest import build_library
    build_library()
    import spmv_sparse_storage_gb300 as sp
    torch.cuda.set_device(0)
    return sp


@pytest.fixture(scope="module")
def big():
    rp = torch.arange(0, Z + 1, PER_ROW, dtype=torch.int64).to(torch.int32).cuda()
    ci = torch.empty(Z, dtype=torch.int32, device="cuda")
    va = torch.empty(Z, dtype=torch.float32, device="cuda")
    step = 1 << 27
    for k0 in range(0, Z, step):
        k1 = min(Z, k0 + step)
        col, val = synth.hashed_entries(k0, k1, C)
        ci[k0:k1].copy_(torch.from_numpy(col))
        va[k0:k1].copy_(torch.from_numpy(val))
    x = torch.from_numpy(synth.hashed_vector(C, 11)).cuda()
    y0 = synth.hashed_vector(R, 29)
    return rp, ci, va, x, y0


def sample_rows():
    rng = np.random.default_rng(5)
    return np.unique(np.concatenate([[0, 1, R // 2, R - 2, R - 1],
                                     rng.integers(0, R, 3000)])).astype(np.int64)


def check_rows(orc, y_gpu, x, y0, rows):
    # the sampled rows as a small CSR over all columns
    rp = np.arange(0, (rows.size + 1) * PER_ROW, PER_ROW, dtype=np.int32)
    cols, vals = [], []
    for r in rows:
        c, v = synth.hashed_entries(int(r) * PER_ROW, int(r) * PER_ROW + PER_ROW, C)
        cols.append(c)
        vals.append(v)
    want, mag = orc.spmv_csr(rp, np.concatenate(cols), np.concatenate(vals), x, y0[rows])
    got = y_gpu[rows].astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-5 * mag + 1e-30)


def test_nnz_just_below_int32(sp, orc, big):
    rp, ci, va, x, y0 = big
    rows = sample_rows()
    xh = x.cpu().numpy()
    with sp.SparseMatrix(R, C, rp, ci, va) as m:
        st = m.stats()
        assert st["nnz"] == Z and st["max_len"] == PER_ROW and st["min_len"] == PER_ROW
        assert st["auto_format"] == "ELL"
        for f in ("CSR", "COO", "ELL", "HYB", "JDS", "SELL"):
            if f != "CSR":
                m.convert(f)
            y = torch.from_numpy(y0).cuda()
            m.run(f, x, y)
            torch.cuda.synchronize()
            check_rows(orc, y.cpu().numpy(), xh, y0, rows)
        with pytest.raises(sp.SpmvError) as ei:
            m.convert("XBLOCK", chunk_cols=64)  # ~2M chunks: more than 65536
        assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
        with pytest.raises(sp.SpmvError) as ei:
            m.convert("XBLOCK")  # 2,570 chunks: nnz + 3 * chunks > INT32_MAX
        assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
