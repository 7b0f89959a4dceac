"""GPU parity with 8-byte values ('Introduction to sparse computing and
performance bottleneck location', section 'Building the problem framework':
values of 4 or 8 bytes) through the C ABI.

Converted arrays are compared bit for bit. The storage layouts do not depend
on the value width, so the oracle's layout conversions (pinned with 4-byte
values) are run with value = k + 1 for nonzero k (exact in float32 below
2^24): every slot then names its source nonzero, and the expected 8-byte
array is value64[source] (+0.0 for padding).

SpMV: per row |y_gpu - y_ref| <= (len + 2) * 2^-52 * (sum_j |a_ij x_j| +
|y0_i|), y_ref from the oracle's compensated fp64 sum (within one rounding
of exact): a sum of len + 1 fp64 terms in any order is within
len * 2^-53 * (sum of magnitudes) of exact, each product within 2^-53 of its
magnitude, and the factor 2 covers both roundings of y_ref and the first
order bound.
"""
import numpy as np
import pytest
import torch

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


def values64(inp, seed):
    """8-byte values that a 4-byte path would round: mantissas of 52 bits,
    exponents over a wide range."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(inp.nnz) * np.exp2(rng.integers(-30, 30, inp.nnz))


def fits(inp, f):
    R, C, Z = inp.num_rows, inp.num_cols, inp.nnz
    lens = np.diff(inp.row_ptrs.astype(np.int64))
    mx = int(lens.max()) if R else 0
    if f == "ELL":
        return R * mx <= min(2**31 - 1, 4 * Z + R)
    if f == "SELL":
        srt = np.sort(lens)[::-1]
        slots = sum(min(128, R - k) * int(srt[k]) for k in range(0, R, 128))
        return slots <= min(2**31 - 1, 4 * Z + R)
    return True


def source_map(orc, inp, f, K=None):
    """Layout arrays from the oracle with value = k + 1: returns dict of the
    index arrays and `src` (source nonzero of each value slot, -1 padding).
    K: the HYB width the library chose."""
    rp, ci = inp.row_ptrs, inp.col_idx
    tag = (np.arange(inp.nnz) + 1).astype(np.float32)
    assert inp.nnz < 2**24
    if f == "COO":
        o = orc.csr_to_coo(rp, ci, tag)
    elif f == "ELL":
        o = orc.csr_to_ell(rp, ci, tag)
    elif f == "HYB":
        o = orc.csr_to_hyb(rp, ci, tag, K)
        o["coo_src"] = o["coo_value"].astype(np.int64) - 1
    elif f == "JDS":
        o = orc.csr_to_jds(rp, ci, tag)
    elif f == "SELL":
        o = orc.csr_to_sell(rp, ci, tag, 128)
    elif f == "XBLOCK":
        o = orc.csr_to_xblock(rp, ci, tag, inp.num_cols, 24576)
    o["src"] = o["value"].astype(np.int64) - 1
    return o


def expect(v64, src):
    out = np.zeros(src.shape[0], np.float64)
    m = src >= 0
    out[m] = v64[src[m]]
    return out


def same64(a, b):
    return a.shape == b.shape and np.array_equal(np.asarray(a, np.float64).view(np.int64),
                                                 np.asarray(b, np.float64).view(np.int64))


def check_f64(sp, orc, inp, seed=0, formats=FORMATS, arrays=True):
    v64 = values64(inp, seed)
    rng = np.random.default_rng(seed + 1)
    x = rng.standard_normal(inp.num_cols)
    y0 = rng.standard_normal(inp.num_rows)
    yref, mag = orc.spmv_csr_f64(inp.row_ptrs, inp.col_idx, v64, x, y0)
    lens = np.diff(inp.row_ptrs.astype(np.int64))
    bound = (lens + 2) * 2.0**-52 * mag + 1e-300
    worst = {}
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(v64)) as m:
        assert m.f64
        for f in formats:
            if not fits(inp, f):
                with pytest.raises(sp.SpmvError) as ei:
                    m.convert(f)
                assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
                continue
            m.convert(f)
            if arrays and f != "CSR":
                got = m.export(f)
                want = source_map(orc, inp, f, got["width"])
                assert same64(got["value"], expect(v64, want["src"])), f
                if f == "HYB":
                    assert same64(got["coo_value"], expect(v64, want["coo_src"]))
                    assert np.array_equal(got["coo_col_idx"], want["coo_col_idx"])
                if f == "XBLOCK":
                    assert np.array_equal(got["col16"], want["col16"])
                    assert np.array_equal(got["row_idx"], want["row_idx"])
                elif f == "COO":
                    assert np.array_equal(got["row_idx"], want["row_idx"])
                else:
                    assert np.array_equal(got["col_idx"], want["col_idx"]), f
            y = dev(y0)
            m.run(f, dev(x), y)
            torch.cuda.synchronize()
            err = np.abs(y.cpu().numpy() - yref)
            ratio = float((err / bound).max()) if err.size else 0.0
            assert ratio <= 1.0, (inp.name, f, ratio)
            worst[f] = ratio
    return worst


def test_fig14_1(sp, orc):
    rp, ci, va = orc.dense_to_csr(synth.fig14_1_dense())
    with sp.SparseMatrix(4, 4, dev(rp), dev(ci), dev(va.astype(np.float64))) as m:
        for f in FORMATS:
            if f != "CSR":
                m.convert(f, ell_width=2, section_rows=2, chunk_cols=2)
            y = torch.zeros(4, dtype=torch.float64, device="cuda")
            m.run(f, dev(np.array([1.0, 2, 3, 4])), y)
            assert y.cpu().tolist() == [15.0, 50.0, 28.0, 24.0], f
        ell = m.export("ELL")
        assert ell["value"].dtype == np.float64
        assert ell["value"].tolist() == [1, 5, 2, 6, 7, 3, 8, 0, 0, 9, 0, 0]


EDGE = {
    "empty_rows": dict(num_rows=3001, num_cols=2000, mean_len=5, empty_frac=0.3),
    "few_long_rows": dict(num_rows=5003, num_cols=60_000, mean_len=7, long_rows=5,
                          long_len=50_000),
    "unsorted_dups": dict(num_rows=2048, num_cols=4096, mean_len=9, unsorted=True),
    "rows_not_mult4": dict(num_rows=1003, num_cols=1003, mean_len=4),
    "wide_short": dict(num_rows=3, num_cols=100_000, mean_len=4000),
    "len_beyond_exact_hist": dict(num_rows=60, num_cols=20_000, mean_len=5000),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(sp, orc, name):
    inp = synth.random_csr(13, name=name, **EDGE[name])
    check_f64(sp, orc, inp, seed=len(name))


def test_needs_eight_bytes(sp, orc):
    """1 + 2^-40 per entry: a 4-byte path would lose the 2^-40 terms."""
    n = 4096
    rp = np.arange(0, 2 * n + 1, 2, dtype=np.int32)
    ci = (np.arange(2 * n, dtype=np.int32) * 7) % n
    v = np.full(2 * n, 1 + 2.0**-40)
    with sp.SparseMatrix(n, n, dev(rp), dev(ci), dev(v)) as m:
        for f in FORMATS:
            if f != "CSR":
                m.convert(f)
            y = torch.zeros(n, dtype=torch.float64, device="cuda")
            m.run(f, torch.ones(n, dtype=torch.float64, device="cuda"), y)
            assert (y.cpu().numpy() == 2 + 2.0**-39).all(), f


def test_full_size_laplace2d(sp, orc):
    inp = synth.make_workload("laplace2d")
    worst = check_f64(sp, orc, inp, formats=("CSR", "ELL", "SELL"), arrays=False)
    print(worst)


def test_type_errors(sp, orc):
    inp = synth.random_csr(3, 100, 100, mean_len=4)
    with sp.SparseMatrix(100, 100, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value.astype(np.float64))) as m:
        with pytest.raises(sp.SpmvError) as ei:  # 4-byte run on an 8-byte handle
            sp.spmv_run(m.handle, "CSR", dev(inp.x), dev(inp.y0))
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        with pytest.raises(sp.SpmvError) as ei:
            m.cg_solve("CSR", dev(inp.y0), dev(inp.x))
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        with pytest.raises(sp.SpmvError) as ei:
            m.convert("XBLOCK", chunk_cols=24577)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        m.convert("XBLOCK", chunk_cols=24576)
    with sp.SparseMatrix(100, 100, dev(inp.row_ptrs), dev(inp.col_idx), dev(inp.value)) as m:
        with pytest.raises(sp.SpmvError) as ei:  # 8-byte run on a 4-byte handle
            sp.spmv_run_f64(m.handle, "CSR", dev(inp.x.astype(np.float64)),
                            dev(inp.y0.astype(np.float64)))
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG


def test_warp_staged_width_24(sp, orc):
    """8-byte values with rows of 12-24 entries: the ELL, HYB (automatic
    width), JDS and SELL conversions take the warp-staged scatters (two
    16-byte copies per 4 values)."""
    rng = np.random.default_rng(77)
    R, C = 3001, 2500
    lens = rng.integers(12, 25, R).astype(np.int64)
    lens[0] = 24
    cols = synth._distinct_sorted_columns(rng, lens, C)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    val = rng.uniform(-1.0, 1.0, cols.size).astype(np.float32)
    inp = synth.CSRInput("wide24", R, C, rp, cols, val, np.zeros(C, np.float32),
                         np.zeros(R, np.float32))
    check_f64(sp, orc, inp, formats=("ELL", "HYB", "JDS", "SELL"))
