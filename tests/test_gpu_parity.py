"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Converters are compared bit for bit (exported device arrays vs the oracle's
conversion of the same CSR input). SpMV results must satisfy, per row,
|y_gpu - y_ref| <= 1e-5 * (sum_j |a_ij x_j| + |y0_i|) + 1e-30 with y_ref in
fp64: fp32 products summed in a different order (shuffle trees, shared and
global atomics) differ from a sequential sum by a few ulps of the magnitude
sum, far inside that bound for rows of up to several thousand entries.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

FORMATS = ("CSR", "COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK")


def xb_fits(C, Z, B):
    """The library's size rule for XBLOCK: at most 65536 chunks and
    nnz + 3 * chunks within int32."""
    nch = (C + B - 1) // B
    return nch <= 65536 and Z + 3 * nch <= 2**31 - 1


def sell_fits(row_ptrs, S):
    """The library's size rule for SELL: total slots (each section of S sorted
    rows padded to its longest row) within int32 and 4*nnz + numRows."""
    lens = np.sort(np.diff(np.asarray(row_ptrs, np.int64)))[::-1]
    R, Z = lens.size, int(lens.sum())
    slots = sum(min(S, R - k) * int(lens[k]) for k in range(0, R, S))
    return slots <= min(2**31 - 1, 4 * Z + R)


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


def same_bits(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    if a.dtype == np.float32:
        a, b = a.view(np.int32), np.asarray(b, np.float32).view(np.int32)
    return a.shape == b.shape and np.array_equal(a, b)


def check_tol(y, yref, mag, what):
    ok, worst = oracle.within_tolerance(y, yref, mag)
    assert ok, f"{what}: worst |err|/bound = {worst:.3g}"
    return worst


def check_matrix(sp, orc, inp, formats=FORMATS, hyb_widths=(0,), arrays=True, ell_ok=True,
                 offset=0, sell_rows=(0,), xb_chunks=(0,)):
    """Convert `inp` to every format on the GPU, compare the arrays with the
    oracle's conversions and the SpMV results with the oracle's y."""
    rp_t = dev(inp.row_ptrs)
    if offset:
        # misaligned views of rowPtrs/colIdx/value/y to exercise the scalar paths
        rp_buf = dev(np.concatenate([np.zeros(offset, np.int32), inp.row_ptrs]))
        rp_t = rp_buf[offset:]
        ci_buf = dev(np.concatenate([np.zeros(offset, np.int32), inp.col_idx]))
        va_buf = dev(np.concatenate([np.zeros(offset, np.float32), inp.value]))
        ci_t, va_t = ci_buf[offset:], va_buf[offset:]
    else:
        ci_t, va_t = dev(inp.col_idx), dev(inp.value)
    x_t = dev(inp.x)
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    R, Z = inp.num_rows, inp.nnz
    results = {}
    with sp.SparseMatrix(R, inp.num_cols, rp_t, ci_t, va_t) as m:
        st = m.stats()
        ost = orc.row_stats(inp.row_ptrs)
        assert st["max_len"] == ost["max_len"]
        assert st["hist_log2"] == ost["hist_log2"].tolist()
        assert st["mean_len"] == pytest.approx(ost["mean"], rel=1e-12, abs=1e-12)
        assert st["var_len"] == pytest.approx(ost["var"], rel=1e-9, abs=1e-9)
        assert st["auto_format"] == orc.select(R, inp.num_cols, Z, ost["max_len"],
                                               st["gather_lines"])
        # the other row statistics, by their definitions over the row lengths
        lens = np.diff(inp.row_ptrs.astype(np.int64))
        if R:
            assert st["min_len"] == int(lens.min())
            assert st["empty_rows"] == int((lens == 0).sum())
            assert st["sum_sq_len"] == int((lens * lens).sum())
            if Z:
                groups = np.add.reduceat(lens, np.arange(0, R, 32))  # 32 consecutive rows
                want = float(groups.max()) / (Z / ((R + 31) // 32))
                assert st["imbalance_warp"] == pytest.approx(want, rel=1e-12)
        if R and ost["max_len"] < 4096:
            assert st["auto_hyb_width"] == orc.hyb_auto_width(inp.row_ptrs)
        for f in formats:
            widths = (hyb_widths if f == "HYB" else sell_rows if f == "SELL" else
                      xb_chunks if f == "XBLOCK" else (None,))
            for w in widths:
                if f == "ELL" and not ell_ok:
                    with pytest.raises(sp.SpmvError) as ei:
                        m.convert("ELL")
                    assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
                    continue
                if f == "SELL" and not sell_fits(inp.row_ptrs, w or 128):
                    with pytest.raises(sp.SpmvError) as ei:
                        m.convert("SELL", section_rows=w)
                    assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
                    with pytest.raises(sp.SpmvError) as ei:
                        m.run("SELL", x_t, dev(inp.y0))
                    assert ei.value.code == sp.SPMV_ERR_NOT_CONVERTED
                    continue
                if f == "XBLOCK" and not xb_fits(inp.num_cols, Z, w or 49152):
                    with pytest.raises(sp.SpmvError) as ei:
                        m.convert("XBLOCK", chunk_cols=w)
                    assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
                    continue
                if f == "HYB":
                    m.convert(f, ell_width=w)
                elif f == "SELL":
                    m.convert(f, section_rows=w)
                elif f == "XBLOCK":
                    m.convert(f, chunk_cols=w)
                else:
                    m.convert(f)
                if arrays:
                    got = m.export(f)
                    compare_arrays(orc, inp, f, got, w, st)
                y_t = dev(inp.y0)
                m.run(f, x_t, y_t)
                torch.cuda.synchronize()
                key = f"{f}{w}" if f in ("HYB", "SELL", "XBLOCK") else f
                results[key] = check_tol(y_t.cpu().numpy(), yref, mag, f"{inp.name}/{key}")
        if st["auto_format"] in formats and (st["auto_format"] != "ELL" or ell_ok):
            y_t = dev(inp.y0)
            m.run("AUTO", x_t, y_t)
            torch.cuda.synchronize()
            check_tol(y_t.cpu().numpy(), yref, mag, f"{inp.name}/AUTO")
    return results


def compare_arrays(orc, inp, f, got, w, st):
    rp, ci, va = inp.row_ptrs, inp.col_idx, inp.value
    if f == "CSR":
        assert same_bits(got["row_ptrs"], rp) and same_bits(got["col_idx"], ci)
    elif f == "COO":
        want = orc.csr_to_coo(rp, ci, va)
        assert same_bits(got["row_idx"], want["row_idx"])
        assert same_bits(got["col_idx"], want["col_idx"])
        assert same_bits(got["value"], want["value"])
    elif f == "ELL":
        want = orc.csr_to_ell(rp, ci, va)
        assert got["width"] == want["width"]
        assert same_bits(got["col_idx"], want["col_idx"])
        assert same_bits(got["value"], want["value"])
        assert same_bits(got["nnz_per_row"], want["nnz_per_row"])
    elif f == "HYB":
        K = w if w else st["auto_hyb_width"]
        K = min(K, st["max_len"])
        want = orc.csr_to_hyb(rp, ci, va, K)
        assert got["width"] == K
        assert same_bits(got["col_idx"], want["col_idx"])
        assert same_bits(got["value"], want["value"])
        assert same_bits(got["nnz_per_row"], want["nnz_per_row"])
        assert same_bits(got["coo_row_idx"], want["coo_row_idx"])
        assert same_bits(got["coo_col_idx"], want["coo_col_idx"])
        assert same_bits(got["coo_value"], want["coo_value"])
    elif f == "JDS":
        want = orc.csr_to_jds(rp, ci, va)
        assert got["width"] == want["max_len"]
        assert same_bits(got["perm"], want["perm"])
        assert same_bits(got["iter_ptr"], want["iter_ptr"])
        assert same_bits(got["col_idx"], want["col_idx"])
        assert same_bits(got["value"], want["value"])
    elif f == "SELL":
        S = w or 128
        want = orc.csr_to_sell(rp, ci, va, S)
        assert got["section_rows"] == S
        assert same_bits(got["perm"], want["perm"])
        assert np.array_equal(got["sec_ptr"].astype(np.int64), want["sec_ptr"])
        assert same_bits(got["col_idx"], want["col_idx"])
        assert same_bits(got["value"], want["value"])
        lens = np.diff(rp)
        assert got["width"] == (int(lens.max()) if lens.size else 0)
    elif f == "XBLOCK":
        B = w or 49152
        want = orc.csr_to_xblock(rp, ci, va, inp.num_cols, B)
        assert got["chunk_cols"] == B and got["num_chunks"] == want["num_chunks"]
        assert np.array_equal(got["chunk_ptr"].astype(np.int64), want["chunk_ptr"])
        assert same_bits(got["row_idx"], want["row_idx"])
        assert np.array_equal(got["col16"], want["col16"])
        assert same_bits(got["value"], want["value"])


# --- the worked example -------------------------------------------------------

def test_fig14_1_every_format(sp, orc):
    rp, ci, va = orc.dense_to_csr(synth.fig14_1_dense())
    inp = synth.CSRInput("fig14_1", 4, 4, rp, ci, va, np.array([1, 2, 3, 4], np.float32),
                         np.zeros(4, np.float32))
    check_matrix(sp, orc, inp, hyb_widths=(0, 1, 2, 3), sell_rows=(0, 1, 2, 3, 4, 100),
                 xb_chunks=(0, 1, 2, 3))
    with sp.SparseMatrix(4, 4, dev(rp), dev(ci), dev(va)) as m:
        for f in ("COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK"):
            m.convert(f, ell_width=2, section_rows=2, chunk_cols=2)
        for f in FORMATS:
            y = torch.zeros(4, device="cuda")
            m.run(f, dev(inp.x), y)
            assert y.cpu().tolist() == [15.0, 50.0, 28.0, 24.0], f
        ell = m.export("ELL")
        assert ell["value"].tolist() == [1, 5, 2, 6, 7, 3, 8, 0, 0, 9, 0, 0]
        assert ell["col_idx"].tolist() == [0, 0, 1, 3, 1, 2, 2, -1, -1, 3, -1, -1]
        jds = m.export("JDS")
        assert jds["perm"].tolist() == [1, 0, 2, 3]
        assert jds["iter_ptr"].tolist() == [0, 4, 7, 8]
        sell = m.export("SELL")  # two sections of two rows, widths 3 and 2
        assert sell["perm"].tolist() == [1, 0, 2, 3]
        assert sell["sec_ptr"].tolist() == [0, 6, 10]
        assert sell["value"].tolist() == [5, 1, 3, 7, 9, 0, 2, 6, 8, 0]
        assert sell["col_idx"].tolist() == [0, 0, 2, 1, 3, -1, 1, 3, 2, -1]
        xb = m.export("XBLOCK")  # chunks of columns {0, 1} and {2, 3}
        assert xb["chunk_ptr"].tolist() == [0, 4, 8]
        assert xb["row_idx"].tolist() == [0, 0, 1, 2, 1, 1, 2, 3]
        assert xb["col16"].tolist() == [0, 1, 0, 1, 0, 1, 0, 1]
        assert xb["value"].tolist() == [1, 7, 5, 2, 3, 9, 8, 6]


# --- irregular and degenerate matrices -------------------------------------------

EDGE = {
    "one_by_one": dict(num_rows=1, num_cols=1, mean_len=1),
    "empty_rows": dict(num_rows=3001, num_cols=2000, mean_len=5, empty_frac=0.3),
    "all_empty": dict(num_rows=777, num_cols=50, mean_len=0, empty_frac=1.0),
    "one_long_row": dict(num_rows=100, num_cols=200_000, mean_len=3, long_rows=1,
                         long_len=150_000),
    "few_long_rows": dict(num_rows=5003, num_cols=60_000, mean_len=7, long_rows=5,
                          long_len=50_000),
    "unsorted": dict(num_rows=2048, num_cols=4096, mean_len=9, unsorted=True),
    "duplicates": dict(num_rows=1500, num_cols=300, mean_len=12, duplicates=True),
    "explicit_zeros": dict(num_rows=1024, num_cols=1024, mean_len=6, zeros_frac=0.3),
    "rows_not_mult4": dict(num_rows=1003, num_cols=1003, mean_len=4),
    "tall_skinny": dict(num_rows=100_000, num_cols=3, mean_len=2),
    "wide_short": dict(num_rows=3, num_cols=100_000, mean_len=4000),
    "len_beyond_exact_hist": dict(num_rows=60, num_cols=20_000, mean_len=5000),
    "many_empty_then_long": dict(num_rows=20_000, num_cols=9000, mean_len=1, empty_frac=0.97,
                                 long_rows=3, long_len=9000),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(sp, orc, name):
    inp = synth.random_csr(11, name=name, **EDGE[name])
    lens = np.diff(inp.row_ptrs)
    mx = int(lens.max()) if lens.size else 0
    R, Z = inp.num_rows, inp.nnz
    ell_ok = R * mx <= min(2**31 - 1, 4 * Z + R)
    check_matrix(sp, orc, inp, hyb_widths=(0, 1, 5), ell_ok=ell_ok, sell_rows=(0, 1, 3, 32),
                 xb_chunks=(0, 1, 7, 1000))


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_arrays(sp, orc, offset):
    inp = synth.random_csr(3, 4001, 3000, mean_len=8, empty_frac=0.05, long_rows=3,
                           long_len=2500, name=f"misaligned{offset}")
    check_matrix(sp, orc, inp, hyb_widths=(0,), offset=offset, ell_ok=False)
    short = synth.random_csr(4, 4001, 3000, mean_len=8, name=f"misaligned{offset}_short")
    check_matrix(sp, orc, short, hyb_widths=(0, 3), offset=offset)


def test_empty_matrix(sp):
    rp = torch.zeros(1, dtype=torch.int32, device="cuda")
    with sp.SparseMatrix(0, 0, rp, torch.empty(0, dtype=torch.int32, device="cuda"),
                         torch.empty(0, device="cuda")) as m:
        for f in ("COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK"):
            m.convert(f)
        for f in FORMATS:
            m.run(f, None, None)
        assert m.stats()["max_len"] == 0


def test_zero_columns_with_entries_rejected(sp):
    rp = dev(np.array([0, 1], np.int32))
    with pytest.raises(sp.SpmvError) as ei:
        sp.spmv_create_csr(1, 0, 1, rp, dev(np.array([0], np.int32)),
                           dev(np.array([1.0], np.float32)))
    assert ei.value.code == sp.SPMV_ERR_COL_OUT_OF_RANGE


# --- full-size workloads (the bench's configurations) ---------------------------

_CACHE = {}


def workload(name):
    if name not in _CACHE:
        _CACHE.clear()
        _CACHE[name] = synth.make_workload(name)
    return _CACHE[name]


@pytest.mark.parametrize("name", ["tiny_uniform", "laplace2d", "uniform_random", "skewed",
                                  "stencil27"])
def test_workload_full_size(sp, orc, name):
    inp = workload(name)
    res = check_matrix(sp, orc, inp, hyb_widths=(0,), ell_ok=(name != "skewed"))
    print(name, {k: round(v, 4) for k, v in res.items()})


def test_skewed_selects_xblock_and_hyb_width_20(sp):
    """Rows of 10-20 random columns plus a few of 1000-5000: the HYB width is
    20, as the format-selection page says; the columns are scattered, so the
    x-blocked list is chosen."""
    inp = workload("skewed")
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        assert m.stats()["gather_lines"] > 30
        assert m.select() == ("XBLOCK", 20)


# --- validation errors (input sanity rules) --------------------------------------

def _create_status(sp, R, C, rp, ci, va):
    import ctypes
    h = ctypes.c_void_p()
    rp_t, ci_t, va_t = dev(rp), dev(ci), dev(va)
    st = sp._lib.spmv_create_csr(ctypes.byref(h), R, C, len(ci), rp_t.data_ptr(),
                                 ci_t.data_ptr() if len(ci) else None,
                                 va_t.data_ptr() if len(va) else None,
                                 torch.cuda.current_stream().cuda_stream)
    if st == sp.SPMV_OK:
        sp._lib.spmv_destroy(h)
    else:
        assert h.value is None
    return st


def test_validation_errors(sp, orc):
    rp, ci, va = orc.dense_to_csr(synth.fig14_1_dense())
    assert _create_status(sp, 4, 4, rp, ci, va) == sp.SPMV_OK
    for bad_rp in ([1, 2, 5, 7, 8], [0, 3, 2, 7, 8], [0, 2, 5, 7, 7], [0, 2, 5, 9, 8]):
        assert _create_status(sp, 4, 4, np.array(bad_rp, np.int32), ci, va) == \
            sp.SPMV_ERR_BAD_ROWPTRS, bad_rp
    for pos, val in ((5, 4), (0, -1), (7, 1 << 30)):
        bad = ci.copy()
        bad[pos] = val
        assert _create_status(sp, 4, 4, rp, bad, va) == sp.SPMV_ERR_COL_OUT_OF_RANGE
    assert _create_status(sp, 4, 3, rp, ci, va) == sp.SPMV_ERR_COL_OUT_OF_RANGE
    bad = ci.copy()
    bad[0] = 9
    assert _create_status(sp, 4, 4, np.array([0, 3, 2, 7, 8], np.int32), bad, va) == \
        sp.SPMV_ERR_BAD_ROWPTRS  # row pointers are reported first
    # the same checks the oracle makes
    assert orc.validate(4, 4, np.array([0, 3, 2, 7, 8], np.int32), ci) == oracle.BAD_ROWPTRS
    # a decrease whose 32-bit difference wraps to a positive value (2e9 -> -2e9),
    # inside a lane's 8 rows, at a lane boundary and at a 2048-row tile boundary
    Z = 10
    ci10, va10 = np.zeros(Z, np.int32), np.ones(Z, np.float32)
    for at in (1005, 1008, 2048):
        rp_w = np.zeros(4097, np.int32)
        rp_w[at] = 2_000_000_000
        rp_w[at + 1] = -2_000_000_000
        rp_w[at + 2:] = Z
        assert orc.validate(4096, 4, rp_w, ci10) == oracle.BAD_ROWPTRS
        assert _create_status(sp, 4096, 4, rp_w, ci10, va10) == sp.SPMV_ERR_BAD_ROWPTRS, at


def test_large_validation_error_position(sp):
    inp = synth.random_csr(5, 200_000, 1000, mean_len=6)
    ci = inp.col_idx.copy()
    ci[len(ci) // 2 + 1] = 1000
    assert _create_status(sp, inp.num_rows, 1000, inp.row_ptrs, ci, inp.value) == \
        sp.SPMV_ERR_COL_OUT_OF_RANGE
    rp = inp.row_ptrs.copy()
    rp[150_000] = rp[150_001] + 1
    assert _create_status(sp, inp.num_rows, 1000, rp, inp.col_idx, inp.value) == \
        sp.SPMV_ERR_BAD_ROWPTRS


# --- API behaviour ------------------------------------------------------------------

def _fig(sp, orc):
    rp, ci, va = orc.dense_to_csr(synth.fig14_1_dense())
    return sp.SparseMatrix(4, 4, dev(rp), dev(ci), dev(va))


def test_not_converted_and_argument_errors(sp, orc):
    with _fig(sp, orc) as m:
        x = dev(np.array([1, 2, 3, 4], np.float32))
        y = torch.zeros(4, device="cuda")
        for f in ("COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK"):
            with pytest.raises(sp.SpmvError) as ei:
                m.run(f, x, y)
            assert ei.value.code == sp.SPMV_ERR_NOT_CONVERTED
        with pytest.raises(sp.SpmvError) as ei:
            m.export("ELL")
        assert ei.value.code == sp.SPMV_ERR_NOT_CONVERTED
        buf = torch.zeros(8, device="cuda")
        with pytest.raises(sp.SpmvError) as ei:
            m.run("CSR", buf[:4], buf[2:6])  # x and y overlap
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        host = torch.zeros(4).pin_memory()
        st = sp._lib.spmv_run(m.handle, sp.SPMV_CSR, x.data_ptr(), host.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
        assert st == sp.SPMV_ERR_INVALID_ARG  # host memory is refused, never touched
        assert host.tolist() == [0, 0, 0, 0]
        with pytest.raises(sp.SpmvError):
            m.run(7, x, y)
        with pytest.raises(sp.SpmvError):
            sp.spmv_convert_hyb(m.handle, -1)
        with pytest.raises(sp.SpmvError) as ei:
            sp.spmv_convert_sell(m.handle, -1)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG


def test_sell_section_heights_and_wide_sections(sp, orc):
    """Section heights that are and are not multiples of 4, numRows not a
    multiple of S, and sections wider than the row-parallel part (split into
    tail items): arrays bit-exact, y within the tolerance."""
    inp = synth.random_csr(31, 9001, 7000, mean_len=6, empty_frac=0.05, long_rows=300,
                           long_len=700, name="sell_wide")
    check_matrix(sp, orc, inp, formats=("SELL",), sell_rows=(0, 1, 2, 4, 5, 64, 100, 128,
                                                              256, 1000, 9001, 20000))
    # some rows beyond the exact histogram range: widths read back from the device
    big = synth.random_csr(32, 3000, 40_000, mean_len=20, long_rows=130, long_len=1500,
                           name="sell_readback")
    check_matrix(sp, orc, big, formats=("SELL",), sell_rows=(0, 4, 7, 128))
    # few slots per row on average (the main part takes 4 rows per thread)
    # with wide sections all the same (tail items)
    narrow = synth.random_csr(34, 100_003, 50_000, mean_len=3, long_rows=5, long_len=1000,
                              name="sell_narrow_wide")
    lens = np.sort(np.diff(narrow.row_ptrs))[::-1]
    slots = sum(min(128, lens.size - k) * int(lens[k]) for k in range(0, lens.size, 128))
    assert slots <= 8 * narrow.num_rows
    check_matrix(sp, orc, narrow, formats=("SELL",), sell_rows=(0, 6, 128))


@pytest.mark.parametrize("max_len", [1, 31, 32, 63, 64, 65, 200, 255, 256])
def test_length_sort_pass_boundary(sp, orc, max_len):
    """Longest row on both sides of 32 (the row sort's single-pass form, two
    kernels, takes at most 32 digits), of 256 (the general form takes one
    8-bit radix pass below it, two from it) and of 64 (rows longer than that
    are copied by the whole warp), over several 2048-row sort tiles with a
    ragged last tile: JDS and SELL arrays bit-exact, perm included."""
    inp = synth.random_csr(70 + max_len, 7001, 9000, mean_len=0 if max_len < 8 else 4,
                           empty_frac=0.1, long_rows=37, long_len=max_len,
                           name=f"sort_boundary_{max_len}")
    assert int(np.diff(inp.row_ptrs).max()) == max_len
    check_matrix(sp, orc, inp, formats=("JDS", "SELL"), sell_rows=(0, 3, 128))


@pytest.mark.parametrize("width", [63, 64, 65])
def test_jds_diagonal_parameter_boundary(sp, orc, width):
    """9000 rows of `width` entries and 40 rows of 100: the first `width`
    diagonals are row-parallel (at least 8192 wide). Up to 64 of them the
    SpMV takes their iterPtr entries as a launch parameter, past 64 from
    shared memory; the 35-36 diagonals of the long rows run as tail tiles."""
    rng = np.random.default_rng(500 + width)
    R, C = 9040, 3000
    lens = np.full(R, width, np.int64)
    lens[rng.choice(R, 40, replace=False)] = 100
    cols = synth._distinct_sorted_columns(rng, lens, C)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    val = rng.uniform(-1.0, 1.0, cols.size).astype(np.float32)
    x = rng.uniform(-1.0, 1.0, C).astype(np.float32)
    y0 = rng.uniform(-1.0, 1.0, R).astype(np.float32)
    check_matrix(sp, orc, synth.CSRInput(f"jds_param{width}", R, C, rp, cols, val, x, y0),
                 formats=("JDS",))


def test_length_sort_two_scan_passes(sp, orc):
    """5,120,077 rows of at most 7 entries: the row sort's per-tile counts
    (8 digits x 2,501 tiles of 2048 rows = 20,008) take two passes of the
    one-block scan, the second ragged; JDS and SELL arrays bit-exact."""
    inp = synth.random_csr(91, 5_120_077, 7, mean_len=2, name="two_scan_passes")
    assert int(np.diff(inp.row_ptrs).max()) == 7
    check_matrix(sp, orc, inp, formats=("JDS", "SELL"))


def test_csr_large_ragged(sp, orc):
    """CSR on 621K nonzeros (2426 full 256-entry warp blocks) with empty rows
    (chunks decoded by search), rows spanning many blocks and nnz not a
    multiple of 256; aligned (16-byte loads) and misaligned (scalar loads)."""
    inp = synth.random_csr(61, 100_003, 50_000, mean_len=7, empty_frac=0.2, long_rows=3,
                           long_len=20_000, name="csr_pipelined")
    assert inp.nnz // 256 >= 8 * 152 and inp.nnz % 256 != 0
    check_matrix(sp, orc, inp, formats=("CSR",))
    check_matrix(sp, orc, inp, formats=("CSR",), offset=1)


def test_xblock_chunkings(sp, orc):
    """Chunk widths that are and are not multiples of 4 (x staged with 16-byte
    or scalar loads), numCols not a multiple of B, empty chunks, rows spread
    over many chunks and CTAs. Up to 256 chunks the build sorts tiles of
    nonzeros in shared memory and decodes rows from the CSR chunk records (B
    = 274: 256 chunks); more chunks take the radix sort of all nonzeros (B =
    273: 257 chunks), converted without a COO conversion first (rows
    expanded) and after it (the COO row array reused)."""
    inp = synth.random_csr(51, 20_011, 70_001, mean_len=9, empty_frac=0.05, long_rows=5,
                           long_len=3000, name="xb_scatter")
    check_matrix(sp, orc, inp, formats=("XBLOCK",), xb_chunks=(0, 1, 3, 16, 273, 274, 1001,
                                                               4096, 49152))
    check_matrix(sp, orc, inp, formats=("COO", "XBLOCK"), xb_chunks=(5, 777))
    # columns only in a few chunks: the others are empty
    band = synth.random_csr(52, 3000, 60_000, mean_len=4, name="xb_narrow")
    band.col_idx[:] = (band.col_idx % 500) + 20_000
    for r in range(band.num_rows):  # keep each row's columns distinct and ascending
        a, b = band.row_ptrs[r], band.row_ptrs[r + 1]
        band.col_idx[a:b] = np.sort(np.unique(band.col_idx[a:b]).tolist() +
                                    list(range(30_000, 30_000 + (b - a) -
                                               np.unique(band.col_idx[a:b]).size)))
    check_matrix(sp, orc, band, formats=("XBLOCK",), xb_chunks=(0, 64, 4000))


def test_xblock_misaligned_x(sp, orc):
    inp = synth.random_csr(53, 5003, 9001, mean_len=7, name="xb_misaligned")
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        for B in (0, 1000, 1024):
            m.convert("XBLOCK", chunk_cols=B)
            for off in (1, 2, 3):
                xb = dev(np.concatenate([np.zeros(off, np.float32), inp.x]))
                y = dev(inp.y0)
                m.run("XBLOCK", xb[off:], y)
                torch.cuda.synchronize()
                check_tol(y.cpu().numpy(), yref, mag, f"xblock B={B} x offset {off}")
        with pytest.raises(sp.SpmvError) as ei:
            m.convert("XBLOCK", chunk_cols=49153)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        with pytest.raises(sp.SpmvError) as ei:
            m.convert("XBLOCK", chunk_cols=-1)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG


def test_sell_reconvert_and_too_large(sp, orc):
    inp = synth.random_csr(33, 2000, 50_000, mean_len=2, long_rows=1, long_len=40_000)
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        # S = 128: the long row pads a section to 128 * 40000 slots, over budget;
        # a failed conversion leaves no SELL behind, a later one replaces it
        assert not sell_fits(inp.row_ptrs, 128) and sell_fits(inp.row_ptrs, 1)
        for S in (1, 0, 3, 8, 2, 128):
            if not sell_fits(inp.row_ptrs, S or 128):
                with pytest.raises(sp.SpmvError) as ei:
                    m.convert("SELL", section_rows=S)
                assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
                with pytest.raises(sp.SpmvError) as ei:
                    m.run("SELL", dev(inp.x), dev(inp.y0))
                assert ei.value.code == sp.SPMV_ERR_NOT_CONVERTED
                continue
            m.convert("SELL", section_rows=S)
            y = dev(inp.y0)
            m.run("SELL", dev(inp.x), y)
            torch.cuda.synchronize()
            check_tol(y.cpu().numpy(), yref, mag, f"sell S={S}")


def test_accumulates_and_streams(sp, orc):
    inp = synth.random_csr(21, 5000, 4000, mean_len=9, empty_frac=0.1)
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    ax = yref - inp.y0.astype(np.float64)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        m = sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                            dev(inp.value))
        for f in ("COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK"):
            m.convert(f)
        for f in FORMATS:
            y = dev(inp.y0)
            m.run(f, dev(inp.x), y)
            m.run(f, dev(inp.x), y)  # y = y0 + 2 A x
            s.synchronize()
            ok, worst = oracle.within_tolerance(y.cpu().numpy(), inp.y0 + 2 * ax,
                                                2 * mag, rel=1e-5)
            assert ok, (f, worst)
        m.close()


def test_guard_bands_untouched(sp, orc):
    inp = synth.random_csr(8, 3001, 2999, mean_len=6, long_rows=2, long_len=20)
    G = 64
    sentinel = np.float32(-7.25e33)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        for f in ("COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK"):
            m.convert(f)
        for f in FORMATS:
            buf = torch.full((inp.num_rows + 2 * G,), float(sentinel), device="cuda")
            y = buf[G:G + inp.num_rows]
            y.copy_(dev(inp.y0))
            xb = torch.full((inp.num_cols + 2 * G,), float(sentinel), device="cuda")
            x = xb[G:G + inp.num_cols]
            x.copy_(dev(inp.x))
            m.run(f, x, y)
            torch.cuda.synchronize()
            b = buf.cpu().numpy()
            assert np.all(b[:G] == sentinel) and np.all(b[-G:] == sentinel), f
            xb2 = xb.cpu().numpy()
            assert np.all(xb2[:G] == sentinel) and np.all(xb2[-G:] == sentinel), f


def test_memory_limit(sp, orc):
    inp = synth.random_csr(4, 20_000, 20_000, mean_len=10)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        sp.spmv_set_memory_limit(1024)
        try:
            with pytest.raises(sp.SpmvError) as ei:
                m.convert("ELL")
            assert ei.value.code == sp.SPMV_ERR_ALLOC
        finally:
            sp.spmv_set_memory_limit(None)
        m.convert("ELL")


def test_hyb_reconvert_widths(sp, orc):
    inp = synth.random_csr(9, 4000, 3000, mean_len=8, long_rows=4, long_len=1500)
    yref, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                         dev(inp.value)) as m:
        with pytest.raises(sp.SpmvError) as ei:
            m.convert("HYB", ell_width=10_000)  # capped at the longest row: over budget
        assert ei.value.code == sp.SPMV_ERR_TOO_LARGE
        for w in (3, 0, 1, 7, 20):
            m.convert("HYB", ell_width=w)
            y = dev(inp.y0)
            m.run("HYB", dev(inp.x), y)
            torch.cuda.synchronize()
            check_tol(y.cpu().numpy(), yref, mag, f"hyb width {w}")


def test_launch_counter_counts_kernels(sp, orc):
    with _fig(sp, orc) as m:
        m.convert("HYB", ell_width=2)
        n0 = sp.spmv_launch_count()
        x = dev(np.array([1, 2, 3, 4], np.float32))
        y = torch.zeros(4, device="cuda")
        m.run("CSR", x, y)
        m.run("HYB", x, y)
        assert sp.spmv_launch_count() - n0 == 3


def test_gather_locality_statistic(sp):
    """Banded matrices touch few 128-byte lines of x per 32 gathers; uniform
    random columns touch nearly 32 (the statistic picks the CSR kernel)."""
    band = synth.laplace2d(256)
    rand = synth.uniform_rows("rand", 200_000, 8)
    got = {}
    for inp in (band, rand):
        with sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                             dev(inp.value)) as m:
            got[inp.name] = m.stats()["gather_lines"]
    assert 0 < got["laplace2d"] <= 8, got
    assert got["rand"] >= 24, got


def wide_rows(seed, num_rows, num_cols, lo, hi, name):
    """Rows of lo..hi distinct sorted columns, the first row exactly hi long;
    values, x and y0 U(-1, 1)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, num_rows).astype(np.int64)
    lens[0] = hi
    cols = synth._distinct_sorted_columns(rng, lens, num_cols)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    val = rng.uniform(-1.0, 1.0, cols.size).astype(np.float32)
    x = rng.uniform(-1.0, 1.0, num_cols).astype(np.float32)
    y0 = rng.uniform(-1.0, 1.0, num_rows).astype(np.float32)
    return synth.CSRInput(name, num_rows, num_cols, rp, cols, val, x, y0)


@pytest.mark.parametrize("offset", [0, 1, 3])
@pytest.mark.parametrize("kind", ["random", "runs"])
def test_warp_staged_row_scatters(sp, orc, offset, kind):
    """Rows of 17-32 entries take the warp-staged scatters: ELL (width 32),
    JDS and SELL (longest row 32; SELL with sections of 1, 7 and 128 rows),
    and HYB at widths 24 and 28, where the warps whose rows hold more entries
    than their buffer read directly. Aligned arrays
    stage by 16-byte asynchronous copies, misaligned views entry by entry; the
    last warp is ragged (5003 rows). "runs": rows of 27 entries with one of
    24 every 50 rows, so that after the length sort most warps of the JDS
    scatter hold consecutive original rows (one contiguous range) and some do
    not; "random": lengths at random, so that no warp does."""
    inp = wide_rows(31 + offset, 5003, 4000, 17, 32, f"wide{offset}")
    if kind == "runs":
        lens = np.full(inp.num_rows, 27, np.int64)
        lens[::50] = 24
        lens[1] = 32
        rng = np.random.default_rng(7 + offset)
        cols = synth._distinct_sorted_columns(rng, lens, inp.num_cols)
        rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        val = rng.uniform(-1.0, 1.0, cols.size).astype(np.float32)
        inp = synth.CSRInput(f"runs{offset}", inp.num_rows, inp.num_cols, rp, cols, val,
                             inp.x, inp.y0)
    check_matrix(sp, orc, inp, formats=("ELL", "HYB", "JDS", "SELL"), hyb_widths=(24, 28),
                 sell_rows=(1, 7, 128), offset=offset)
