"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Every check here compares the oracle with something other than itself:
arrays printed in the pages' figures (tests/golden/), dense brute force with
NumPy, closed forms of stencil matrices, round trips and layout invariants.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import load_golden

FIG = load_golden("fig14_1.json")


def fig_csr(orc):
    return orc.dense_to_csr(np.array(FIG["dense"]["rows"], np.float32))


# --- worked example of Fig. 14.1 ------------------------------------------

def test_fig14_1_csr(orc):
    rp, ci, v = fig_csr(orc)
    assert rp.tolist() == FIG["csr"]["rowPtrs"]
    assert ci.tolist() == FIG["csr"]["colIdx"]
    assert v.tolist() == FIG["csr"]["value"]


def test_fig14_1_coo(orc):
    coo = orc.csr_to_coo(*fig_csr(orc))
    assert coo["row_idx"].tolist() == FIG["coo"]["rowIdx"]
    assert coo["col_idx"].tolist() == FIG["coo"]["colIdx"]
    assert coo["value"].tolist() == FIG["coo"]["value"]


def test_fig14_1_ell(orc):
    ell = orc.csr_to_ell(*fig_csr(orc))
    assert ell["width"] == FIG["ell"]["width"]
    for i, (gv, gc) in enumerate(zip(FIG["ell"]["value"], FIG["ell"]["colIdx"])):
        if gv is None:
            # padding slot: value 0 (page), column -1 (our reading of '*')
            assert ell["value"][i] == 0.0 and ell["col_idx"][i] == -1
        else:
            assert ell["value"][i] == gv and ell["col_idx"][i] == gc
    assert ell["nnz_per_row"].tolist() == [2, 3, 2, 1]


def test_fig14_1_ell_index_formula(orc):
    """Slot i = t*numRows + row, so row = i % numRows for every real entry."""
    rp, ci, v = fig_csr(orc)
    ell = orc.csr_to_ell(rp, ci, v)
    R = ell["num_rows"]
    dense = np.array(FIG["dense"]["rows"], np.float32)
    for i in range(ell["value"].shape[0]):
        if ell["col_idx"][i] >= 0:
            assert dense[i % R, ell["col_idx"][i]] == ell["value"][i]


def test_fig14_1_jds(orc):
    rp, ci, v = fig_csr(orc)
    jds = orc.csr_to_jds(rp, ci, v)
    assert np.diff(rp).tolist() == FIG["jds"]["row_lengths_before_sort"]
    assert jds["perm"].tolist() == FIG["jds"]["row"]
    assert jds["iter_ptr"].tolist() == FIG["jds"]["iterPtr"]
    dense = np.array(FIG["dense"]["rows"], np.float32)
    for i, (row, pos) in enumerate(FIG["jds"]["value_order"]):
        nz_cols = np.flatnonzero(dense[row])
        assert jds["col_idx"][i] == nz_cols[pos]
        assert jds["value"][i] == dense[row, nz_cols[pos]]


def test_fig14_1_spmv_every_format(orc):
    rp, ci, v = fig_csr(orc)
    x = np.array(FIG["spmv"]["x"], np.float32)
    y0 = np.array(FIG["spmv"]["y0"], np.float32)
    want = FIG["spmv"]["y"]
    y, _ = orc.spmv_csr(rp, ci, v, x, y0)
    assert y.tolist() == want
    coo = orc.csr_to_coo(rp, ci, v)
    assert orc.spmv_coo(4, coo["row_idx"], coo["col_idx"], coo["value"], x, y0).tolist() == want
    assert orc.spmv_ell(orc.csr_to_ell(rp, ci, v), x, y0).tolist() == want
    assert orc.spmv_jds(orc.csr_to_jds(rp, ci, v), x, y0).tolist() == want
    for K in range(0, 5):
        assert orc.spmv_hyb(orc.csr_to_hyb(rp, ci, v, K), x, y0).tolist() == want


def test_fig14_1_hyb_width2(orc):
    """K = 2 on Fig. 14.1: only row 1's third entry (column 3, value 9) moves."""
    hyb = orc.csr_to_hyb(*fig_csr(orc), 2)
    assert hyb["value"].tolist() == [1, 5, 2, 6, 7, 3, 8, 0]
    assert hyb["col_idx"].tolist() == [0, 0, 1, 3, 1, 2, 2, -1]
    assert hyb["coo_row_idx"].tolist() == [1]
    assert hyb["coo_col_idx"].tolist() == [3]
    assert hyb["coo_value"].tolist() == [9]


def test_hyb_schematic_counts(orc):
    g = load_golden("hyb_schematic.json")
    lens = np.array(g["row_lengths"])
    R = lens.shape[0]
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ci = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    v = np.arange(1, rp[-1] + 1, dtype=np.float32)
    ell = orc.csr_to_ell(rp, ci, v)
    assert ell["width"] == g["ell_only_width"]
    assert int((ell["col_idx"] < 0).sum()) == g["ell_only_padding"]
    hyb = orc.csr_to_hyb(rp, ci, v, g["hyb_width"])
    assert int((hyb["col_idx"] < 0).sum()) == g["hyb_padding"]
    assert hyb["coo_row_idx"].tolist() == g["coo_rowIdx"]
    assert hyb["value"].shape[0] == R * g["hyb_width"]


# --- dense brute force -----------------------------------------------------

def dense_of(inp):
    A = np.zeros((inp.num_rows, inp.num_cols), np.float64)
    rows = np.repeat(np.arange(inp.num_rows), np.diff(inp.row_ptrs))
    np.add.at(A, (rows, inp.col_idx), inp.value.astype(np.float64))
    return A


CASES = [
    dict(num_rows=1, num_cols=1),
    dict(num_rows=7, num_cols=5, mean_len=2),
    dict(num_rows=33, num_cols=64, mean_len=6, empty_frac=0.3),
    dict(num_rows=64, num_cols=64, mean_len=3, long_rows=1, long_len=64),
    dict(num_rows=50, num_cols=40, mean_len=5, unsorted=True),
    dict(num_rows=40, num_cols=30, mean_len=5, duplicates=True),
    dict(num_rows=45, num_cols=45, mean_len=4, zeros_frac=0.3),
    dict(num_rows=20, num_cols=64, mean_len=0, empty_frac=1.0),
]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_spmv_matches_dense_brute_force(orc, seed, case):
    inp = synth.random_csr(seed, **CASES[case])
    want = inp.y0.astype(np.float64) + dense_of(inp) @ inp.x.astype(np.float64)
    y, mag = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
    # the magnitude sum bounds |y - y0| and is at least |y0|
    assert np.all(mag + 1e-12 >= np.abs(y - inp.y0))
    assert np.all(mag >= np.abs(inp.y0))


def entry_magnitudes(inp):
    """Per row: sum over its stored entries of |a_k x_col(k)|, plus |y0|."""
    rows = np.repeat(np.arange(inp.num_rows), np.diff(inp.row_ptrs))
    mag = np.zeros(inp.num_rows, np.float64)
    np.add.at(mag, rows, np.abs(inp.value.astype(np.float64) *
                                inp.x.astype(np.float64)[inp.col_idx]))
    return mag + np.abs(inp.y0.astype(np.float64))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_spmv_rows_matches_dense_brute_force(orc, case):
    """The same definition over a chosen list of rows (the form used to check
    sampled rows of very large matrices): entry i of the result is row
    rows[i] of A x + y0. The list has repeats, is in no particular order and
    is shorter than the row count where it can be, so that a result indexed by
    list position instead of row number fails."""
    inp = synth.random_csr(3, **CASES[case])
    R = inp.num_rows
    rng = np.random.default_rng(100 + case)
    n = max(1, (2 * R) // 3)
    rows = rng.integers(0, R, size=n)
    if n > 2:
        rows[1] = rows[0]  # a repeat
        rows[-1] = R - 1   # the last row
    full = inp.y0.astype(np.float64) + dense_of(inp) @ inp.x.astype(np.float64)
    y, mag = orc.spmv_csr_rows(rows, inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0)
    np.testing.assert_allclose(y, full[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mag, entry_magnitudes(inp)[rows], rtol=1e-12, atol=1e-12)


def test_spmv_unit_vectors_give_columns(orc):
    """x = e_j gives y - y0 = column j of A (exactly: one product per entry)."""
    inp = synth.random_csr(5, 17, 13, mean_len=4)
    A = dense_of(inp)
    for j in range(13):
        x = np.zeros(13, np.float32)
        x[j] = 1.0
        y, _ = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, x, inp.y0)
        assert np.array_equal(y - inp.y0.astype(np.float64), A[:, j])


# --- closed forms -----------------------------------------------------------

@pytest.mark.parametrize("side", [1, 2, 5, 16])
def test_laplace2d_closed_form(orc, side):
    """x = 1: row sum of the 5-point Laplacian is 4 - (#in-grid neighbours):
    0 inside, 1 on an edge, 2 at a corner (4 for a 1x1 grid)."""
    inp = synth.laplace2d(side)
    x = np.ones(inp.num_cols, np.float32)
    y, _ = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, x, inp.y0)
    i, j = np.divmod(np.arange(side * side), side)
    nb = (i > 0).astype(int) + (i < side - 1) + (j > 0) + (j < side - 1)
    assert np.array_equal(y - inp.y0.astype(np.float64), 4.0 - nb)
    lens = np.diff(inp.row_ptrs)
    assert np.array_equal(lens, 1 + nb)


def test_laplace2d_full_size_counts():
    """2048^2 grid with dropped out-of-grid neighbours: 5*n^2 - 4*n entries."""
    n = 2048
    assert 5 * n * n - 4 * n == 20_963_328


@pytest.mark.parametrize("side", [1, 3, 6])
def test_stencil27_closed_form(orc, side):
    """x = 1: y - y0 = diag + sum(off) = 1 + 2*sum(off) since every off-diagonal
    is positive; the row length is the product of the per-axis neighbour counts."""
    inp = synth.stencil27(side)
    x = np.ones(inp.num_cols, np.float32)
    y, _ = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, x, inp.y0)
    rp = inp.row_ptrs
    for r in range(inp.num_rows):
        seg = inp.value[rp[r]:rp[r + 1]].astype(np.float64)
        cols = inp.col_idx[rp[r]:rp[r + 1]]
        off = seg[cols != r].sum()
        diag = seg[cols == r][0]
        assert diag == np.float32(1.0 + off)
        assert y[r] - np.float64(inp.y0[r]) == pytest.approx(diag + off, rel=1e-12)
    c = np.arange(side)
    per_axis = 1 + (c > 0).astype(int) + (c < side - 1)
    want = (per_axis[:, None, None] * per_axis[None, :, None] * per_axis[None, None, :]).ravel()
    assert np.array_equal(np.diff(rp), want)


def test_stencil27_full_size_count():
    """160^3 grid: (3*160 - 2)^3 entries."""
    assert (3 * 160 - 2) ** 3 == 109_215_352


# --- round trips and invariants --------------------------------------------

def _inputs():
    yield synth.random_csr(0, 60, 50, mean_len=5, empty_frac=0.2, long_rows=2, long_len=40)
    yield synth.random_csr(1, 40, 30, mean_len=5, unsorted=True)
    yield synth.random_csr(2, 30, 20, mean_len=6, duplicates=True)
    yield synth.random_csr(3, 25, 25, mean_len=0, empty_frac=1.0)
    yield synth.random_csr(4, 0, 0)
    yield synth.uniform_rows("u", 64, 8)
    yield synth.laplace2d(9)


@pytest.mark.parametrize("idx", range(7))
def test_round_trips_bit_exact(orc, idx):
    inp = list(_inputs())[idx]
    rp, ci, v = inp.row_ptrs, inp.col_idx, inp.value
    R = inp.num_rows
    coo = orc.csr_to_coo(rp, ci, v)
    assert np.array_equal(orc.coo_to_csr(R, coo["row_idx"]), rp)
    assert np.array_equal(coo["col_idx"], ci) and np.array_equal(coo["value"], v)
    for conv, back in [(orc.csr_to_ell, orc.ell_to_csr), (orc.csr_to_jds, orc.jds_to_csr)]:
        f = conv(rp, ci, v)
        rp2, ci2, v2 = back(f)
        assert np.array_equal(rp2, rp) and np.array_equal(ci2, ci)
        assert np.array_equal(v2.view(np.int32), v.view(np.int32))
    maxlen = int(np.diff(rp).max()) if R else 0
    for K in sorted({0, 1, 3, maxlen}):
        rp2, ci2, v2 = orc.hyb_to_csr(orc.csr_to_hyb(rp, ci, v, K))
        assert np.array_equal(rp2, rp) and np.array_equal(ci2, ci)
        assert np.array_equal(v2.view(np.int32), v.view(np.int32))


@pytest.mark.parametrize("idx", range(7))
def test_layout_invariants(orc, idx):
    inp = list(_inputs())[idx]
    rp, ci, v = inp.row_ptrs, inp.col_idx, inp.value
    R, Z = inp.num_rows, inp.nnz
    lens = np.diff(rp)
    ell = orc.csr_to_ell(rp, ci, v)
    assert int(ell["nnz_per_row"].sum()) == Z
    K = ell["width"]
    assert ell["value"].shape[0] == R * K
    slot = np.arange(R * K)
    t, r = np.divmod(slot, max(R, 1))
    assert np.array_equal(ell["col_idx"] >= 0, t < lens[r] if R else slot < 0)
    jds = orc.csr_to_jds(rp, ci, v)
    perm = jds["perm"]
    assert np.array_equal(np.sort(perm), np.arange(R))
    plen = lens[perm]
    assert np.all(plen[:-1] >= plen[1:])  # longest first
    same = plen[:-1] == plen[1:]
    assert np.all(perm[:-1][same] < perm[1:][same])  # stable
    ip = jds["iter_ptr"]
    assert ip[0] == 0 and ip[-1] == Z
    width = np.diff(ip)
    assert np.array_equal(width, [(lens > t).sum() for t in range(width.shape[0])])


@pytest.mark.parametrize("idx", range(7))
def test_format_spmvs_agree(orc, idx):
    inp = list(_inputs())[idx]
    rp, ci, v = inp.row_ptrs, inp.col_idx, inp.value
    y, _ = orc.spmv_csr(rp, ci, v, inp.x, inp.y0)
    coo = orc.csr_to_coo(rp, ci, v)
    ys = [orc.spmv_coo(inp.num_rows, coo["row_idx"], coo["col_idx"], coo["value"], inp.x, inp.y0),
          orc.spmv_ell(orc.csr_to_ell(rp, ci, v), inp.x, inp.y0),
          orc.spmv_jds(orc.csr_to_jds(rp, ci, v), inp.x, inp.y0),
          orc.spmv_hyb(orc.csr_to_hyb(rp, ci, v, 2), inp.x, inp.y0)]
    for yy in ys:
        np.testing.assert_allclose(yy, y, rtol=1e-12, atol=1e-12)


# --- validation (the page's input sanity rules) -----------------------------

def test_validate(orc):
    rp, ci, v = fig_csr(orc)
    assert orc.validate(4, 4, rp, ci) == oracle.OK
    bad = rp.copy(); bad[2] = 1; bad[1] = 3           # not monotone
    assert orc.validate(4, 4, bad, ci) == oracle.BAD_ROWPTRS
    bad = rp.copy(); bad[0] = 1                        # does not start at 0
    assert orc.validate(4, 4, bad, ci) == oracle.BAD_ROWPTRS
    bad = rp.copy(); bad[4] = 7                        # does not end at nnz
    assert orc.validate(4, 4, bad, ci) == oracle.BAD_ROWPTRS
    badc = ci.copy(); badc[5] = 4                      # column == numCols
    assert orc.validate(4, 4, rp, badc) == oracle.COL_RANGE
    badc = ci.copy(); badc[0] = -1                     # negative column
    assert orc.validate(4, 4, rp, badc) == oracle.COL_RANGE
    assert orc.validate(4, 3, rp, ci) == oracle.COL_RANGE  # column 3 >= 3 columns
    both = rp.copy(); both[1] = 6
    assert orc.validate(4, 4, both, badc) == oracle.BAD_ROWPTRS  # rowPtrs first


def test_validate_decrease_that_wraps(orc):
    # 0, 2e9, -2e9, 10: every 32-bit difference of neighbours is non-negative
    # after wrapping, yet the sequence decreases; "never decreases" (section
    # 5.3 of the SpGEMM page) is a comparison of neighbours
    rp = np.array([0, 2_000_000_000, -2_000_000_000, 10], np.int32)
    wrapped = rp[1:] - rp[:-1]  # int32 arithmetic wraps
    assert (wrapped >= 0).all() and not (rp[1:] >= rp[:-1]).all()
    assert orc.validate(3, 4, rp, np.zeros(10, np.int32)) == oracle.BAD_ROWPTRS


# --- row statistics -----------------------------------------------------------

@pytest.mark.parametrize("idx", range(7))
def test_row_stats(orc, idx):
    inp = list(_inputs())[idx]
    lens = np.diff(inp.row_ptrs).astype(np.int64)
    st = orc.row_stats(inp.row_ptrs)
    if lens.size == 0:
        assert st["max_len"] == 0 and st["mean"] == 0.0
        return
    assert st["max_len"] == lens.max()
    assert st["mean"] == pytest.approx(lens.mean(), rel=1e-14)
    assert st["var"] == pytest.approx(lens.var(), rel=1e-12, abs=1e-12)
    bins = np.where(lens == 0, 0, np.floor(np.log2(np.maximum(lens, 1))).astype(int) + 1)
    assert np.array_equal(st["hist_log2"], np.bincount(bins, minlength=33))


# --- selection: outcomes the selection page states in words --------------------

def test_select_outcomes_described_by_page(orc):
    # regular stencil-like rows (scientific computing) -> ELL
    assert orc.select(4_194_304, 4_194_304, 20_963_328, 5, 3.5) == "ELL"
    assert orc.select(4_096_000, 4_096_000, 109_215_352, 27, 9.0) == "ELL"
    # 99% of rows of length 10-20 plus rows longer than 1000 -> HYB of width 20
    # (with columns close together; scattered columns take the x-blocked list)
    inp = synth.skewed(n=20_000, n_long=2, seed=3)
    lens = np.diff(inp.row_ptrs)
    big = 2_000_000  # the same row mix at a size bound by bandwidth
    assert orc.select(big, big, int(big * inp.nnz / inp.num_rows), int(lens.max()), 4.0) == "HYB"
    assert orc.select(big, big, int(big * inp.nnz / inp.num_rows), int(lens.max()),
                      32.0) == "XBLOCK"
    assert orc.hyb_auto_width(inp.row_ptrs) == 20
    # short irregular rows -> COO; moderate spread with long rows -> CSR
    assert orc.select(1_000_000, 1_000_000, 5_000_000, 40, 32.0) == "COO"
    assert orc.select(1_000_000, 1_000_000, 30_000_000, 100, 4.0) == "CSR"


def test_select_small_matrices_take_csr(orc):
    """Below 4 MiB of compulsory bytes (8 per nonzero, 12 per row, 4 per
    column) the choice is CSR whatever the row mix; at the boundary the
    other rules apply."""
    assert orc.select(4096, 4096, 32_768, 8, 32.0) == "CSR"  # 327,680 bytes
    assert orc.select(4, 4, 8, 3, 0.0) == "CSR"
    assert orc.select(0, 0, 0, 0, 0.0) == "CSR"
    # 8*Z + 12*R + 4*C = 4 MiB exactly: not below, so ELL for equal rows
    R = 65_536
    Z = (4_194_304 - 16 * R) // 8
    assert 8 * Z + 12 * R + 4 * R == 4_194_304
    assert orc.select(R, R, Z, Z // R, 1.0) == "ELL"
    assert orc.select(R - 1, R - 1, Z, Z // R + 1, 1.0) == "CSR"


def test_hyb_auto_width_quantile(orc):
    lens = np.array([1] * 99 + [50])
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    assert orc.hyb_auto_width(rp) == 1
    lens = np.array([1] * 98 + [50, 50])
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    assert orc.hyb_auto_width(rp) == 50
