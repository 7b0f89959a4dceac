"""Pins of the sectioned-ELL variant of JDS ('Regularized Formats (ELL,
Hybrid ELL-COO and JDS)', section 'JDS format', variant paragraph) in the
oracle, against facts fixed by the page and by independent oracle paths."""
import numpy as np
import pytest

import synth
from conftest import load_golden
from test_oracle_pins import _inputs, dense_of, CASES

G = load_golden("sell_fig14_1.json")


def fig_csr(orc):
    return orc.dense_to_csr(synth.fig14_1_dense())


def test_fig14_1_sections_of_two(orc):
    s = orc.csr_to_sell(*fig_csr(orc), G["section_rows"])
    assert s["perm"].tolist() == G["row"]
    assert s["sec_ptr"].tolist() == G["secPtr"]
    for i, (gv, gc) in enumerate(zip(G["value"], G["colIdx"])):
        if gv is None:
            assert s["value"][i] == 0.0 and s["col_idx"][i] == -1
        else:
            assert s["value"][i] == gv and s["col_idx"][i] == gc


def test_fig14_1_spmv(orc):
    x = np.array([1, 2, 3, 4], np.float32)
    for S in (1, 2, 3, 4, 100):
        s = orc.csr_to_sell(*fig_csr(orc), S)
        assert orc.spmv_sell(s, x, np.zeros(4, np.float32)).tolist() == [15, 50, 28, 24]


@pytest.mark.parametrize("idx", range(7))
def test_one_section_is_ell_of_sorted_rows(orc, idx):
    """With S >= numRows there is a single section: slot (t, s) must equal
    the ELL slot (t, perm[s]) of the oracle's ELL (an independent path)."""
    inp = list(_inputs())[idx]
    R = inp.num_rows
    s = orc.csr_to_sell(inp.row_ptrs, inp.col_idx, inp.value, max(R, 1))
    ell = orc.csr_to_ell(inp.row_ptrs, inp.col_idx, inp.value)
    K = ell["width"]
    assert s["col_idx"].shape[0] == R * K
    if R * K:
        t, j = np.divmod(np.arange(R * K), R)
        src = t * R + s["perm"][j]
        assert np.array_equal(s["col_idx"], ell["col_idx"][src])
        assert np.array_equal(s["value"].view(np.int32), ell["value"][src].view(np.int32))
    assert np.array_equal(s["perm"], orc.csr_to_jds(inp.row_ptrs, inp.col_idx, inp.value)["perm"])


@pytest.mark.parametrize("idx", range(7))
@pytest.mark.parametrize("S", [1, 3, 32, 128])
def test_round_trip_and_padding(orc, idx, S):
    inp = list(_inputs())[idx]
    rp, ci, v = inp.row_ptrs, inp.col_idx, inp.value
    s = orc.csr_to_sell(rp, ci, v, S)
    rp2, ci2, v2 = orc.sell_to_csr(s)
    assert np.array_equal(rp2, rp) and np.array_equal(ci2, ci)
    assert np.array_equal(v2.view(np.int32), v.view(np.int32))
    slots = s["col_idx"].shape[0]
    pad = int((s["col_idx"] < 0).sum())
    assert slots - pad == inp.nnz
    lens = np.diff(rp)
    ell_pad = inp.num_rows * (int(lens.max()) if lens.size else 0) - inp.nnz
    assert pad <= ell_pad  # the page: far less padding than one ELL
    if S == 1:
        assert pad == 0
    # every section is padded exactly to its first (longest) row
    R = inp.num_rows
    plen = lens[s["perm"]]
    for k in range((R + S - 1) // S):
        h = min(S, R - k * S)
        assert s["sec_ptr"][k + 1] - s["sec_ptr"][k] == h * plen[k * S]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_spmv_matches_dense(orc, case):
    inp = synth.random_csr(4, **CASES[case])
    want = inp.y0.astype(np.float64) + dense_of(inp) @ inp.x.astype(np.float64)
    for S in (1, 4, 128):
        s = orc.csr_to_sell(inp.row_ptrs, inp.col_idx, inp.value, S)
        np.testing.assert_allclose(orc.spmv_sell(s, inp.x, inp.y0), want, rtol=1e-12, atol=1e-12)
