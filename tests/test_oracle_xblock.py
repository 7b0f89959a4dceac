"""Pins of the x-blocked list ('Introduction to sparse computing and
performance bottleneck location', section 'Building the problem framework':
split x into chunks, one thread block per chunk's nonzeros) in the oracle:
hand-worked Fig. 14.1 chunkings, reduction to COO for a single chunk, dense
brute force, round trips and layout invariants."""
import numpy as np
import pytest

import synth
from conftest import load_golden
from test_oracle_pins import CASES, _inputs, dense_of

G = load_golden("xblock_fig14_1.json")


def fig(orc):
    return orc.dense_to_csr(synth.fig14_1_dense())


@pytest.mark.parametrize("case", range(len(G["cases"])))
def test_fig14_1_chunkings(orc, case):
    g = G["cases"][case]
    xb = orc.csr_to_xblock(*fig(orc), 4, g["chunk_cols"])
    assert xb["chunk_ptr"].tolist() == g["chunk_ptr"]
    assert xb["row_idx"].tolist() == g["row_idx"]
    assert xb["col16"].tolist() == g["col16"]
    assert xb["value"].tolist() == g["value"]
    x = np.array([1, 2, 3, 4], np.float32)
    assert orc.spmv_xblock(xb, x, np.zeros(4, np.float32)).tolist() == [15, 50, 28, 24]


@pytest.mark.parametrize("idx", range(7))
def test_single_chunk_is_coo(orc, idx):
    """With B >= numCols there is one chunk: the oracle's COO (an independent
    path) followed by padding to a multiple of 4."""
    inp = list(_inputs())[idx]
    C = inp.num_cols
    if C > 65536:
        pytest.skip("local columns are 16 bits")
    xb = orc.csr_to_xblock(inp.row_ptrs, inp.col_idx, inp.value, C, max(C, 1))
    coo = orc.csr_to_coo(inp.row_ptrs, inp.col_idx, inp.value)
    Z = inp.nnz
    assert xb["chunk_ptr"].tolist() == ([0, (Z + 3) // 4 * 4] if C else [0])
    assert np.array_equal(xb["row_idx"][:Z], coo["row_idx"])
    assert np.array_equal(xb["col16"][:Z].astype(np.int32), coo["col_idx"])
    assert np.array_equal(xb["value"][:Z].view(np.int32), coo["value"].view(np.int32))
    assert (xb["row_idx"][Z:] == -1).all() and not xb["col16"][Z:].any()
    assert not xb["value"][Z:].view(np.int32).any()


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("B", [1, 7, 64, 1000])
def test_spmv_matches_dense(orc, case, B):
    inp = synth.random_csr(1, **CASES[case])
    xb = orc.csr_to_xblock(inp.row_ptrs, inp.col_idx, inp.value, inp.num_cols, B)
    y = orc.spmv_xblock(xb, inp.x, inp.y0)
    want = dense_of(inp) @ inp.x.astype(np.float64) + inp.y0
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("idx", range(7))
@pytest.mark.parametrize("B", [1, 5, 256])
def test_round_trip_and_invariants(orc, idx, B):
    inp = list(_inputs())[idx]
    rp, ci, v = inp.row_ptrs, inp.col_idx, inp.value
    R, C = inp.num_rows, inp.num_cols
    xb = orc.csr_to_xblock(rp, ci, v, C, B)
    cp, rows, cols = xb["chunk_ptr"], xb["row_idx"], xb["col16"]
    nch = xb["num_chunks"]
    assert nch == (C + B - 1) // B
    assert (cp % 4 == 0).all() and (np.diff(cp) >= 0).all()
    counts = np.bincount(ci // B, minlength=nch) if inp.nnz else np.zeros(nch, np.int64)
    for c in range(nch):
        seg = rows[cp[c]:cp[c + 1]]
        real = seg[seg >= 0]
        assert real.size == counts[c]
        assert (seg[:real.size] >= 0).all() and (seg[real.size:] == -1).all()
        assert seg.size - real.size < 4
        assert (np.diff(real) >= 0).all()  # CSR order: rows ascend
        lc = cols[cp[c]:cp[c] + real.size].astype(np.int64)
        assert (lc < B).all() and (c * B + lc < C).all()
    # entries keep their CSR order inside a row: round trip exact for sorted rows
    rp2, ci2, v2 = orc.xblock_to_csr(xb)
    assert np.array_equal(rp2, rp)
    order_ok = all((np.diff(ci[rp[r]:rp[r + 1]]) >= 0).all() for r in range(R))
    if order_ok:
        assert np.array_equal(ci2, ci) and np.array_equal(v2.view(np.int32), v.view(np.int32))
    else:  # same multiset per row
        for r in range(R):
            a = sorted(zip(ci[rp[r]:rp[r + 1]].tolist(), v[rp[r]:rp[r + 1]].tolist()))
            b = sorted(zip(ci2[rp[r]:rp[r + 1]].tolist(), v2[rp[r]:rp[r + 1]].tolist()))
            assert a == b
