"""Pins of the oracle's SpMV with 8-byte values ('Introduction to sparse
computing and performance bottleneck location', section 'Building the
problem framework': values and x entries of 4 or 8 bytes) against exact
rational arithmetic and hand-checked cases."""
from fractions import Fraction

import numpy as np
import pytest

import synth


def exact_rows(inp, value, x, y0):
    """y_i = y0_i + sum a x in exact rationals, rounded once to fp64."""
    out = []
    for r in range(inp.num_rows):
        acc = Fraction(float(y0[r]))
        for k in range(inp.row_ptrs[r], inp.row_ptrs[r + 1]):
            acc += Fraction(float(value[k])) * Fraction(float(x[inp.col_idx[k]]))
        out.append(float(acc))
    return np.array(out)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_exact_rationals(orc, seed):
    inp = synth.random_csr(seed, 70, 60, mean_len=9, empty_frac=0.1, long_rows=2, long_len=55,
                           duplicates=seed == 2)
    rng = np.random.default_rng(100 + seed)
    value = rng.standard_normal(inp.nnz) * np.exp(rng.uniform(-20, 20, inp.nnz))
    x = rng.standard_normal(inp.num_cols)
    y0 = rng.standard_normal(inp.num_rows)
    y, mag = orc.spmv_csr_f64(inp.row_ptrs, inp.col_idx, value, x, y0)
    want = exact_rows(inp, value, x, y0)
    # compensated sum: within two roundings of the exact value
    assert np.all(np.abs(y - want) <= 2 * 2.0**-53 * np.abs(want) + 1e-300)
    assert np.all(mag >= np.abs(y0)) and np.all(mag + 1e-300 >= np.abs(y - y0) * (1 - 1e-15))


def test_fig14_1(orc):
    rp, ci, va = orc.dense_to_csr(synth.fig14_1_dense())
    y, _ = orc.spmv_csr_f64(rp, ci, va.astype(np.float64), np.array([1.0, 2, 3, 4]),
                            np.zeros(4))
    assert y.tolist() == [15.0, 50.0, 28.0, 24.0]


def test_needs_eight_byte_values(orc):
    """1 + 2^-40 is not a float32: a 4-byte value path would give exactly 2."""
    rp = np.array([0, 2], np.int32)
    ci = np.array([0, 1], np.int32)
    v = np.array([1 + 2.0**-40, 1 + 2.0**-40])
    y, _ = orc.spmv_csr_f64(rp, ci, v, np.ones(2), np.zeros(1))
    assert y[0] == 2 + 2.0**-39


def test_cancellation_needs_compensation(orc):
    """1e16 + 1 - 1e16: a plain fp64 running sum gives 0; the exact value is 1."""
    rp = np.array([0, 3], np.int32)
    ci = np.array([0, 1, 2], np.int32)
    y, _ = orc.spmv_csr_f64(rp, ci, np.array([1e16, 1.0, -1e16]), np.ones(3), np.zeros(1))
    assert y[0] == 1.0
    # and the product error term: (1 + 2^-30)^2 = 1 + 2^-29 + 2^-60, minus 1
    rp = np.array([0, 2], np.int32)
    ci = np.array([0, 1], np.int32)
    a = 1 + 2.0**-30
    y, _ = orc.spmv_csr_f64(rp, ci, np.array([a, -1.0]), np.array([a, 1.0]), np.zeros(1))
    assert y[0] == 2.0**-29 + 2.0**-60
