"""Pins of the oracle's conjugate gradient for A·X + Y = 0 ('Sparse Matrices
and Basic Formats (COO and CSR)', section 'Background & SpMV': the iterative
solver for positive-definite A that motivates the SpMV), against facts that
the mathematics fixes independently of the code: closed-form eigenpairs of
the Dirichlet Laplacian, finite termination in as many steps as there are
distinct eigenvalues, a dense direct solve, and the monotone decrease of the
A-norm error."""
import numpy as np
import pytest

import synth


def dense(inp):
    A = np.zeros((inp.num_rows, inp.num_cols), np.float64)
    for r in range(inp.num_rows):
        for k in range(inp.row_ptrs[r], inp.row_ptrs[r + 1]):
            A[r, inp.col_idx[k]] += float(inp.value[k])
    return A


def laplace_eigvec(m, p, q):
    """Eigenpair (p, q) of the 5-point Dirichlet Laplacian (diagonal 4,
    neighbours -1) on an m x m grid: v(i, j) = sin((i+1) p pi/(m+1))
    sin((j+1) q pi/(m+1)), lambda = 4 - 2 cos(p pi/(m+1)) - 2 cos(q pi/(m+1))."""
    t = np.pi / (m + 1)
    i = np.arange(1, m + 1)
    v = np.outer(np.sin(i * p * t), np.sin(i * q * t)).ravel()
    return v, 4.0 - 2.0 * np.cos(p * t) - 2.0 * np.cos(q * t)


@pytest.mark.parametrize("m,p,q", [(7, 1, 1), (7, 2, 5), (12, 3, 3), (9, 9, 1)])
def test_laplacian_eigenvector_converges_in_one_step(orc, m, p, q):
    """Y an eigenvector of A with eigenvalue lambda: the first step length is
    1/lambda and X_1 = -Y/lambda solves A·X + Y = 0 (to the rounding of Y to
    fp32)."""
    lap = synth.laplace2d(m)
    v, lam = laplace_eigvec(m, p, q)
    Y = v.astype(np.float32)
    res = orc.cg(lap.row_ptrs, lap.col_idx, lap.value, Y, max_iter=50, tol=1e-5)
    assert res["iterations"] == 1 and res["status"] == 0
    np.testing.assert_allclose(res["x"], -Y.astype(np.float64) / lam, rtol=0,
                               atol=1e-6 * np.abs(Y).max() / lam)
    assert res["gnorm"][1] <= 1e-6 * np.linalg.norm(Y.astype(np.float64))


def test_finite_termination_distinct_eigenvalues(orc):
    """A diagonal matrix with 4 distinct eigenvalues: CG ends in exactly 4
    steps (the Krylov space has dimension 4)."""
    n = 40
    diag = np.array([1.0, 2.0, 5.0, 10.0])[np.arange(n) % 4]
    rp = np.arange(n + 1, dtype=np.int32)
    ci = np.arange(n, dtype=np.int32)
    rng = np.random.default_rng(3)
    Y = rng.uniform(-1, 1, n).astype(np.float32)
    res = orc.cg(rp, ci, diag.astype(np.float32), Y, max_iter=20, tol=1e-12)
    assert res["iterations"] == 4 and res["status"] == 0
    g = res["gnorm"] / np.linalg.norm(Y.astype(np.float64))
    assert g[4] <= 1e-12 and g[3] > 1e-6
    np.testing.assert_allclose(res["x"], -Y.astype(np.float64) / diag, rtol=1e-12)


def test_three_laplacian_modes_three_steps(orc):
    """Y a combination of 3 eigenvectors of distinct eigenvalues: 3 steps.
    Rounding Y to fp32 leaves ~6e-8 of every other mode, which the degree-3
    residual polynomial (roots at the 3 eigenvalues) amplifies by up to ~500
    at the top of the spectrum, so the third residual is ~1e-5, not 0; the
    second is of order 1."""
    m = 10
    lap = synth.laplace2d(m)
    parts = [laplace_eigvec(m, p, q) for p, q in ((1, 1), (2, 3), (5, 4))]
    Y64 = sum(c * v for c, (v, _) in zip((1.0, -0.5, 0.25), parts))
    Y = Y64.astype(np.float32)
    res = orc.cg(lap.row_ptrs, lap.col_idx, lap.value, Y, max_iter=30, tol=1e-4)
    assert res["iterations"] == 3 and res["status"] == 0
    g = res["gnorm"] / np.linalg.norm(Y.astype(np.float64))
    assert g[3] <= 1e-4 and g[2] > 0.1
    A = dense(lap)
    assert np.linalg.norm(A @ res["x"] + Y) <= 1e-4 * np.linalg.norm(Y.astype(np.float64))


@pytest.mark.parametrize("which", ["laplace", "spd"])
def test_matches_dense_direct_solve(orc, which):
    inp = synth.laplace2d(6) if which == "laplace" else synth.spd_random(5, 150)
    A = dense(inp)
    Y = inp.y0
    want = np.linalg.solve(A, -Y.astype(np.float64))
    res = orc.cg(inp.row_ptrs, inp.col_idx, inp.value, Y, max_iter=inp.num_rows, tol=1e-13)
    assert res["status"] == 0 and res["iterations"] <= inp.num_rows
    np.testing.assert_allclose(res["x"], want, rtol=0, atol=1e-10 * np.abs(want).max())


def test_a_norm_error_decreases_and_recurrence_matches(orc):
    """||X_k - X*||_A falls at every step (CG minimises it over the Krylov
    space), and the recurrence gradient equals A·X_k + Y."""
    inp = synth.spd_random(7, 300, pairs_per_row=4.0)
    A = dense(inp)
    Y = inp.y0.astype(np.float64)
    xs = np.linalg.solve(A, -Y)
    prev = np.inf
    for k in range(1, 12):
        res = orc.cg(inp.row_ptrs, inp.col_idx, inp.value, inp.y0, max_iter=k, tol=0.0)
        assert res["iterations"] == k and res["status"] == 1
        e = res["x"] - xs
        en = float(np.sqrt(e @ A @ e))
        assert en < prev
        prev = en
        true_g = np.linalg.norm(A @ res["x"] + Y)
        assert abs(res["gnorm"][k] - true_g) <= 1e-10 * np.linalg.norm(Y)


def test_starting_guess(orc):
    inp = synth.spd_random(9, 120)
    A = dense(inp)
    want = np.linalg.solve(A, -inp.y0.astype(np.float64))
    res = orc.cg(inp.row_ptrs, inp.col_idx, inp.value, inp.y0, X0=inp.x, max_iter=200,
                 tol=1e-12)
    np.testing.assert_allclose(res["x"], want, atol=1e-9 * np.abs(want).max())
    # g_0 = A·X_0 + Y
    assert res["gnorm"][0] == pytest.approx(
        np.linalg.norm(A @ inp.x.astype(np.float64) + inp.y0), rel=1e-12)


def test_degenerate_cases(orc):
    lap = synth.laplace2d(4)
    n = lap.num_rows
    res = orc.cg(lap.row_ptrs, lap.col_idx, lap.value, np.zeros(n, np.float32), max_iter=10)
    assert res["iterations"] == 0 and res["status"] == 0 and not res["x"].any()
    # max_iter = 0: only g_0
    res = orc.cg(lap.row_ptrs, lap.col_idx, lap.value, lap.y0, max_iter=0, tol=1e-9)
    assert res["iterations"] == 0 and res["status"] == 1
    # not positive definite: -I
    rp = np.arange(n + 1, dtype=np.int32)
    res = orc.cg(rp, np.arange(n, dtype=np.int32), -np.ones(n, np.float32), lap.y0,
                 max_iter=10, tol=1e-9)
    assert res["status"] == 2 and res["iterations"] == 0
    # empty system
    res = orc.cg(np.zeros(1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32),
                 np.zeros(0, np.float32), max_iter=5)
    assert res["iterations"] == 0 and res["status"] == 0
