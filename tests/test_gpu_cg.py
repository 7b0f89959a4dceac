"""GPU parity of the conjugate-gradient solve (A·X + Y = 0) through the C ABI
against the fp64 oracle.

Tolerances. The GPU keeps X, g, d, q in fp32 and sums inner products in
fp32 within a block, fp64 across blocks; the oracle is fp64 throughout.
  * First iterations: each step perturbs the iterate by a few fp32 roundings
    relative to its size, amplified at most by the condition number kappa of
    the small test matrices (kappa <= ~20 for the random SPD ones, ~400 for a
    32x32 Laplacian); after k <= 5 steps the iterates agree to
    1e-4 * max|X| (>= 10 * k * kappa * 2^-24 for kappa <= 20).
  * At the stop: the GPU's X must satisfy the oracle's own check in fp64,
    |A·X + Y| <= 5 * tol * |Y| (the fp32 recurrence residual drifts from the
    true one by O(kappa * 2^-24 * |Y|), far below tol = 1e-4 * |Y| here), and
    the iteration count is within 10% (+3) of the oracle's.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

FMTS = ("CSR", "COO", "ELL", "HYB", "JDS", "SELL")


@pytest.fixture(scope="module")
def sp():
    from conftest import build_library
    build_library()
    import spmv_sparse_storage_gb300 as sp
    torch.cuda.set_device(0)
    return sp


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def true_residual(orc, inp, X, Y):
    g, _ = orc.spmv_csr(inp.row_ptrs, inp.col_idx, inp.value, X.astype(np.float32), Y)
    return float(np.linalg.norm(g)) / max(float(np.linalg.norm(Y.astype(np.float64))), 1e-300)


def solve(sp, m, fmt, Y, X0, max_iter, tol):
    x = dev(X0)
    info = m.cg_solve(fmt, dev(Y), x, max_iter=max_iter, tol=tol)
    torch.cuda.synchronize()
    return x.cpu().numpy(), info


def matrix(sp, inp, formats=FMTS):
    m = sp.SparseMatrix(inp.num_rows, inp.num_cols, dev(inp.row_ptrs), dev(inp.col_idx),
                        dev(inp.value))
    for f in formats:
        if f != "CSR":
            m.convert(f)
    return m


CASES = {
    "laplace32": lambda: synth.laplace2d(32),
    "spd_1001": lambda: synth.spd_random(41, 1001, pairs_per_row=3.0),  # rows % 4 != 0
    "spd_4096": lambda: synth.spd_random(42, 4096, pairs_per_row=6.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_converges_like_the_oracle(sp, orc, case):
    inp = CASES[case]()
    Y = inp.y0
    X0 = np.zeros(inp.num_rows, np.float32)
    tol = 1e-4
    want = orc.cg(inp.row_ptrs, inp.col_idx, inp.value, Y, X0, max_iter=2000, tol=tol)
    assert want["status"] == 0
    with matrix(sp, inp) as m:
        for f in FMTS + ("AUTO",):
            X, info = solve(sp, m, f, Y, X0, 2000, tol)
            assert info["status"] == 0, (f, info)
            assert info["residual_norm"] <= tol * info["y_norm"] * (1 + 1e-6)
            assert info["y_norm"] == pytest.approx(np.linalg.norm(Y.astype(np.float64)),
                                                   rel=1e-6)
            assert true_residual(orc, inp, X, Y) <= 5 * tol, f
            k, kw = info["iterations"], want["iterations"]
            assert abs(k - kw) <= 0.1 * kw + 3, (f, k, kw)


@pytest.mark.parametrize("case", ["spd_1001", "spd_4096"])
@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_first_iterates_match(sp, orc, case, k):
    inp = CASES[case]()
    Y, X0 = inp.y0, inp.x  # a nonzero starting guess
    want = orc.cg(inp.row_ptrs, inp.col_idx, inp.value, Y, X0, max_iter=k, tol=0.0)
    assert want["iterations"] == k
    scale = np.abs(want["x"]).max()
    with matrix(sp, inp) as m:
        for f in FMTS:
            X, info = solve(sp, m, f, Y, X0, k, 0.0)
            assert info["iterations"] == k and info["status"] == 1, (f, info)
            err = np.abs(X.astype(np.float64) - want["x"]).max()
            assert err <= 1e-4 * scale, (f, k, err / scale)
            assert info["residual_norm"] == pytest.approx(want["gnorm"][k], rel=1e-4), f


@pytest.mark.parametrize("p,q", [(1, 1), (3, 7)])
def test_laplacian_eigenvector_one_step(sp, p, q):
    """Y an eigenvector of the 32x32 Dirichlet Laplacian (closed form): one
    step with alpha = 1/lambda gives X = -Y/lambda."""
    m_ = 32
    lap = synth.laplace2d(m_)
    t = np.pi / (m_ + 1)
    i = np.arange(1, m_ + 1)
    v = np.outer(np.sin(i * p * t), np.sin(i * q * t)).ravel()
    lam = 4.0 - 2.0 * np.cos(p * t) - 2.0 * np.cos(q * t)
    Y = v.astype(np.float32)
    with matrix(sp, lap, ("ELL", "SELL")) as m:
        for f in ("ELL", "SELL", "CSR"):
            X, info = solve(sp, m, f, Y, np.zeros_like(Y), 20, 1e-5)
            assert info["iterations"] == 1 and info["status"] == 0, (f, info)
            np.testing.assert_allclose(X, -Y / lam, rtol=0, atol=1e-5 * np.abs(Y).max() / lam)


def test_degenerate_and_errors(sp, orc):
    lap = synth.laplace2d(8)
    n = lap.num_rows
    with matrix(sp, lap, ("ELL",)) as m:
        X, info = solve(sp, m, "ELL", np.zeros(n, np.float32), np.zeros(n, np.float32), 10, 1e-6)
        assert info["iterations"] == 0 and info["status"] == 0 and not X.any()
        X, info = solve(sp, m, "ELL", lap.y0, lap.x, 0, 1e-6)
        assert info["iterations"] == 0 and info["status"] == 1
        assert np.array_equal(X, lap.x)  # maxIter 0 leaves the guess
        with pytest.raises(sp.SpmvError) as ei:
            m.cg_solve("SELL", dev(lap.y0), dev(lap.x))
        assert ei.value.code == sp.SPMV_ERR_NOT_CONVERTED
        buf = torch.zeros(2 * n, device="cuda")
        with pytest.raises(sp.SpmvError) as ei:
            m.cg_solve("ELL", buf[:n], buf[n // 2:n // 2 + n])
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        with pytest.raises(sp.SpmvError) as ei:
            m.cg_solve("ELL", dev(lap.y0), dev(lap.x), max_iter=-1)
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
        with pytest.raises(sp.SpmvError) as ei:
            m.cg_solve("ELL", dev(lap.y0), dev(lap.x), tol=float("nan"))
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG
    # -I is not positive definite: stops before the first update
    rp = np.arange(n + 1, dtype=np.int32)
    with sp.SparseMatrix(n, n, dev(rp), dev(np.arange(n, dtype=np.int32)),
                         dev(-np.ones(n, np.float32))) as m:
        m.convert("ELL")
        for f in ("ELL", "CSR"):
            X, info = solve(sp, m, f, lap.y0, np.zeros(n, np.float32), 10, 1e-6)
            assert info["status"] == 2 and info["iterations"] == 0, (f, info)
            assert not X.any()
    # non-square
    rect = synth.random_csr(5, 10, 12, mean_len=3)
    with sp.SparseMatrix(10, 12, dev(rect.row_ptrs), dev(rect.col_idx), dev(rect.value)) as m:
        with pytest.raises(sp.SpmvError) as ei:
            m.cg_solve("CSR", dev(np.zeros(10, np.float32)), dev(np.zeros(10, np.float32)))
        assert ei.value.code == sp.SPMV_ERR_INVALID_ARG


def test_full_size_laplace2d(sp, orc):
    """The bench's CG workload (2048x2048 Laplacian, ELL): 40 iterations from
    X = 0. Checked by properties that hold at any size: the GPU's recurrence
    residual equals the true |A·X + Y| recomputed in fp64 by the oracle (to
    fp32 drift, 1e-3 relative), and its decrease over 40 steps is within 2%
    of the oracle's fp64 run of the same 40 steps."""
    inp = synth.make_workload("laplace2d")
    Y = inp.y0
    X0 = np.zeros(inp.num_rows, np.float32)
    want = orc.cg(inp.row_ptrs, inp.col_idx, inp.value, Y, X0, max_iter=40, tol=0.0)
    with matrix(sp, inp, ("ELL",)) as m:
        X, info = solve(sp, m, "ELL", Y, X0, 40, 0.0)
    assert info["iterations"] == 40 and info["status"] == 1
    ynorm = np.linalg.norm(Y.astype(np.float64))
    tr = true_residual(orc, inp, X, Y) * ynorm
    assert abs(info["residual_norm"] - tr) <= 1e-3 * tr
    ratio_gpu = info["residual_norm"] / ynorm
    ratio_orc = want["gnorm"][40] / want["gnorm"][0]
    assert ratio_gpu == pytest.approx(ratio_orc, rel=0.02)
