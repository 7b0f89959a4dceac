"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only *builds inputs*: CSR arrays (rowPtrs, colIdx, value) plus the
dense vectors x and y0, drawn from NumPy's PCG64 generator. It holds none of
the SpMV arithmetic and none of the format conversions; both the CPU oracle
and the CUDA library consume what it returns.

Workloads (all fp32 values, int32 indices, seed 0 unless stated):

* ``tiny_uniform``  4096 x 4096, exactly 8 nonzeros per row, columns uniform
  without replacement and sorted (32,768 nonzeros).
* ``laplace2d``     5-point Laplacian on a 2048 x 2048 grid, natural ordering
  r = i*2048 + j, Dirichlet boundary (neighbours outside the grid dropped),
  diagonal 4.0 and off-diagonals -1.0 (4,194,304 rows, 20,963,328 nonzeros).
* ``uniform_random`` 1,000,000 x 1,000,000, exactly 5 nonzeros per row,
  columns uniform without replacement, sorted (a 4 MB x vector gathered at
  random, the teaching example of "Introduction to sparse computing and
  performance bottleneck location", section "Building the problem framework").
* ``skewed``        2,000,000 x 2,000,000; row lengths uniform in [10, 20]
  except 200 rows (chosen without replacement) with lengths uniform in
  [1000, 5000]; columns uniform without replacement, sorted.
* ``stencil27``     27-point stencil on a 160^3 grid, Dirichlet boundary,
  off-diagonals uniform in [0.5, 1.5), diagonal = 1 + sum of the row's
  off-diagonal magnitudes (diagonally dominant); 4,096,000 rows, 109,215,352
  nonzeros.

In every workload x and y0 are uniform in [-1, 1).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "CSRInput",
    "WORKLOADS",
    "fig14_1_dense",
    "make_workload",
    "random_csr",
    "laplace2d",
    "stencil27",
    "uniform_rows",
    "skewed",
    "vectors",
]


@dataclass
class CSRInput:
    """One synthetic problem: a CSR matrix plus the vectors x and y0."""

    name: str
    num_rows: int
    num_cols: int
    row_ptrs: np.ndarray  # int32, num_rows + 1
    col_idx: np.ndarray  # int32, nnz
    value: np.ndarray  # float32, nnz
    x: np.ndarray  # float32, num_cols
    y0: np.ndarray  # float32, num_rows

    @property
    def nnz(self) -> int:
        return int(self.col_idx.shape[0])


def fig14_1_dense() -> np.ndarray:
    """The 4x4 example matrix of Fig. 14.1 in the PMPP notes "Sparse Matrices
    and Basic Formats (COO and CSR)" (rows eq0..eq3, columns x0..x3)."""
    return np.array(
        [[1, 7, 0, 0],
         [5, 0, 3, 9],
         [0, 2, 8, 0],
         [0, 0, 0, 6]], dtype=np.float32)


def _row_ptrs_from_lengths(lens: np.ndarray) -> np.ndarray:
    rp = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    np.cumsum(lens, out=rp[1:])
    if rp[-1] > np.iinfo(np.int32).max:
        raise ValueError("nnz exceeds int32")
    return rp.astype(np.int32)


def _distinct_sorted_columns(rng: np.random.Generator, lens: np.ndarray,
                             num_cols: int) -> np.ndarray:
    """Per row, ``lens[r]`` distinct columns drawn uniformly from
    [0, num_cols), returned row after row, ascending within each row.

    Draws all columns at once, then redraws any repeated (row, column) pair
    until none is left; the result depends only on the generator state."""
    lens = np.asarray(lens, dtype=np.int64)
    if lens.size and lens.max() > num_cols:
        raise ValueError("a row is longer than the number of columns")
    rows = np.repeat(np.arange(lens.shape[0], dtype=np.int64), lens)
    key = rows * num_cols + rng.integers(0, num_cols, rows.shape[0], dtype=np.int64)
    while True:
        key.sort()
        dup = np.flatnonzero(key[1:] == key[:-1]) + 1
        if dup.size == 0:
            break
        key[dup] = (key[dup] // num_cols) * num_cols + rng.integers(
            0, num_cols, dup.size, dtype=np.int64)
    return (key % num_cols).astype(np.int32)


def vectors(rng: np.random.Generator, num_rows: int, num_cols: int):
    x = rng.uniform(-1.0, 1.0, num_cols).astype(np.float32)
    y0 = rng.uniform(-1.0, 1.0, num_rows).astype(np.float32)
    return x, y0


def uniform_rows(name: str, n: int, per_row: int, seed: int = 0) -> CSRInput:
    """n x n, exactly ``per_row`` distinct sorted uniform columns per row.
    Draw order: columns, values, x, y0."""
    rng = np.random.default_rng(seed)
    lens = np.full(n, per_row, dtype=np.int64)
    col = _distinct_sorted_columns(rng, lens, n)
    val = rng.uniform(-1.0, 1.0, col.shape[0]).astype(np.float32)
    x, y0 = vectors(rng, n, n)
    return CSRInput(name, n, n, _row_ptrs_from_lengths(lens), col, val, x, y0)


def skewed(n: int = 2_000_000, n_long: int = 200, short=(10, 20),
           long=(1000, 5000), seed: int = 0, name: str = "skewed") -> CSRInput:
    """Row lengths uniform in ``short`` (inclusive) except ``n_long`` rows
    (chosen without replacement) with lengths uniform in ``long``.
    Draw order: short lengths, long-row choice, long lengths, columns,
    values, x, y0."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(short[0], short[1] + 1, n, dtype=np.int64)
    long_rows = rng.choice(n, n_long, replace=False)
    lens[long_rows] = rng.integers(long[0], long[1] + 1, n_long, dtype=np.int64)
    col = _distinct_sorted_columns(rng, lens, n)
    val = rng.uniform(-1.0, 1.0, col.shape[0]).astype(np.float32)
    x, y0 = vectors(rng, n, n)
    return CSRInput(name, n, n, _row_ptrs_from_lengths(lens), col, val, x, y0)


def _stencil(name: str, dims, offsets, draw_values, seed: int) -> CSRInput:
    """Grid stencil with Dirichlet boundary: a neighbour outside the grid is
    dropped. Rows in natural (row-major) order; within a row the columns are
    ascending because ``offsets`` is listed in ascending linear offset."""
    rng = np.random.default_rng(seed)
    dims = tuple(int(d) for d in dims)
    n = int(np.prod(dims))
    coords = np.unravel_index(np.arange(n, dtype=np.int64), dims)
    strides = np.array([int(np.prod(dims[i + 1:])) for i in range(len(dims))],
                       dtype=np.int64)
    m = len(offsets)
    valid = np.ones((n, m), dtype=bool)
    cols = np.empty((n, m), dtype=np.int64)
    for s, off in enumerate(offsets):
        lin = np.zeros(n, dtype=np.int64)
        for a, d in enumerate(off):
            c = coords[a] + d
            valid[:, s] &= (c >= 0) & (c < dims[a])
            lin += d * strides[a]
        cols[:, s] = np.arange(n, dtype=np.int64) + lin
    vals = draw_values(rng, n, m, valid)
    lens = valid.sum(axis=1)
    col = cols[valid].astype(np.int32)
    val = vals[valid].astype(np.float32)
    x, y0 = vectors(rng, n, n)
    return CSRInput(name, n, n, _row_ptrs_from_lengths(lens), col, val, x, y0)


def laplace2d(side: int = 2048, seed: int = 0, name: str = "laplace2d") -> CSRInput:
    """5-point Laplacian: diagonal 4.0, each in-grid neighbour -1.0."""
    offsets = [(-1, 0), (0, -1), (0, 0), (0, 1), (1, 0)]

    def draw(rng, n, m, valid):
        v = np.full((n, m), -1.0, dtype=np.float32)
        v[:, 2] = 4.0
        return v

    return _stencil(name, (side, side), offsets, draw, seed)


def stencil27(side: int = 160, seed: int = 0, name: str = "stencil27") -> CSRInput:
    """27-point stencil: off-diagonals uniform in [0.5, 1.5); the diagonal is
    1 + the sum (in float64, then rounded to float32) of the row's in-grid
    off-diagonal values. Draw order: one (n, 27) value block, x, y0."""
    offsets = [(a, b, c) for a in (-1, 0, 1) for b in (-1, 0, 1) for c in (-1, 0, 1)]
    center = offsets.index((0, 0, 0))

    def draw(rng, n, m, valid):
        v = rng.uniform(0.5, 1.5, (n, m)).astype(np.float32)
        off = valid.copy()
        off[:, center] = False
        diag = 1.0 + np.where(off, np.abs(v.astype(np.float64)), 0.0).sum(axis=1)
        v[:, center] = diag.astype(np.float32)
        return v

    return _stencil(name, (side, side, side), offsets, draw, seed)


def random_csr(seed: int, num_rows: int, num_cols: int, *, mean_len: float = 4.0,
               empty_frac: float = 0.0, long_rows: int = 0, long_len: int = 0,
               unsorted: bool = False, duplicates: bool = False,
               zeros_frac: float = 0.0, name: str = "random") -> CSRInput:
    """Small irregular CSR matrices for edge-case parity tests.

    Row lengths are Poisson(mean_len) capped at num_cols; a fraction of rows is
    forced empty; ``long_rows`` rows get ``long_len`` entries. Columns are
    distinct and sorted unless ``unsorted`` (shuffled within the row) or
    ``duplicates`` (drawn with replacement, so a column may repeat in a row).
    A fraction ``zeros_frac`` of the stored values is an explicit 0.0."""
    rng = np.random.default_rng(seed)
    lens = np.minimum(rng.poisson(mean_len, num_rows), num_cols).astype(np.int64)
    if num_rows:
        lens[rng.random(num_rows) < empty_frac] = 0
        if long_rows:
            pick = rng.choice(num_rows, min(long_rows, num_rows), replace=False)
            lens[pick] = min(long_len, num_cols) if not duplicates else long_len
    if num_cols == 0:
        lens[:] = 0
    if duplicates:
        col = rng.integers(0, max(num_cols, 1), int(lens.sum()), dtype=np.int64).astype(np.int32)
    else:
        col = _distinct_sorted_columns(rng, lens, num_cols)
        if unsorted:
            rp = _row_ptrs_from_lengths(lens)
            for r in range(num_rows):
                seg = col[rp[r]:rp[r + 1]]
                rng.shuffle(seg)
    val = rng.uniform(-1.0, 1.0, col.shape[0]).astype(np.float32)
    if zeros_frac > 0 and val.size:
        val[rng.random(val.size) < zeros_frac] = 0.0
    x, y0 = vectors(rng, num_rows, num_cols)
    return CSRInput(name, num_rows, num_cols, _row_ptrs_from_lengths(lens), col, val, x, y0)


def spd_random(seed: int, n: int, pairs_per_row: float = 3.0, name: str = "spd_random"
               ) -> CSRInput:
    """Symmetric, strictly diagonally dominant n x n matrix (so symmetric
    positive definite): about ``pairs_per_row`` random off-diagonal pairs
    (i, j) / (j, i) per row, both with the same value uniform in [-1, -0.1);
    a pair drawn twice holds the sum of its draws. Diagonal = 1 + the sum (in
    float64, then rounded to float32) of the row's |off-diagonal| values.
    Columns ascending within a row. Draw order: pair rows, pair columns,
    pair values, x, y0."""
    rng = np.random.default_rng(seed)
    m = int(round(pairs_per_row * n))
    i = rng.integers(0, n, m)
    j = rng.integers(0, n, m)
    v = rng.uniform(-1.0, -0.1, m).astype(np.float32)
    keep = i != j
    i, j, v = i[keep], j[keep], v[keep]
    rows = np.concatenate([i, j])
    cols = np.concatenate([j, i])
    vals = np.concatenate([v, v]).astype(np.float64)
    key = rows.astype(np.int64) * n + cols
    uk, inv = np.unique(key, return_inverse=True)
    acc = np.zeros(uk.shape[0], np.float64)
    np.add.at(acc, inv, vals)
    off_r, off_c = uk // n, uk % n
    off_v = acc.astype(np.float32)
    diag = 1.0 + np.bincount(off_r, weights=np.abs(off_v.astype(np.float64)), minlength=n)
    r_all = np.concatenate([off_r, np.arange(n)])
    c_all = np.concatenate([off_c, np.arange(n)])
    v_all = np.concatenate([off_v, diag.astype(np.float32)])
    order = np.lexsort((c_all, r_all))
    lens = np.bincount(r_all, minlength=n).astype(np.int64)
    x, y0 = vectors(rng, n, n)
    return CSRInput(name, n, n, _row_ptrs_from_lengths(lens), c_all[order].astype(np.int32),
                    v_all[order].astype(np.float32), x, y0)


def hashed_entries(k0: int, k1: int, num_cols: int):
    """Columns and values of nonzeros k0 .. k1-1 of a large matrix defined by
    closed forms (no stored randomness, so any slice can be made on demand):
    column = (k * 40503 + 17) mod numCols, value = ((k * 2246822519) mod 65521)
    / 65521 - 0.5 in float32."""
    k = np.arange(k0, k1, dtype=np.int64)
    col = ((k * 40503 + 17) % num_cols).astype(np.int32)
    val = (((k * 2246822519) % 65521).astype(np.float64) / 65521.0 - 0.5).astype(np.float32)
    return col, val


def hashed_vector(n: int, salt: int) -> np.ndarray:
    """x or y0 of the large matrix: ((i * 1103515245 + salt) mod 4093) / 4093 - 0.5."""
    i = np.arange(n, dtype=np.int64)
    return (((i * 1103515245 + salt) % 4093).astype(np.float64) / 4093.0 - 0.5).astype(np.float32)


WORKLOADS = {
    "tiny_uniform": lambda seed=0: uniform_rows("tiny_uniform", 4096, 8, seed),
    "laplace2d": lambda seed=0: laplace2d(2048, seed),
    "uniform_random": lambda seed=0: uniform_rows("uniform_random", 1_000_000, 5, seed),
    "skewed": lambda seed=0: skewed(seed=seed),
    "stencil27": lambda seed=0: stencil27(160, seed),
}


def make_workload(name: str, seed: int = 0) -> CSRInput:
    """Build one of the five named workloads (see the module docstring)."""
    try:
        return WORKLOADS[name](seed)
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None
