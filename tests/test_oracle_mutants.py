"""The pins are strong enough: plant a plausible mistake in a copy of the
oracle's C source (a dropped term, a wrong index, a reversed order, a
transposed layout), build it on the CPU, and check that at least one pin
test fails against the mutant. The real oracle is never modified."""
import os

import numpy as np
import pytest

import oracle
from oracle import build as obuild
import test_oracle_pins as pins

SRC = open(obuild.SRC).read()

MUTANTS = {
    "csr_drops_y0": ("y[r] = (double)y0[r] + s;\n        if (mag)", "y[r] = s;\n        if (mag)"),
    "csr_skips_first_entry": ("for (int64_t r = 0; r < R; ++r) {\n        double s = 0.0, a = 0.0;\n"
                              "        for (int64_t k = rowPtrs[r]; k",
                              "for (int64_t r = 0; r < R; ++r) {\n        double s = 0.0, a = 0.0;\n"
                              "        for (int64_t k = rowPtrs[r] + 1; k"),
    "csr_wrong_sign": ("            s += p;\n            a += fabs(p);\n        }\n        y[r] = (double)y0[r] + s;\n        if (mag)",
                       "            s -= p;\n            a += fabs(p);\n        }\n        y[r] = (double)y0[r] + s;\n        if (mag)"),
    "ell_row_major": ("                   int32_t *ellCol, float *ellVal) {\n"
                      "    for (int64_t r = 0; r < R; ++r) {\n"
                      "        int64_t len = (int64_t)rowPtrs[r + 1] - rowPtrs[r];\n"
                      "        nnzPerRow[r] = (int32_t)len;\n"
                      "        for (int64_t t = 0; t < K; ++t) {\n"
                      "            int64_t i = t * R + r;",
                      "                   int32_t *ellCol, float *ellVal) {\n"
                      "    for (int64_t r = 0; r < R; ++r) {\n"
                      "        int64_t len = (int64_t)rowPtrs[r + 1] - rowPtrs[r];\n"
                      "        nnzPerRow[r] = (int32_t)len;\n"
                      "        for (int64_t t = 0; t < K; ++t) {\n"
                      "            int64_t i = r * K + t;"),
    "ell_pad_col_zero": ("                ellCol[i] = -1;\n                ellVal[i] = 0.0f;\n            }\n        }\n    }\n}",
                         "                ellCol[i] = 0;\n                ellVal[i] = 0.0f;\n            }\n        }\n    }\n}"),
    "jds_ascending": ("for (int64_t len = maxLen; len >= 0; --len) {\n        first[len] = acc;",
                      "for (int64_t len = 0; len <= maxLen; ++len) {\n        first[len] = acc;"),
    "jds_iterptr_off_by_one": ("longer -= count[t + 1];", "longer -= count[t];"),
    "jds_unstable": ("    for (int64_t r = 0; r < R; ++r) {\n        int64_t len = rowPtrs[r + 1] - rowPtrs[r];\n        perm[first[len]] = (int32_t)r;",
                     "    for (int64_t r = R - 1; r >= 0; --r) {\n        int64_t len = rowPtrs[r + 1] - rowPtrs[r];\n        perm[first[len]] = (int32_t)r;"),
    "jds_spmv_no_unpermute": ("y[perm[s]] += acc;", "y[s] += acc;"),
    "hyb_width_off_by_one": ("int64_t inEll = len < K ? len : K;",
                             "int64_t inEll = len < K ? len : (K > 0 ? K - 1 : 0);"),
    "coo_row_shift": ("rowIdx[k] = (int32_t)r;", "rowIdx[k] = (int32_t)(r > 0 ? r - 1 : 0);"),
    "validate_rejects_empty_rows": ("if (rowPtrs[r + 1] < rowPtrs[r]) return OR_BAD_ROWPTRS;",
                                    "if (rowPtrs[r + 1] <= rowPtrs[r]) return OR_BAD_ROWPTRS;"),
    "validate_col_off_by_one": ("(int64_t)colIdx[k] >= C", "(int64_t)colIdx[k] > C"),
    "stats_sample_variance": ("*var = R > 0 ? ss / (double)R : 0.0;",
                              "*var = R > 1 ? ss / (double)(R - 1) : 0.0;"),
    "auto_width_strict": ("if (100 * cum >= 99 * R) break;", "if (100 * cum > 99 * R) break;"),
    "cg_alpha_uses_dd": ("double alpha = gg / dq;", "double alpha = gg / dot_f64(R, d, d);"),
    "cg_beta_inverted": ("double beta = ggNew / gg;", "double beta = gg / ggNew;"),
    "cg_gradient_sign": ("            g[i] += alpha * q[i];", "            g[i] -= alpha * q[i];"),
    "cg_direction_sign": ("d[i] = -g[i] + beta * d[i];", "d[i] = -g[i] - beta * d[i];"),
    "cg_drops_y": ("        g[i] += (double)Y[i];", "        g[i] += 0.0 * (double)Y[i];"),
    "cg_no_restart_from_x0": ("X[i] = X0 ? (double)X0[i] : 0.0;", "X[i] = 0.0;"),
    "xblock_global_column": ("xbCol[i] = (uint16_t)(colIdx[k] - c * B);",
                             "xbCol[i] = (uint16_t)(colIdx[k]);"),
    "xblock_no_padding": ("slots += (cnt[c] + 3) / 4 * 4;", "slots += cnt[c];"),
    "xblock_rows_reversed": ("    if (xbRow) {\n        for (int64_t r = 0; r < R; ++r)",
                             "    if (xbRow) {\n        for (int64_t r = R - 1; r >= 0; --r)"),
    "xblock_spmv_drops_chunk_base": ("(double)x[c * B + xbCol[i]]", "(double)x[xbCol[i]]"),
    "f64_values_as_float": ("            double p = value[k] * x[colIdx[k]];\n"
                            "            double e = fma(value[k], x[colIdx[k]], -p);",
                            "            double p = (double)(float)value[k] * x[colIdx[k]];\n"
                            "            double e = fma((double)(float)value[k], x[colIdx[k]], -p);"),
    "f64_no_product_error": ("            c += e;", "            c += 0.0 * e;"),
    "f64_plain_sum": ("            neumaier_add(&s, &c, p);", "            s += p;"),
    "f64_drops_y0": ("double s = y0[r], c = 0.0, a = fabs(y0[r]);",
                     "double s = 0.0, c = 0.0, a = fabs(y0[r]);"),
    "csr_rows_y0_by_position": ("y[i] = (double)y0[r] + s;\n        mag[i] = a + fabs((double)y0[r]);",
                                "y[i] = (double)y0[i] + s;\n        mag[i] = a + fabs((double)y0[i]);"),
    "csr_rows_skips_first_entry": ("int64_t r = rows[i];\n        double s = 0.0, a = 0.0;\n"
                                   "        for (int64_t k = rowPtrs[r]; k",
                                   "int64_t r = rows[i];\n        double s = 0.0, a = 0.0;\n"
                                   "        for (int64_t k = rowPtrs[r] + 1; k"),
    "sell_row_major": ("                    int64_t i = slots + t * h + j;",
                       "                    int64_t i = slots + j * w + t;"),
    "sell_width_from_last_row": ("        int64_t w = rowPtrs[order[s0] + 1] - rowPtrs[order[s0]];",
                                 "        int64_t w = rowPtrs[order[s0 + h - 1] + 1] - rowPtrs[order[s0 + h - 1]];"),
}


def _pin_calls():
    calls = [(pins.test_fig14_1_csr, {}), (pins.test_fig14_1_coo, {}),
             (pins.test_fig14_1_ell, {}), (pins.test_fig14_1_ell_index_formula, {}),
             (pins.test_fig14_1_jds, {}), (pins.test_fig14_1_spmv_every_format, {}),
             (pins.test_fig14_1_hyb_width2, {}), (pins.test_hyb_schematic_counts, {}),
             (pins.test_validate, {}), (pins.test_hyb_auto_width_quantile, {}),
             (pins.test_select_outcomes_described_by_page, {})]
    calls += [(pins.test_spmv_matches_dense_brute_force, {"seed": 0, "case": c})
              for c in range(len(pins.CASES))]
    calls += [(pins.test_spmv_rows_matches_dense_brute_force, {"case": c})
              for c in range(len(pins.CASES))]
    calls += [(pins.test_laplace2d_closed_form, {"side": 5})]
    import test_oracle_sell as sell
    calls += [(sell.test_fig14_1_sections_of_two, {}), (sell.test_fig14_1_spmv, {})]
    calls += [(sell.test_round_trip_and_padding, {"idx": i, "S": 3}) for i in range(7)]
    import test_oracle_xblock as xbk
    calls += [(xbk.test_fig14_1_chunkings, {"case": c}) for c in range(3)]
    calls += [(xbk.test_single_chunk_is_coo, {"idx": i}) for i in (0, 5, 6)]
    calls += [(xbk.test_spmv_matches_dense, {"case": c, "B": 7}) for c in (2, 3)]
    calls += [(xbk.test_round_trip_and_invariants, {"idx": i, "B": 5}) for i in (0, 5, 6)]
    import test_oracle_f64 as f64
    calls += [(f64.test_matches_exact_rationals, {"seed": 0}), (f64.test_fig14_1, {}),
              (f64.test_needs_eight_byte_values, {}),
              (f64.test_cancellation_needs_compensation, {})]
    import test_oracle_cg as cg
    calls += [(cg.test_laplacian_eigenvector_converges_in_one_step, {"m": 7, "p": 2, "q": 5}),
              (cg.test_finite_termination_distinct_eigenvalues, {}),
              (cg.test_three_laplacian_modes_three_steps, {}),
              (cg.test_matches_dense_direct_solve, {"which": "spd"}),
              (cg.test_a_norm_error_decreases_and_recurrence_matches, {}),
              (cg.test_starting_guess, {}), (cg.test_degenerate_cases, {})]
    for i in range(7):
        calls += [(pins.test_round_trips_bit_exact, {"idx": i}),
                  (pins.test_layout_invariants, {"idx": i}),
                  (pins.test_row_stats, {"idx": i}),
                  (pins.test_format_spmvs_agree, {"idx": i})]
    return calls


def test_validate_accepts_empty_rows(orc):
    rp = np.array([0, 0, 2, 2, 3], np.int32)
    ci = np.array([0, 1, 2], np.int32)
    assert orc.validate(4, 3, rp, ci) == oracle.OK


def run_pins_against(lib_path):
    """Run every pin against the library at ``lib_path``; return the names of
    the pins that failed."""
    mut = oracle.Oracle(oracle.load(lib_path))
    failures = []
    for fn, kw in _pin_calls() + [(test_validate_accepts_empty_rows, {})]:
        try:
            fn(mut, **kw)
        except (AssertionError, MemoryError, ValueError, IndexError):
            failures.append(fn.__name__)
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    """A mutant that writes out of bounds may crash: it runs in a child
    process, and a crash counts as caught."""
    import subprocess
    import sys
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    out = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", out, str(src), "-lm"], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]\n"
            "import test_oracle_mutants as m\n"
            "f = m.run_pins_against(%r)\n"
            "print('FAILED_PINS', len(f), f)\n"
            "sys.exit(3 if f else 0)\n") % (here, os.path.dirname(here), out)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=300)
    assert res.returncode != 0, f"no pin caught mutant {name}: {res.stdout[-500:]}"
