"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the oracle's C source (a transposed or shifted operand,
a wrong sign, a dropped absolute value, an unstable placement, a wrong run
order, a run split too eagerly, a run value taken from the wrong run, a dropped
entry), builds it with gcc on the CPU, runs the pins of test_oracle_pins.py on
it, and expects at least one of them to fail.  Every planted mistake keeps all
memory accesses in bounds, so a mutant can only compute wrong numbers."""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "vs_oracle.c")

MUTANTS = {
    # or_spmm_ab: columns of B taken in reverse (an index mistake)
    "ab_operand_column": ("            double b = B[j * ldb + c];\n            out[i * ldo + c] += a * b;",
                          "            double b = B[j * ldb + (w - 1 - c)];\n            out[i * ldo + c] += a * b;"),
    # or_spmm_ab: the product subtracted (a sign mistake)
    "ab_sign": ("            out[i * ldo + c] += a * b;\n            D[i * ldo + c]",
                "            out[i * ldo + c] -= a * b;\n            D[i * ldo + c]"),
    # or_spmm_ab: the error scale without absolute values
    "ab_scale_without_abs": ("            D[i * ldo + c] += fabs(a) * fabs(b);",
                             "            D[i * ldo + c] += a * b;"),
    # or_spmm_ba: the sign of A dropped
    "ba_sign_of_a": ("            out[c * ldo + j] += b * a;",
                     "            out[c * ldo + j] += b * fabs(a);"),
    # or_spmm_ba: reads B at the output column instead of the contracted row
    "ba_transposed_operand": ("            double b = B[c * ldb + i];\n            out[c * ldo + j] += b * a;",
                              "            double b = B[c * ldb + (j < i ? j : i)];\n            out[c * ldo + j] += b * a;"),
    # or_csr_build: entries placed in reverse input order (not stable)
    "csr_unstable": ("    for (int64_t t = 0; t < nnz; t++) {\n        int64_t p = count[maj[t]];",
                     "    for (int64_t t = nnz - 1; t >= 0; t--) {\n        int64_t p = count[maj[t]];"),
    # or_csr_build: the last entry of every slice loses its value
    "csr_drops_value": ("        if (val_bytes > 0) memcpy(dst + p * val_bytes, src + t * val_bytes, (size_t)val_bytes);",
                        "        if (val_bytes > 0 && p + 1 != ptr[maj[t] + 1]) memcpy(dst + p * val_bytes, src + t * val_bytes, (size_t)val_bytes);\n"
                        "        else if (val_bytes > 0) memset(dst + p * val_bytes, 0, (size_t)val_bytes);"),
    # or_vcs_build: runs in descending value order
    "vcs_value_order": ("    if (a->vkey != b->vkey) return a->vkey < b->vkey ? -1 : 1;",
                        "    if (a->vkey != b->vkey) return a->vkey < b->vkey ? 1 : -1;"),
    # or_vcs_build: a new run at every index change (runs split)
    "vcs_split_runs": ("|| e[k].vkey != e[k - 1].vkey;",
                       "|| e[k].vkey != e[k - 1].vkey || e[k].mnr != e[k - 1].mnr;"),
    # or_vcs_build: indices ordered by input position instead of ascending
    "vcs_index_order": ("    if (a->mnr != b->mnr) return a->mnr < b->mnr ? -1 : 1;\n    if (a->t != b->t)",
                        "    if (a->t != b->t) return a->t < b->t ? -1 : 1;\n    if (a->mnr != b->mnr)"),
    # or_vcs_triples: every entry of a slice carries the slice's first run value
    "vcs_triples_run_value": ("                ta[k] = (double)values[r];",
                              "                ta[k] = (double)values[major_ptr[m]];"),
    # or_spmm_ab_rows: the sampled rows read the wrong column of B
    "ab_rows_operand_column": ("            double b = B[j * ldb + c];\n            out[s * w + c] += a * b;",
                               "            double b = B[j * ldb + (w - 1 - c)];\n            out[s * w + c] += a * b;"),
    # or_spmm_ba_cols: the sampled columns drop the sign of A
    "ba_cols_sign_of_a": ("            out[s * w + c] += b * a;",
                          "            out[s * w + c] += b * fabs(a);"),
    # or_view_triples: the row scaling indexed by the column (a transposed statistic)
    "view_scale_index": ("        if (row_scale) v = row_scale[ti[k]] * v;",
                         "        if (row_scale) v = row_scale[tj[k] < ti[k] ? tj[k] : ti[k]] * v;"),
    # or_view_triples: log instead of log1p
    "view_log_not_log1p": ("        if (map == 1) v = log1p(v);",
                           "        if (map == 1) v = log(v > 0 ? v : 1.0);"),
    # or_spmm_slices: the merge of private outputs leaves out the last thread
    "slices_merge_drops_thread": ("            for (int k = 0; k < T; k++) {\n                const double *y = priv",
                                  "            for (int k = 0; k + 1 < T; k++) {\n                const double *y = priv"),
    # or_spmm_slices: a VCS run's value taken from the entry index (wrong array index)
    "slices_value_by_entry": ("                for (int64_t k = k0; k < k1; k++) {\n                    const double *x = X + (int64_t)idx[k] * w;",
                              "                for (int64_t k = k0; k < k1; k++) {\n                    a = vals[k < hi ? k : q];\n                    const double *x = X + (int64_t)idx[k] * w;"),
    # or_spmm_slices: each thread's slice range ends one slice early
    "slices_range_short": ("        if (k == T - 1) s1 = n_major;",
                           "        if (k == T - 1) s1 = n_major;\n        if (s1 > s0) s1 -= 1;"),
}


def _pin_battery():
    """Every pin of test_oracle_pins with its parameter values."""
    yield pins.test_golden_worked_example_layouts
    for layout in ("csr", "csc", "vcsr", "vcsc"):
        yield lambda layout=layout: pins.test_golden_worked_example_products(layout)
    yield pins.test_golden_signed_zero_runs
    for seed in (0, 1, 2):
        for row in (True, False):
            yield lambda seed=seed, row=row: pins.test_csr_build_is_stable_counting_sort(seed, row)
    yield pins.test_csr_keeps_input_order_under_permutation
    for seed in (0, 1, 2, 3):
        for values in ("counts", "signed_zero", "normal"):
            yield lambda seed=seed, values=values: pins.test_vcs_build_matches_bruteforce(seed, values)
    yield pins.test_vcs_invariants_on_tiny_workload
    yield pins.test_vcs_is_independent_of_input_order
    for seed in (0, 1):
        yield lambda seed=seed: pins.test_products_equal_dense_matmul_exactly(seed)
    yield pins.test_dot_product_identity
    yield pins.test_permutation_matrix_permutes_exactly
    yield pins.test_empty_rows_zero_width_and_empty_matrix
    yield pins.test_duplicates_are_summed
    yield pins.test_vcs_and_csr_products_agree_on_workload
    yield pins.test_sampled_products_match_full
    yield pins.test_golden_view_worked_example
    yield pins.test_view_closed_forms
    for threads in (1, 3, 8):
        yield lambda threads=threads: pins.test_threaded_products_match_serial(threads)
    yield pins.test_threaded_products_equal_dense_matmul_exactly


def _failing_pins() -> int:
    failed = 0
    for pin in _pin_battery():
        try:
            pin()
        except Exception:  # an assertion, or an error the planted mistake provoked
            failed += 1
    return failed


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is needed to build the mutants")
    return tmp_path_factory.mktemp("oracle_mutants")


def test_unmodified_oracle_passes_every_pin():
    assert _failing_pins() == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, workdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the planted mistake's anchor is not unique"
    path_c = os.path.join(workdir, f"{name}.c")
    path_so = os.path.join(workdir, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", path_c, "-o", path_so, "-lm"], check=True)
    with oracle.use_library(path_so):
        caught = _failing_pins()
    assert caught > 0, f"no pin catches the planted mistake {name!r}"
