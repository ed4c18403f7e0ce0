"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Each mutant is the oracle's C source with one small edit (a dropped term, a transposed
operand, a flipped sign, a reversed sum, a flipped filter, a swapped index).  It is
compiled into a temporary library, swapped in for the real one, and the pins of
``test_oracle_pins.py`` are run against it: at least one pin must fail.  Nothing here
touches a GPU.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

GEMM_PINS = [
    lambda: pins.test_left_identity_gives_B(37, 37, 53),
    lambda: pins.test_right_identity_gives_A(29, 41, 41),
    lambda: pins.test_permutation_permutes_rows_of_B(),
    lambda: pins.test_permutation_on_the_right_permutes_columns_of_A(),
    lambda: pins.test_all_ones_gives_K(7, 300, 5),
    lambda: pins.test_rank_one(64),
    lambda: pins.test_triangular_closed_forms_fix_operand_orientation(),
    lambda: pins.test_arithmetic_series_counts_every_term(5),
    lambda: pins.test_brute_force_4x4_small_integers_match_numpy_exactly(),
    lambda: pins.test_random_floats_match_numpy_float64(33, 65, 17),
    lambda: pins.test_sum_runs_over_k_ascending(),
    lambda: pins.test_entries_equal_full_product_bit_for_bit(),
]
GENERAL_PINS = [
    lambda: pins.test_general_with_alpha_one_beta_zero_is_the_product(),
    lambda: pins.test_general_beta_zero_never_reads_C(),
    lambda: pins.test_general_zero_product_scales_the_accumulator(),
    lambda: pins.test_general_closed_form_with_dyadic_weights(),
    lambda: pins.test_general_matches_numpy_float64(),
]
CONV_PINS = [
    lambda: pins.test_conv_all_ones_counts_taps(),
    lambda: pins.test_conv_delta_filter_is_a_shifted_crop(),
    lambda: pins.test_conv_matches_scipy_correlate(),
    lambda: pins.test_im2col_matches_numpy_sliding_windows(),
    lambda: pins.test_two_routes_to_the_convolution_agree_exactly(),
    lambda: pins.test_im2col_worked_example_from_the_pages(),
]

# (name, exact text in oracle.c, replacement, pins that must catch it)
MUTANTS = [
    ("drop_last_k", "for (int64_t k = 0; k < g->K; ++k) {", "for (int64_t k = 0; k + 1 < g->K; ++k) {", GEMM_PINS),
    ("skip_first_k", "for (int64_t k = 0; k < g->K; ++k) {", "for (int64_t k = 1; k < g->K; ++k) {", GEMM_PINS),
    ("reverse_k", "for (int64_t k = 0; k < g->K; ++k) {", "for (int64_t k = g->K - 1; k >= 0; --k) {", GEMM_PINS),
    ("minus_sign", "c[j] = c[j] + prod;", "c[j] = c[j] - prod;", GEMM_PINS),
    ("transposed_A", "(double)g->A[i * g->lda + k]", "(double)g->A[k * g->lda + i]", GEMM_PINS),
    ("transposed_B", "const double prod = a * (double)b[j];",
     "const double prod = a * (double)g->B[j * g->ldb + k];", GEMM_PINS),
    ("no_zero_init", "for (int64_t j = 0; j < g->N; ++j) c[j] = 0.0;", "", GEMM_PINS),
    ("entries_drop_last", "for (int64_t k = 0; k < e->K; ++k) {", "for (int64_t k = 0; k + 1 < e->K; ++k) {",
     GEMM_PINS),
    ("general_beta_times_alpha", "prod + beta * C[i * ldc + j]", "prod + alpha * C[i * ldc + j]", GENERAL_PINS),
    ("general_no_alpha", "const double prod = alpha * D[i * ldd + j];", "const double prod = D[i * ldd + j];",
     GENERAL_PINS),
    ("general_reads_C_always", "(beta != 0.0) ? prod + beta * C[i * ldc + j] : prod", "prod + beta * C[i * ldc + j]",
     GENERAL_PINS),
    ("conv_flipped_filter", "* R1 + r1) * R2 + r2) * R3 + r3;", "* R1 + r1) * R2 + r2) * R3 + (R3 - 1 - r3);",
     CONV_PINS),
    ("conv_drop_channel", "for (int64_t ci = 0; ci < c->Cin; ++ci)", "for (int64_t ci = 1; ci < c->Cin; ++ci)",
     CONV_PINS),
    ("im2col_swapped_taps", "(((ci * in[0] + (p0 + r0)) * in[1] + (p1 + r1))",
     "(((ci * in[0] + (p0 + r1)) * in[1] + (p1 + r0))", CONV_PINS),
    ("im2col_col_major_outputs", "col[r * ncols + n] = x[xidx];",
     "col[r * ncols + (((p3 * out[2] + p2) * out[1] + p1) * out[0] + p0)] = x[xidx];", CONV_PINS),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor for %s not found in oracle.c" % name
    mutated = src.replace(old, new, 1)
    path_c = tmp_path / (name + ".c")
    path_so = tmp_path / (name + ".so")
    path_c.write_text(mutated)
    subprocess.run(["gcc", *oracle.CFLAGS, str(path_c), "-o", str(path_so), "-lm"], check=True)
    return str(path_so)


_CHILD = r"""
import ctypes, sys
import numpy as np
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
import test_oracle_mutants as m
oracle._load()
mutant = ctypes.CDLL({so!r})
for fn in ("oracle_gemm", "oracle_gemm_entries", "oracle_gemm_general", "oracle_conv4d_direct", "oracle_im2col4d"):
    getattr(mutant, fn).argtypes = getattr(oracle._lib, fn).argtypes
    getattr(mutant, fn).restype = ctypes.c_int
oracle._lib = mutant
checks = dict((mm[0], mm[3]) for mm in m.MUTANTS)[{name!r}]
caught = 0
for check in checks:
    try:
        with np.errstate(all="ignore"):
            check()
    except AssertionError:
        caught += 1
print("CAUGHT", caught)
"""


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, checks):
    # The pins run in a child process: a mutant that indexes out of bounds may crash,
    # and a crash counts as caught.
    so = _build_mutant(tmp_path, name, old, new)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(tests_dir), tests=tests_dir, so=so, name=name)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if proc.returncode < 0:          # killed by a signal (out-of-bounds access)
        return
    assert proc.returncode == 0, proc.stderr[-2000:]
    caught = int(proc.stdout.strip().split("CAUGHT")[-1])
    assert caught >= 1, "no pin caught the planted mistake %s" % name


def test_unmutated_oracle_passes_every_pin():
    for check in GEMM_PINS + GENERAL_PINS + CONV_PINS:
        check()
