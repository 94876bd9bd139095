"""The oracle's pins have teeth: each test here plants one plausible mistake
in a temporary copy of the oracle's C source, builds it on the CPU, swaps it
in for the real oracle, and checks that the pins of test_oracle_pins reject
it.  The real oracle is restored afterwards; nothing here touches a GPU."""
import os
import shutil
import tempfile

import pytest

import oracle
from oracle import build as oracle_build

import test_oracle_pins as pins

# (name, text in gemm_oracle.c, replacement)
MUTATIONS = [
    ("dropped_last_term", "for (int64_t k = 0; k < K; ++k) {\n        double product = decode[a_row[k]] * decode[b_row[k]];",
     "for (int64_t k = 0; k < K - 1; ++k) {\n        double product = decode[a_row[k]] * decode[b_row[k]];"),
    ("wrong_sign", "        sum += product;\n        abs_sum += fabs(product);\n    }\n    *c_out",
     "        sum -= product;\n        abs_sum += fabs(product);\n    }\n    *c_out"),
    ("transposed_b", "dot_entry(K, A + i * K, B + j * K,", "dot_entry(K, A + i * K, B + j,"),
    ("swapped_index", "C + i * N + j,\n                      absum ? absum + i * N + j",
     "C + j * M + i,\n                      absum ? absum + i * N + j"),
    ("ties_round_down", "if (rest > 0.5 || (rest == 0.5 && (n & 1u))) n += 1u;", "if (rest > 0.5) n += 1u;"),
    ("ties_round_up", "if (rest > 0.5 || (rest == 0.5 && (n & 1u))) n += 1u;", "if (rest >= 0.5) n += 1u;"),
    ("signed_absum", "        abs_sum += fabs(product);\n    }\n    *c_out", "        abs_sum += product;\n    }\n    *c_out"),
    ("normal_decode_off_by_one", "biased_exp - 15 - 10", "biased_exp - 15 - 9"),
    ("subnormal_decode", "magnitude = ldexp((double)fraction, -24);", "magnitude = ldexp((double)fraction, -25);"),
    ("binade_carry_lost", "        n = 1024u;\n        exponent += 1;", "        n = 1024u;"),
    ("fp32_result_truncated", "*d_out = (float)sum;", "*d_out = (float)(sum * (1.0 - 0x1p-30));"),
    ("nn_wrong_stride", "decode[b_col[k * N]]", "decode[b_col[k * K]]"),
]

# pins that must, between them, catch every mutation (each one runs on the mutant)
PIN_CHECKS = [
    lambda: pins.test_f16_to_f64_exhaustive_against_numpy(),
    lambda: pins.test_f64_to_f16_golden_cases(),
    lambda: pins.test_f64_to_f16_midpoints_ties_to_even(),
    lambda: pins.test_hand_worked_cases(),
    lambda: [pins.test_brute_force_exact_rationals(s) for s in range(6)],
    lambda: pins.test_identity_operands(),
    lambda: pins.test_permutation_operands(),
    lambda: [pins.test_integer_operands_exact(s) for s in [(37, 53, 200), (9, 130, 1000)]],
    lambda: pins.test_rank1_closed_form((16, 24, 64)),
    lambda: [pins.test_nn_f32_integer_operands_exact(s) for s in [(37, 53, 200)]],
    lambda: pins.test_nn_f32_agrees_with_nt_sums(),
    lambda: [pins.test_nn_f32_brute_force_exact_rationals(s) for s in range(3)],
]


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_unmutated_copy_passes_every_pin(workdir):
    src = os.path.join(workdir, "same.c")
    shutil.copy(oracle_build.SRC, src)
    _with_library(oracle_build.compile_source(src, os.path.join(workdir, "same.so")), lambda: [c() for c in PIN_CHECKS])


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(workdir, name, old, new):
    text = open(oracle_build.SRC).read()
    assert text.count(old) == 1, "mutation site for %s not found exactly once" % name
    src = os.path.join(workdir, name + ".c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    so = oracle_build.compile_source(src, os.path.join(workdir, name + ".so"))

    def caught():
        for check in PIN_CHECKS:
            try:
                check()
            except AssertionError:
                return True
        return False

    assert _with_library(so, caught), "no pin rejects the planted mistake %s" % name


def _with_library(path, fn):
    saved = oracle._lib
    oracle._lib = oracle.load_library(path)
    try:
        return fn()
    finally:
        oracle._lib = saved
