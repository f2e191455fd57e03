"""Plant plausible mistakes in a temporary copy of the C oracle and check that
the pins in test_oracle.py reject every one of them (CPU only).

Each mutation is a one-line textual edit of nm_oracle.c compiled into a
throw-away library; the real oracle source is never touched.  Mutations keep
every memory access in bounds.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle as pins
from tests.golden_examples import load_examples

SRC = os.path.join(os.path.dirname(oracle.__file__), "nm_oracle.c")

MUTANTS = {
    "bit_order_reversed": ("(uint32_t)1u << (k % 32);", "(uint32_t)1u << (31 - k % 32);"),
    "bit_index_mod16": ("(uint32_t)1u << (k % 32);", "(uint32_t)1u << (k % 16);"),
    "values_reversed_in_group": ("values[r * Lv + g * N + kept] = W[r * K + k];",
                                 "values[r * Lv + g * N + (N - 1 - kept)] = W[r * K + k];"),
    "packed_read_reversed": ("oracle_half_to_double(values[vbase + j])",
                             "oracle_half_to_double(values[vbase + (N - 1 - j)])"),
    "dropped_first_term": ("acc += p;\n                    sabs += fabs(p);\n                }\n            }\n            y[",
                           "if (k != 0) acc += p;\n                    sabs += fabs(p);\n                }\n            }\n            y["),
    "abs_sum_signed": ("sabs += fabs(p);\n                        ++j;",
                       "sabs += p;\n                        ++j;"),
    "x_reversed": ("oracle_half_to_double(x[(int64_t)b * ldx + k]);\n                    acc",
                   "oracle_half_to_double(x[(int64_t)b * ldx + (K - 1 - k)]);\n                    acc"),
    "half_bias_off": ("e - 25", "e - 24"),
    "subnormal_scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "unpack_no_zero_fill": ("W_out[r * K + k] = 0;", "W_out[r * K + k] = values[r * Lv + g * N];"),
    "bad_count_only_excess": ("if (kept != N)\n                ++bad;", "if (kept > N)\n                ++bad;"),
    "topn_tie_to_higher_k": ("(a2 == aq && q2 < q)", "(a2 == aq && q2 > q)"),
    "sign_dropped": ("return sign ? -v : v;", "return v;"),
}


def _pins():
    ex = load_examples()
    yield lambda: pins.test_half_decode_matches_numpy_for_every_bit_pattern()
    for e in ex:
        yield lambda e=e: pins.test_pack_matches_hand_worked_examples(e)
        if e.bad == 0:
            yield lambda e=e: pins.test_unpack_matches_hand_worked_examples(e)
    yield lambda: pins.test_pack_matches_numpy_gather_and_bitpack(2, 4, 17, 96)
    yield lambda: pins.test_pack_counts_invalid_groups()
    yield lambda: pins.test_unpack_inverts_pack(2, 4)
    yield lambda: pins.test_spmv_matches_dense_numpy_matmul(2, 4, 2)
    yield lambda: pins.test_spmv_one_hot_picks_a_column_of_the_masked_matrix()
    yield lambda: pins.test_topn_mask_rule()


def test_unmutated_copy_passes_all_pins(tmp_path):
    lib = _build(tmp_path, None)
    oracle.use_library(lib)
    try:
        for pin in _pins():
            pin()
    finally:
        oracle.use_library(None)


def _build(tmp_path, mutation):
    src = open(SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) == 1, "mutation anchor must be unique: %r" % old
        src = src.replace(old, new)
    cpath = os.path.join(tmp_path, "mutant.c")
    lpath = os.path.join(tmp_path, "libmutant.so")
    with open(cpath, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", lpath, cpath, "-lm"], check=True)
    return lpath


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    with tempfile.TemporaryDirectory() as d:
        lib = _build(d, MUTANTS[name])
        oracle.use_library(lib)
        try:
            caught = 0
            for pin in _pins():
                try:
                    pin()
                except AssertionError:
                    caught += 1
            assert caught > 0, "planted mistake %r passed every pin" % name
        finally:
            oracle.use_library(None)
