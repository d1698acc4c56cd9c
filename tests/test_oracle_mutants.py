"""Planted mistakes: each case compiles a copy of oracle/oracle.c with one
plausible bug (a dropped term, a wrong index or sign, a transposed operand, a
wrong rounding or clamp) and checks that the pins reject it. The mistakes are
planted in the oracle, on the CPU, in a temporary directory."""
import os

import pytest

import oracle
import test_oracle_barrier as TB
import test_oracle_pins as T
import test_oracle_pins_widen as TW

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "rank order ascending from 0 instead of root first": (
        "order[n++] = root;\n    for (int r = 0; r < nranks; ++r)\n        if (r != root) order[n++] = r;",
        "for (int r = 0; r < nranks; ++r)\n        order[n++] = r;"),
    "last rank dropped from the sum": (
        "for (int t = 1; t < nranks; ++t) {\n            if (op == ORC_SUM) acc = acc + widen",
        "for (int t = 1; t < nranks - 1; ++t) {\n            if (op == ORC_SUM) acc = acc + widen"),
    "Max keeps the later operand on ties": (
        "(op == ORC_MAX && x > acc)", "(op == ORC_MAX && x >= acc)"),
    "Max lets a NaN replace the accumulator": (
        "(op == ORC_MAX && x > acc)", "(op == ORC_MAX && !(x <= acc))"),
    "bf16 rounds half up": (
        "if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u)))", "if (dropped >= 0x8000u)"),
    "f16 subnormal shift off by one": (
        "int shift = (e >= -14) ? 13 : (-1 - e);", "int shift = (e >= -14) ? 13 : (-e);"),
    "f16 widening exponent off by one": (
        "v = ldexpf((float)(1024 + m), e - 25);", "v = ldexpf((float)(1024 + m), e - 24);"),
    "16-bit Sum rounds to the output type after every add": (
        "if (op == ORC_SUM) acc = acc + widen(dtype, src[order[t]], k);",
        "if (op == ORC_SUM) { uint32_t tmp = 0; acc = acc + widen(dtype, src[order[t]], k);"
        " narrow_store(dtype, &tmp, 0, acc); acc = widen(dtype, &tmp, 0); }"),
    "floating accumulator kept in double": (
        "float acc = widen(dtype, src[order[0]], k);", "double acc = widen(dtype, src[order[0]], k);"),
    "Prod adds instead of multiplying": (
        "else acc = acc * widen(dtype, src[order[t]], k);", "else acc = acc + widen(dtype, src[order[t]], k);"),
    "treduce writes one column past the valid box": (
        "for (int64_t j = 0; j < valid_cols; ++j)", "for (int64_t j = 0; j <= valid_cols; ++j)"),
    "reduce_scatter chunk bounds rounded up": (
        "return (r * rows) / nranks;", "return (r * rows + nranks - 1) / nranks;"),
    "all_to_all_v lower clamp dropped": (
        "if (c < 0) c = 0;\n            if (c > max_recv) c = max_recv;\n            recv_counts[d][s]",
        "if (c > max_recv) c = max_recv;\n            recv_counts[d][s]"),
    "all_to_all_v source and destination slots transposed": (
        "(size_t)(s * max_recv + i) * row_bytes,\n                       (const char*)inputs[s] + (size_t)(d * max_recv + i) * row_bytes",
        "(size_t)(d * max_recv + i) * row_bytes,\n                       (const char*)inputs[s] + (size_t)(s * max_recv + i) * row_bytes"),
    "all_to_all_v count published to the wrong peer": (
        "recv_counts[d][s] = (int32_t)c;", "recv_counts[s][d] = (int32_t)c;"),
    "allreduce reduces each window in its own rank-first order": (
        "oracle_treduce((const void* const*)snap, nranks, 0, win[r]",
        "oracle_treduce((const void* const*)snap, nranks, r, win[r]"),
    "combine with kAdd overwrites": (
        "if (atomic == ORC_ATOMIC_NONE) {", "if (1) {"),
    "credit barrier waits for equality": (
        "if (wait_eq ? (v != gen[r]) : (v < gen[r])) ready = 0;", "if (v != gen[r]) ready = 0;"),
    "credit barrier epilogue subtracts one credit too few": (
        "if (s != r) signal[r * N + s] -= generations;", "if (s != r) signal[r * N + s] -= generations - 1;"),
}


def pins():
    """The pin checks run against each mutant (fast ones, every area)."""
    o = oracle
    return [
        lambda: T.test_rank_order_golden(o),
        lambda: T.test_treduce_golden_base_plus_100r(o),
        lambda: T.test_treduce_closed_form(o, "f32", "sum", 4, (5, 7, 9)),
        lambda: T.test_treduce_closed_form(o, "bf16", "sum", 8, (5, 7, 9)),
        lambda: T.test_treduce_closed_form(o, "f16", "max", 3, (5, 7, 9)),
        lambda: T.test_treduce_closed_form(o, "i32", "min", 2, (128, 32, 32)),
        lambda: T.test_max_min_tie_and_nan_reading(o),
        lambda: T.test_padding_never_written(o),
        lambda: T.test_f32_to_bf16_matches_torch(o),
        lambda: T.test_f32_to_f16_matches_numpy(o),
        lambda: T.test_f16_to_f32_matches_numpy(o),
        lambda: T.test_reduce_scatter_bounds_golden(o),
        lambda: T.test_all_to_all_v_golden(o),
        lambda: T.test_all_to_all_v_tagged_rows(o, 3, 12, 5),
        lambda: TW.test_allreduce_order_golden(o),
        lambda: TW.test_prod_golden(o),
        lambda: TW.test_combine_golden(o),
        lambda: TB.test_complete_call_self_clears(o, 3, 2),
        lambda: TB.test_missing_rank_golden(o),
    ]


def caught(lib_path):
    saved = oracle._lib
    oracle._lib = oracle.load(lib_path)
    try:
        for check in pins():
            try:
                check()
            except AssertionError:
                return True
        return False
    finally:
        oracle._lib = saved


def test_the_pins_accept_the_oracle(orc):
    assert not caught(orc.build())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_the_pins_reject_a_planted_mistake(orc, name, tmp_path):
    find, repl = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(find) >= 1, "the mutation site moved: " + name
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(text.replace(find, repl, 1))
    lib = oracle.compile_source(str(mutant), str(tmp_path / "liboracle_mutant.so"))
    assert caught(lib), "no pin rejects: " + name
