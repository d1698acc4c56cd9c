"""The other reading of the accumulator's precision: the TREDUCE article (§3.1)
declares the accumulator tile with the destination's element type, so every
partial sum would be rounded to that type before the next rank is added. The
oracle carries that reading as test infrastructure (the library accumulates
in binary32 with one rounding at the end). Here it is pinned by hand-worked
cases and compared with the binary32 accumulator on the input recipe of the
8-rank bf16 N(0, 1) workload, which shows what the binary32 accumulator
changes."""
import numpy as np
import pytest

import oracle
import synth


def bf16_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f16_to_f32(b):
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float32)


def one(values, enc):
    return [enc(np.array([v], np.float32)) for v in values]


@pytest.mark.parametrize("dtype,big", [("bf16", 256.0), ("f16", 2048.0)])
@pytest.mark.parametrize("root", [0, 1])
def test_hand_worked_partial_rounding(dtype, big, root):
    """big + 1 + 1 where big + 1 is a tie between two representable values:
    rounded to even after every add it stays at big; in binary32 the sum is
    big + 2, which the type represents exactly."""
    enc, dec, code = ((synth.f32_to_bf16_bits, bf16_to_f32, oracle.BF16) if dtype == "bf16"
                      else (synth.f32_to_f16_bits, f16_to_f32, oracle.F16))
    srcs = one([big, 1.0, 1.0], enc)
    native, b32 = np.zeros(1, np.uint16), np.zeros(1, np.uint16)
    assert oracle.treduce_sum_native_acc(srcs, native, 1, 1, 1, code, root=root) == 0
    assert oracle.treduce(srcs, b32, 1, 1, 1, oracle.SUM, code, root=root) == 0
    assert dec(native)[0] == big
    assert dec(b32)[0] == big + 2


def test_f32_readings_coincide():
    n, rows, cols = 5, 16, 64
    srcs = [synth.values(("uniform", -1e3, 1e3), "f32", 77 + r, rows * cols) for r in range(n)]
    a, b = np.zeros(rows * cols, np.float32), np.zeros(rows * cols, np.float32)
    assert oracle.treduce_sum_native_acc(srcs, a, rows, cols, cols, oracle.F32, root=2) == 0
    assert oracle.treduce(srcs, b, rows, cols, cols, oracle.SUM, oracle.F32, root=2) == 0
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_exact_partials_coincide():
    """Small integers whose partial sums the type holds exactly: both
    readings give the exact sum."""
    n, k = 8, 300
    base = (np.arange(k) % 7 - 3).astype(np.float32)
    srcs = [synth.f32_to_bf16_bits(base + r) for r in range(n)]
    a, b = np.zeros(k, np.uint16), np.zeros(k, np.uint16)
    assert oracle.treduce_sum_native_acc(srcs, a, 1, k, k, oracle.BF16) == 0
    assert oracle.treduce(srcs, b, 1, k, k, oracle.SUM, oracle.BF16) == 0
    assert np.array_equal(a, b)
    assert np.array_equal(bf16_to_f32(b), n * base + n * (n - 1) / 2)


def test_binary32_accumulator_on_the_bf16_workload_recipe():
    """8 ranks of bf16 N(0, 1) values (the seeds and distribution of the
    4000 x 4000 workload, first 64k elements): the binary32 accumulator stays
    within half an output ulp of the exact sum plus the summation bound, and is
    closer on average than rounding every partial sum."""
    n, k = 8, 1 << 16
    srcs = [synth.values(("normal", 0, 1), "bf16", synth.BASE_SEED + r, k) for r in range(n)]
    x = np.stack([bf16_to_f32(s).astype(np.float64) for s in srcs])
    exact = x.sum(axis=0)                     # exact: few bits per value, far from overflow
    nat, b32 = np.zeros(k, np.uint16), np.zeros(k, np.uint16)
    assert oracle.treduce_sum_native_acc(srcs, nat, 1, k, k, oracle.BF16) == 0
    assert oracle.treduce(srcs, b32, 1, k, k, oracle.SUM, oracle.BF16) == 0
    err_b32 = np.abs(bf16_to_f32(b32).astype(np.float64) - exact)
    err_nat = np.abs(bf16_to_f32(nat).astype(np.float64) - exact)
    half_ulp = np.spacing(np.abs(bf16_to_f32(b32)).astype(np.float32)).astype(np.float64) * 2 ** 15
    bound = half_ulp + (n - 1) * 2.0 ** -24 * np.abs(x).sum(axis=0)
    assert np.all(err_b32 <= bound + 1e-30)
    assert err_b32.mean() < err_nat.mean()
    assert err_nat.max() > err_b32.max()
    differ = float(np.mean(nat != b32))
    assert 0.05 < differ < 0.95               # the two readings disagree on many elements
