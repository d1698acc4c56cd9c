"""Randomised properties of the oracle (hypothesis, CPU only): for any small
shape, rank count, root and values, Max / Min return an input element that
bounds every rank's, Sum lies within the recursive-summation bound of the
exact sum, nothing outside the valid box is written, and all_to_all_v's
counts and placements follow the clamp."""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from test_oracle_pins import DT, OPS  # noqa: E402

shapes = st.tuples(st.integers(1, 6), st.integers(1, 9), st.integers(0, 4))   # rows, cols, extra pitch


@settings(max_examples=120, deadline=None)
@given(shape=shapes, n=st.integers(1, 9), root_frac=st.floats(0, 0.999), seed=st.integers(0, 2 ** 31),
       op=st.sampled_from(["sum", "max", "min"]))
def test_treduce_f32_properties(orc, shape, n, root_frac, seed, op):
    rows, cols, extra = shape
    ld = cols + extra
    root = int(root_frac * n)
    rng = np.random.default_rng(seed)
    srcs = [(rng.standard_normal((rows, ld)) * 10.0 ** rng.integers(-3, 4)).astype(np.float32) for _ in range(n)]
    dst = np.full((rows, ld), 7.25, np.float32)
    assert orc.treduce(srcs, dst, rows, cols, ld, OPS[op], DT["f32"], root=root) == 0
    stack = np.stack([s[:, :cols] for s in srcs]).astype(np.float64)
    out = dst[:, :cols].astype(np.float64)
    if op == "max":
        assert np.all(out == stack.max(0))
    elif op == "min":
        assert np.all(out == stack.min(0))
    else:
        for i in range(rows):
            for j in range(cols):
                xs = stack[:, i, j].tolist()
                bound = (n - 1) * 2.0 ** -24 * math.fsum(abs(x) for x in xs) * (1 + 1e-6)
                assert abs(out[i, j] - math.fsum(xs)) <= bound + 1e-300
    assert np.all(dst[:, cols:] == 7.25)


@settings(max_examples=120, deadline=None)
@given(n=st.integers(1, 6), tr=st.integers(0, 30), size=st.integers(0, 5), seed=st.integers(0, 2 ** 31))
def test_all_to_all_v_properties(orc, n, tr, size, seed):
    rng = np.random.default_rng(seed)
    mr = tr // n
    inputs = [rng.integers(0, 2 ** 16, size=(tr, size), dtype=np.uint64).astype(np.uint16) for _ in range(n)]
    targets = [np.full((tr, size), 0xABCD, np.uint16) for _ in range(n)]
    sc = [rng.integers(-5, mr + 6, size=n).astype(np.int32) for _ in range(n)]
    rc = [np.full(n, 99, np.int32) for _ in range(n)]
    assert orc.all_to_all_v(inputs, targets, sc, rc, tr, size, 2) == 0
    for d in range(n):
        for s in range(n):
            c = min(max(int(sc[s][d]), 0), mr)
            assert rc[d][s] == c
            np.testing.assert_array_equal(targets[d][s * mr:s * mr + c], inputs[s][d * mr:d * mr + c])
            assert np.all(targets[d][s * mr + c:(s + 1) * mr] == 0xABCD)
        assert np.all(targets[d][n * mr:] == 0xABCD)
