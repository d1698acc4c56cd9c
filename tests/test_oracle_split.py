"""The full-size GPU parity tests run the oracle on row slices in host
threads. Here, on the CPU: that split run writes exactly what one oracle call
writes, padding included, for every element type and op, with uneven splits,
more threads than rows, and a root other than 0 (TREDUCE); the same for the
allreduce over windows."""
import numpy as np
import pytest

import oracle
from gpu_util import oracle_allreduce_threaded, oracle_treduce_threaded


@pytest.mark.parametrize("dtype,np_t", [(oracle.F32, np.float32), (oracle.I32, np.int32),
                                        (oracle.BF16, np.uint16), (oracle.F16, np.uint16)])
@pytest.mark.parametrize("op", [oracle.SUM, oracle.MAX, oracle.MIN])
@pytest.mark.parametrize("threads,root", [(1, 0), (3, 2), (7, 0), (64, 4)])
def test_row_split_equals_one_call(dtype, np_t, op, threads, root):
    rng = np.random.default_rng(100 + threads)
    rows, ld, vr, vc, n = 29, 40, 23, 37, 5
    if np_t is np.float32:
        srcs = [rng.standard_normal((rows, ld)).astype(np.float32) * 100 for _ in range(n)]
    elif np_t is np.int32:
        srcs = [rng.integers(-2 ** 31, 2 ** 31, (rows, ld), dtype=np.int64).astype(np.int32) for _ in range(n)]
    else:
        # finite 16-bit encodings (exponent field below all-ones)
        srcs = [(rng.integers(0, 2 ** 16, (rows, ld)) & 0xBFFF).astype(np.uint16) for _ in range(n)]
    one = np.full((rows, ld), 7, dtype=np_t)
    split = one.copy()
    assert oracle.treduce(srcs, one, vr, vc, ld, op, dtype, root=root) == 0
    assert oracle_treduce_threaded(srcs, split, vr, vc, ld, op, dtype, threads, root=root) == 0
    assert np.array_equal(split.view(np.uint8), one.view(np.uint8))


@pytest.mark.parametrize("dtype,np_t", [(oracle.F32, np.float32), (oracle.F16, np.uint16)])
@pytest.mark.parametrize("op", [oracle.SUM, oracle.MAX, oracle.PROD])
@pytest.mark.parametrize("threads", [1, 4, 50])
def test_allreduce_row_split_equals_one_call(dtype, np_t, op, threads):
    rng = np.random.default_rng(200 + threads)
    n, rows, cols, ld = 5, 31, 37, 40
    if np_t is np.float32:
        wins = [rng.standard_normal((rows, ld)).astype(np.float32) for _ in range(n)]
    else:
        wins = [(rng.integers(0, 2 ** 16, (rows, ld)) & 0xBFFF).astype(np.uint16) for _ in range(n)]
    one = [w.copy() for w in wins]
    split = [w.copy() for w in wins]
    assert oracle.allreduce(one, rows, cols, ld, op, dtype) == 0
    assert oracle_allreduce_threaded(split, rows, cols, ld, op, dtype, threads) == 0
    for a, b in zip(one, split):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
