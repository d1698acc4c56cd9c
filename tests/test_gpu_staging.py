"""Every source-loading form of the reductions against the oracle, bit for bit
(PTOC_REDUCE_STAGING=regs: the sources go into registers; =bulk: the
bulk-copy engine stages each rank's tile segment in shared memory; =tma:
TREDUCE through tensor maps over the valid box, 2-D boxes loaded into shared
memory and the result box stored back clipped to the valid box; the window
reductions run the register form under it): the odd small shapes of TREDUCE,
in place, reduce_scatter + allgather and allreduce, then the TREDUCE workloads
and the 8-window reduce_scatter at full size. The forms share the fold
arithmetic, so they must agree everywhere; after each test no staged wait has
given up (ptoc_wait_faults)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tile_level_collective_gb300 as P
from gpu_util import (NP_STORE, ORC_DT, ORC_OP, bits, first_diff, oracle_allreduce_threaded, oracle_treduce_threaded,
                      to_dev, to_host)
import test_gpu_collectives as coll
import test_gpu_widen as widen
from test_gpu_treduce import PCODE, SMALL, run_case

pytestmark = pytest.mark.gpu

FORMS = ["regs", "bulk", "tma"]


@pytest.fixture(params=FORMS)
def form(request, monkeypatch):
    monkeypatch.setenv("PTOC_REDUCE_STAGING", request.param)
    P.ptoc_wait_faults()            # start from a zero count
    yield request.param
    torch.cuda.synchronize()
    assert P.ptoc_wait_faults() == 0


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_small_shapes(form, dtype, op):
    for case in SMALL:
        n, rows, cols, ld, vr, vc, root, off = case
        run_case(dtype, op, n, rows, cols, ld, vr, vc, root=root, offset=off, seed=hash(case) % 1000,
                 specials=True)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_in_place_and_multi_tile_rows(form, dtype, op):
    run_case(dtype, op, 4, 12, 70, 72, 11, 66, root=2, inplace=True, seed=3)
    # in place with valid rows of a multiple of 16 bytes (the tensor form applies)
    run_case(dtype, op, 4, 12, 64, 72, 11, 64, root=1, inplace=True, seed=4)
    # rows of several tiles with a partial last tile, every rank count of one group
    for n in range(2, 9):
        run_case(dtype, op, n, 3, 3000, 3008, 3, 2999, root=n - 1, seed=40 + n)
        # the same with valid rows of a multiple of 16 bytes: several boxes per
        # row and a ragged last box for the tensor form
        run_case(dtype, op, n, 9, 3000, 3008, 7, 2992, root=0, seed=50 + n)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max"])
def test_reduce_scatter_allgather(form, dtype, op):
    for case in coll.RS_CASES:
        coll.test_reduce_scatter_then_allgather(dtype, op, case)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "prod"])
def test_allreduce(form, dtype, op):
    for case in widen.AR_CASES:
        widen.test_allreduce_small(dtype, op, case)


def test_treduce_bf16_n8_4096_valid4000_full(form):
    """8 ranks, bf16 [4096, 4096], valid 4000 x 4000 inside NaN-sentinel
    padding; Sum, Max, Min: every element of dst against the oracle."""
    w = synth.treduce_bf16_n8_4096_valid4000()
    host = [w.slice(r) for r in range(w.nranks)]
    dev = [to_dev(h) for h in host]
    for op in w.ops:
        want = np.full((w.rows, w.ld), w.dst_pad, dtype=np.uint16)
        dst = to_dev(want)
        P.ptoc_treduce(dev, dst, w.rows, w.cols, w.valid_rows, w.valid_cols, w.ld, P.OPS[op], P.BF16)
        assert oracle_treduce_threaded(host, want, w.valid_rows, w.valid_cols, w.ld, ORC_OP[op],
                                       oracle.BF16) == 0
        got = to_host(dst, np.uint16)
        assert np.array_equal(got, want), op + ": " + first_diff(got, want)


@pytest.mark.parametrize("which", ["f32_sum", "i32_max"])
def test_treduce_n8_16384x8192_full(form, which):
    """8 ranks of [16384, 8192]: f32 Sum over U[-1e3, 1e3] and int32 Max over
    U[-2^30, 2^30]; every one of the 134,217,728 elements against the oracle."""
    if which == "f32_sum":
        w, dt, op, np_t = synth.treduce_f32_n8_16384x8192(), "f32", "sum", np.float32
    else:
        w, dt, op, np_t = synth.treduce_i32_n8_16384x8192(), "i32", "max", np.int32
    host = [w.slice(r) for r in range(w.nranks)]
    dev = [to_dev(h) for h in host]
    dst = torch.empty(w.rows, w.ld, dtype=torch.float32 if dt == "f32" else torch.int32, device="cuda")
    P.ptoc_treduce(dev, dst, w.rows, w.cols, w.valid_rows, w.valid_cols, w.ld, P.OPS[op], PCODE[dt])
    want = np.zeros((w.rows, w.ld), np_t)
    assert oracle_treduce_threaded(host, want, w.valid_rows, w.valid_cols, w.ld, ORC_OP[op], ORC_DT[dt]) == 0
    got = to_host(dst, np_t)
    assert np.array_equal(bits(got), bits(want)), first_diff(got, want)


def test_reduce_scatter_f16_n8_8192x4096_full(form):
    """8 windows fp16 [8192, 4096], N(0, 1), Sum: every element of every
    window against the oracle."""
    cfg = synth.WINDOWS_F16_N8_8192X4096
    n, rows, cols, ld = cfg["nranks"], cfg["rows"], cfg["cols"], cfg["ld"]
    host = [synth.window(r) for r in range(n)]
    dev = [to_dev(h) for h in host]
    P.ptoc_reduce_scatter(dev, rows, cols, ld, P.SUM, P.F16)
    assert oracle.reduce_scatter(host, rows, cols, ld, oracle.SUM, oracle.F16) == 0
    for r in range(n):
        got = to_host(dev[r], np.uint16)
        assert np.array_equal(got, host[r]), "window %d: %s" % (r, first_diff(got, host[r]))


def test_wait_faults_reads_zero_when_idle():
    """The fault count is readable at any idle point and restarts at zero."""
    torch.cuda.synchronize()
    P.ptoc_wait_faults()
    assert P.ptoc_wait_faults() == 0


@pytest.mark.parametrize("kind", ["bulk", "tma"])
def test_waits_that_run_out_are_counted_and_recovered(kind, monkeypatch):
    """Failure detection without a GPU fault: with a bound of 1 ns on each
    wait for a copy (PTOC_WAIT_NS), waits run out. The blocks concerned count
    a fault, store nothing, wait (with the full bound) for their own copies in
    flight and return; the launch ends, every element of dst is either still
    the sentinel or the oracle's value, and the next call with the default
    bound is complete and counts no fault."""
    monkeypatch.setenv("PTOC_REDUCE_STAGING", kind)
    n, rows, cols = 8, 2048, 4096            # f32, 16-byte rows: both forms apply
    rng = np.random.default_rng(77)
    host = [rng.standard_normal((rows, cols)).astype(np.float32) for _ in range(n)]
    dev = [to_dev(h) for h in host]
    want = np.zeros((rows, cols), np.float32)
    assert oracle_treduce_threaded(host, want, rows, cols, cols, oracle.SUM, oracle.F32) == 0
    sentinel = np.full((rows, cols), 0xFFD5FFD5, dtype=np.uint32).view(np.float32)
    torch.cuda.synchronize()
    P.ptoc_wait_faults()
    monkeypatch.setenv("PTOC_WAIT_NS", "1")
    dst = to_dev(sentinel)
    P.ptoc_treduce(dev, dst, rows, cols, rows, cols, cols, P.SUM, P.F32)
    torch.cuda.synchronize()
    faults = P.ptoc_wait_faults()
    got = bits(to_host(dst, np.float32))
    untouched = got == 0xFFD5FFD5
    assert faults > 0 and untouched.any()
    assert np.array_equal(got[~untouched], bits(want)[~untouched])
    monkeypatch.delenv("PTOC_WAIT_NS")
    dst = to_dev(sentinel)
    P.ptoc_treduce(dev, dst, rows, cols, rows, cols, cols, P.SUM, P.F32)
    torch.cuda.synchronize()
    assert P.ptoc_wait_faults() == 0
    got = to_host(dst, np.float32)
    assert np.array_equal(bits(got), bits(want)), first_diff(got, want)


def test_allreduce_f16_n8_8192x4096_full(form):
    """8 windows fp16 [8192, 4096], N(0, 1), Sum, fused allreduce in the form
    under test (the tensor setting runs the register form here): every
    element of every window against the oracle."""
    cfg = synth.WINDOWS_F16_N8_8192X4096
    n, rows, cols, ld = cfg["nranks"], cfg["rows"], cfg["cols"], cfg["ld"]
    host = [synth.window(r) for r in range(n)]
    dev = [to_dev(h) for h in host]
    P.ptoc_allreduce(dev, rows, cols, ld, P.SUM, P.F16)
    assert oracle_allreduce_threaded(host, rows, cols, ld, oracle.SUM, oracle.F16) == 0
    for r in range(n):
        got = to_host(dev[r], np.uint16)
        assert np.array_equal(got, host[r]), "window %d: %s" % (r, first_diff(got, host[r]))
