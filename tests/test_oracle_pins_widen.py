"""Pins for the oracle's allreduce (with Prod), broadcast, symmetric
all_to_all and all_to_all_v combine: closed forms, hand-worked examples in
tests/golden/, the dispatch -> combine round trip, identities with the pinned
reduce_scatter / allgather / all_to_all_v, and the product error bound."""
import math

import numpy as np
import pytest

from conftest import golden
from test_oracle_pins import DT, OPS, STORE, base_grid, dec, enc

PROD = 3


def wins_closed_form(n, rows, cols, ld, dtype, pad=0x3C):
    base = base_grid(rows, cols)
    out = []
    for r in range(n):
        w = np.full((rows, ld), pad, dtype=np.float64)
        w[:, :cols] = base + 100 * r
        out.append(enc(w, dtype))
    return out, base


@pytest.mark.parametrize("dtype", ["f32", "i32", "f16"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("n", [1, 2, 5, 8])
def test_allreduce_closed_form(orc, dtype, op, n):
    rows, cols, ld = 9, 13, 16
    wins, base = wins_closed_form(n, rows, cols, ld, dtype)
    orig = [w.copy() for w in wins]
    assert orc.allreduce(wins, rows, cols, ld, OPS[op], DT[dtype]) == 0
    want = {"sum": n * base + 100 * n * (n - 1) // 2, "max": base + 100 * (n - 1), "min": base}[op]
    for r in range(n):
        np.testing.assert_array_equal(dec(wins[r][:, :cols], dtype), want)
        np.testing.assert_array_equal(wins[r][:, cols:], orig[r][:, cols:])    # padding kept


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min", "prod"])
def test_allreduce_equals_reduce_scatter_then_allgather(orc, dtype, op):
    n, rows, cols, ld = 5, 11, 7, 9
    rng = np.random.default_rng(4)
    wins = [enc(np.where(np.arange(ld) < cols, rng.integers(-3, 4, size=(rows, ld)) * 0.5, 7.0), dtype)
            if dtype != "i32" else rng.integers(-9, 10, size=(rows, ld)).astype(np.int32) for _ in range(n)]
    a = [w.copy() for w in wins]
    b = [w.copy() for w in wins]
    opc = PROD if op == "prod" else OPS[op]
    assert orc.allreduce(a, rows, cols, ld, opc, DT[dtype]) == 0
    assert orc.reduce_scatter(b, rows, cols, ld, opc, DT[dtype]) == 0
    assert orc.allgather(b, rows, cols, ld, DT[dtype]) == 0
    for r in range(n):
        assert np.array_equal(a[r].view(np.uint8), b[r].view(np.uint8))


def test_prod_golden(orc):
    g = golden("allreduce_prod.json")
    v = g["f32"]["values"]
    wins = [np.array([[x]], np.float32) for x in v]
    orc.allreduce(wins, 1, 1, 1, PROD, DT["f32"])
    assert all(w[0, 0] == np.float32(g["f32"]["product"]) for w in wins)
    for case in g["i32"]:
        wins = [np.array([[x]], np.int32) for x in case["values"]]
        orc.allreduce(wins, 1, 1, 1, PROD, DT["i32"])
        assert all(int(w[0, 0]) == case["product"] for w in wins), case


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("n", [2, 3, 8])
def test_prod_closed_form_small_integers(orc, dtype, n):
    """Factors in {-2, ..., 2}: every partial product is an integer of at most
    2^8 in magnitude, exact in every type; the expected value is Python's
    exact product (zero factors included)."""
    rows, cols = 5, 625
    i, j = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    wins = [enc(((3 * i + 7 * j + 11 * r) % 5) - 2, dtype) if dtype != "i32"
            else (((3 * i + 7 * j + 11 * r) % 5) - 2).astype(np.int32) for r in range(n)]
    want = np.ones((rows, cols), dtype=np.int64)
    for r in range(n):
        want *= ((3 * i + 7 * j + 11 * r) % 5) - 2
    orc.allreduce(wins, rows, cols, cols, PROD, DT[dtype])
    for w in wins:
        np.testing.assert_array_equal(dec(w, dtype), want)


def test_prod_int32_wraps(orc):
    rng = np.random.default_rng(8)
    n = 4
    vals = [rng.integers(-2 ** 31, 2 ** 31, size=(3, 50), dtype=np.int64) for _ in range(n)]
    wins = [v.astype(np.int32) for v in vals]
    orc.allreduce(wins, 3, 50, 50, PROD, DT["i32"])
    want = np.ones((3, 50), dtype=object)
    for v in vals:
        want = want * v.astype(object)
    want = np.vectorize(lambda x: ((int(x) + 2 ** 31) % 2 ** 32) - 2 ** 31)(want)
    np.testing.assert_array_equal(wins[0], want.astype(np.int64))


@pytest.mark.parametrize("n", [2, 4, 8])
def test_prod_f32_error_bound(orc, n):
    """|fl(prod) - prod| <= ((1 + 2^-24)^(N-1) - 1) |prod|: N-1 roundings."""
    rng = np.random.default_rng(n)
    wins = [rng.uniform(0.5, 2.0, size=(1, 2048)).astype(np.float32) * rng.choice([-1, 1], size=(1, 2048)).astype(np.float32)
            for _ in range(n)]
    orig = [w.copy() for w in wins]
    orc.allreduce(wins, 1, 2048, 2048, PROD, DT["f32"])
    for j in range(2048):
        exact = math.prod(float(o[0, j]) for o in orig)
        bound = ((1 + 2.0 ** -24) ** (n - 1) - 1) * abs(exact) * (1 + 1e-9)
        assert abs(float(wins[0][0, j]) - exact) <= bound


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_broadcast(orc, dtype):
    n, rows, cols, ld = 4, 6, 10, 12
    wins, _ = wins_closed_form(n, rows, cols, ld, dtype)
    orig = [w.copy() for w in wins]
    for root in range(n):
        ws = [w.copy() for w in orig]
        assert orc.broadcast(ws, root, rows, cols, ld, DT[dtype]) == 0
        for s in range(n):
            np.testing.assert_array_equal(ws[s][:, :cols], orig[root][:, :cols])
            np.testing.assert_array_equal(ws[s][:, cols:], orig[s][:, cols:])
    assert orc.broadcast(wins, 4, rows, cols, ld, DT[dtype]) != 0      # root out of range


@pytest.mark.parametrize("n,tr,size", [(1, 3, 4), (3, 10, 5), (4, 16, 2)])
def test_all_to_all_is_all_to_all_v_with_full_counts(orc, n, tr, size):
    rng = np.random.default_rng(n + tr)
    mr = tr // n
    inputs = [rng.integers(0, 2 ** 16, size=(tr, size), dtype=np.uint64).astype(np.uint16) for _ in range(n)]
    t1 = [np.full((tr, size), 0xFFFF, np.uint16) for _ in range(n)]
    t2 = [np.full((tr, size), 0xFFFF, np.uint16) for _ in range(n)]
    assert orc.all_to_all(inputs, t1, tr, size, 2) == 0
    sc = [np.full(n, mr, np.int32) for _ in range(n)]
    rc = [np.zeros(n, np.int32) for _ in range(n)]
    assert orc.all_to_all_v(inputs, t2, sc, rc, tr, size, 2) == 0
    for d in range(n):
        np.testing.assert_array_equal(t1[d], t2[d])
        for s in range(n):       # block s of target d is block d of input s
            np.testing.assert_array_equal(t1[d][s * mr:(s + 1) * mr], inputs[s][d * mr:(d + 1) * mr])
        assert np.all(t1[d][n * mr:] == 0xFFFF)


def test_combine_golden(orc):
    g = golden("all_to_all_v_combine.json")
    n, tr, size = g["nranks"], g["target_rows"], g["size"]
    wins = [np.array(w, np.int32).reshape(tr, size) for w in g["windows"]]
    rc = [np.array(c, np.int32) for c in g["recv_counts"]]
    for atomic, key in ((0, "expected_none"), (1, "expected_add")):
        outs = [np.array(o, np.int32).reshape(tr, size) for o in g["outputs_before"]]
        assert orc.all_to_all_v_combine(wins, outs, rc, tr, size, atomic, DT["i32"]) == 0
        for s in range(n):
            np.testing.assert_array_equal(outs[s].ravel(), g[key][s])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("n,tr,size", [(2, 8, 3), (4, 21, 5), (5, 40, 4)])
def test_dispatch_then_combine_round_trip(orc, dtype, n, tr, size):
    """all_to_all_v then its combine with kNone returns every dispatched row to
    the place it came from; with kAdd onto a copy of the input it doubles those
    rows (small half-integers: exact in every type). Rows that were not sent
    keep the output's prior content."""
    rng = np.random.default_rng(tr * n)
    mr = tr // n
    vals = [rng.integers(-20, 21, size=(tr, size)) * 0.5 for _ in range(n)]
    inputs = [enc(v, dtype) if dtype != "i32" else (v * 2).astype(np.int32) for v in vals]
    targets = [np.zeros_like(inputs[0]) for _ in range(n)]
    sc = [rng.integers(-2, mr + 3, size=n).astype(np.int32) for _ in range(n)]
    rc = [np.zeros(n, np.int32) for _ in range(n)]
    eb = inputs[0].itemsize
    assert orc.all_to_all_v(inputs, targets, sc, rc, tr, size, eb) == 0
    sent = [np.zeros(tr, bool) for _ in range(n)]
    for s in range(n):
        for d in range(n):
            c = min(max(int(sc[s][d]), 0), mr)
            sent[s][d * mr:d * mr + c] = True
    outs = [np.full_like(inputs[0], 0) for _ in range(n)]
    for o in outs:
        o.view(np.uint8)[...] = 0x77
    before = [o.copy() for o in outs]
    assert orc.all_to_all_v_combine(targets, outs, rc, tr, size, 0, DT[dtype]) == 0
    for s in range(n):
        np.testing.assert_array_equal(outs[s][sent[s]], inputs[s][sent[s]])
        np.testing.assert_array_equal(outs[s][~sent[s]], before[s][~sent[s]])
    outs = [x.copy() for x in inputs]
    assert orc.all_to_all_v_combine(targets, outs, rc, tr, size, 1, DT[dtype]) == 0
    for s in range(n):
        got, orig = dec(outs[s], dtype), dec(inputs[s], dtype)
        np.testing.assert_array_equal(got[sent[s]], 2 * orig[sent[s]])
        np.testing.assert_array_equal(got[~sent[s]], orig[~sent[s]])


def test_allreduce_order_golden(orc):
    """Every window gets the reduction in rank order 0..N-1, whatever its own
    rank: with ranks holding (1, 1, 2^24) that is 1 + 1 + 2^24 = 2^24 + 2 on
    every window (a rank-first order would give 2^24 on window 2)."""
    g = golden("treduce_rank_order_f32.json")
    want = next(c["expected_sum"] for c in g["cases"] if c["root"] == 0)
    wins = [np.array([[v]], np.float32) for v in g["values"]]
    assert orc.allreduce(wins, 1, 1, 1, OPS["sum"], DT["f32"]) == 0
    assert all(w[0, 0] == np.float32(want) for w in wins)
