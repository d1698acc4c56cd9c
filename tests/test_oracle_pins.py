"""Pins for the oracle: it is checked against what the pages and mathematics fix,
never against itself. Closed forms (TREDUCE article §7.1), brute force on tiny
inputs, library conversions (torch bfloat16 / numpy float16), error bounds of
recursive summation, hand-worked examples in tests/golden/, and the invariants
the pages state (N = 1 is a copy, empty regions and padding are never written,
allgather after reduce_scatter equals the full reduction, all_to_all_v clamps
and publishes its counts)."""
import math

import numpy as np
import pytest
import torch

from conftest import golden

OPS = {"sum": 0, "max": 1, "min": 2}
DT = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}
STORE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "i32": np.int32}


# ---- encoding helpers: library conversions only (torch / numpy) -------------

def enc(values, dtype):
    """Python / numpy numbers -> storage encodings, by library routines."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "i32":
        return v.astype(np.int32)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    t = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def dec(bits, dtype):
    """Storage encodings -> float64, by library routines."""
    b = np.asarray(bits)
    if dtype in ("f32", "i32"):
        return b.astype(np.float64)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    t = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def ulp16(x, dtype):
    """Spacing of the 16-bit type's values at magnitude |x|."""
    mant = 10 if dtype == "f16" else 7
    emin = -14 if dtype == "f16" else -126
    a = np.maximum(np.abs(x), 2.0 ** emin)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def run_treduce(orc, srcs, dtype, op, vr, vc, ld, root=0, dst=None, fill=None):
    if dst is None:
        dst = np.zeros_like(srcs[0])
        if fill is not None:
            dst.view(np.uint16 if dst.itemsize == 2 else np.uint32)[...] = fill
    rc = orc.treduce(srcs, dst, vr, vc, ld, OPS[op], DT[dtype], root=root)
    assert rc == 0
    return dst


def base_grid(rows, cols):
    """Small asymmetric integers, so a transposed or mis-strided index changes
    the value: base[i, j] = ((7 i + 3 j) mod 11) - 5."""
    i, j = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    return ((7 * i + 3 * j) % 11) - 5


# ---- TREDUCE: closed form of the page's own test ---------------------------

@pytest.mark.parametrize("dtype", ["f32", "i32", "f16", "bf16"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("nranks", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("shape", [(1, 256, 256), (128, 32, 32), (5, 7, 9)])
def test_treduce_closed_form(orc, dtype, op, nranks, shape):
    """Rank r holds base + 100 r (TREDUCE article §7.1). Every partial sum is an
    integer below 2^24, so binary32 accumulation is exact in any order and the
    result is the closed form, rounded once to the output type by a library
    routine: Sum = N base + 100 N(N-1)/2, Max = base + 100 (N-1), Min = base."""
    rows, cols, ld = shape
    base = base_grid(rows, cols)
    stored = []
    for r in range(nranks):
        full = np.zeros((rows, ld))
        full[:, :cols] = base + 100 * r
        stored.append(enc(full, dtype))
    for root in sorted({0, nranks - 1}):
        dst = run_treduce(orc, stored, dtype, op, rows, cols, ld, root=root, fill=0xFFD5)
        vals = np.stack([dec(s[:, :cols], dtype) for s in stored])  # what was stored
        if op == "sum":
            exact = vals.sum(axis=0)  # exact: small integers in binary64
            if dtype != "i32":
                # closed form holds for exactly representable inputs (f32 / f16 here)
                if dtype in ("f32", "f16"):
                    np.testing.assert_array_equal(exact, nranks * base + 100 * nranks * (nranks - 1) // 2)
            want = enc(exact, dtype)
        elif op == "max":
            want = enc(vals.max(axis=0), dtype)
            if dtype in ("f32", "i32", "f16"):
                np.testing.assert_array_equal(vals.max(axis=0), base + 100 * (nranks - 1))
        else:
            want = enc(vals.min(axis=0), dtype)
            np.testing.assert_array_equal(vals.min(axis=0), dec(enc(base, dtype), dtype))
        np.testing.assert_array_equal(dst[:, :cols], want)
        # columns between valid_cols and ld are never written
        pad = dst[:, cols:].view(np.uint16 if dst.itemsize == 2 else np.uint32)
        assert np.all(pad == 0xFFD5)


def test_treduce_golden_base_plus_100r(orc):
    g = golden("treduce_base_plus_100r.json")
    n, base = g["nranks"], np.array(g["base"])
    for dtype in ("f32", "i32"):
        srcs = [enc(base + 100 * r, dtype).reshape(1, -1) for r in range(n)]
        for op in ("sum", "max", "min"):
            dst = run_treduce(orc, srcs, dtype, op, 1, base.size, base.size)
            np.testing.assert_array_equal(dst.ravel(), np.array(g["expected"][op], dtype=STORE[dtype]))


def test_treduce_large_shape_chunked(orc):
    """128 x 32 int32 (TREDUCE article §7.2): the result is the per-element
    reduction whatever the tiling, checked against the closed form."""
    g = golden("treduce_large_shape_chunked.json")
    rows, cols = g["rows"], g["cols"]
    base = base_grid(rows, cols)
    for n in (2, 4):
        srcs = [(base + 100 * r).astype(np.int32) for r in range(n)]
        for op, want in (("sum", n * base + 100 * n * (n - 1) // 2),
                         ("max", base + 100 * (n - 1)), ("min", base)):
            dst = run_treduce(orc, srcs, "i32", op, rows, cols, cols)
            np.testing.assert_array_equal(dst, want)


# ---- Max / Min semantics: brute force on tiny inputs -----------------------

@pytest.mark.parametrize("dtype", ["f32", "i32", "f16", "bf16"])
@pytest.mark.parametrize("nranks", [2, 3, 4])
def test_max_min_brute_force(orc, dtype, nranks):
    """All {-2,-1,0,1,2}^N combinations, one per element, against Python's
    max / min over the ranks."""
    import itertools
    combos = np.array(list(itertools.product([-2, -1, 0, 1, 2], repeat=nranks)))
    m = combos.shape[0]
    srcs = [enc(combos[:, r], dtype).reshape(1, m) for r in range(nranks)]
    for op, f in (("max", max), ("min", min)):
        for root in range(nranks):
            dst = run_treduce(orc, srcs, dtype, op, 1, m, m, root=root)
            want = enc([f(c) for c in combos.tolist()], dtype)
            np.testing.assert_array_equal(dst.ravel(), want)


def test_max_min_tie_and_nan_reading(orc):
    """Reading for TMAX / TMIN (TREDUCE article §1.3 names the ops only):
    equal values keep the earlier operand in rank order, so +0 / -0 ties return
    the root's zero; a NaN never replaces the accumulator; a NaN root stays."""
    pz, nz = np.float32(0.0), np.float32(-0.0)
    nan = np.array([0x7FC01234], dtype=np.uint32).view(np.float32)[0]
    a = np.array([[pz, nz, 1.0, nan]], dtype=np.float32)
    b = np.array([[nz, pz, nan, 2.0]], dtype=np.float32)
    for op in ("max", "min"):
        d0 = run_treduce(orc, [a, b], "f32", op, 1, 4, 4, root=0)
        d1 = run_treduce(orc, [a, b], "f32", op, 1, 4, 4, root=1)
        bits0, bits1 = d0.view(np.uint32).ravel(), d1.view(np.uint32).ravel()
        assert bits0[0] == 0x00000000 and bits0[1] == 0x80000000     # root 0 zeros kept
        assert bits1[0] == 0x80000000 and bits1[1] == 0x00000000     # root 1 zeros kept
        assert bits0[2] == np.float32(1.0).view(np.uint32)           # NaN never replaces
        assert bits0[3] == 0x7FC01234                                # NaN root stays, bits kept
        assert bits1[2] == 0x7FC01234                                # NaN root stays
        assert d1.ravel()[3] == 2.0


# ---- invariants stated by the pages -----------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "i32", "f16", "bf16"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_single_rank_is_a_copy(orc, dtype, op):
    """nranks == 1 is a plain copy (TREDUCE article §4.3), bit for bit, NaN
    payloads and negative zeros included."""
    rng = np.random.default_rng(7)
    w = 2 if dtype in ("f16", "bf16") else 4
    bits = rng.integers(0, 2 ** (8 * w), size=(6, 11), dtype=np.uint64)
    src = bits.astype(np.uint16 if w == 2 else np.uint32).view(STORE[dtype])
    src = np.ascontiguousarray(src)
    dst = run_treduce(orc, [src], dtype, op, 6, 11, 11)
    assert np.array_equal(dst.view(np.uint8), src.view(np.uint8))


@pytest.mark.parametrize("dtype", ["f32", "i32", "f16", "bf16"])
def test_empty_region_writes_nothing(orc, dtype):
    g = golden("treduce_empty_rows.json")
    srcs = [np.ones((16, 32), dtype=STORE[dtype]) for _ in range(3)]
    for shp in g["shapes"]:
        dst = np.full((16, 32), g["sentinel"], dtype=np.int64).astype(STORE[dtype]) \
            if dtype in ("f32", "i32") else np.full((16, 32), 0xFFFF, dtype=np.uint16)
        before = dst.copy()
        for op in ("sum", "max", "min"):
            rc = orc.treduce(srcs, dst, shp["valid_rows"], shp["valid_cols"], 32, OPS[op], DT[dtype])
            assert rc == 0
        assert np.array_equal(dst.view(np.uint8), before.view(np.uint8))


def test_padding_never_written(orc):
    """Only the valid box of dst is written: the NaN-sentinel layout of the
    4000 x 4000-in-4096 workload, at a small size."""
    rows, ld, vr, vc, n = 9, 16, 6, 11, 4
    rng = np.random.default_rng(3)
    srcs = []
    for _ in range(n):
        s = np.full((rows, ld), 0x7FD5, dtype=np.uint16)
        s[:vr, :vc] = enc(rng.standard_normal((vr, vc)), "bf16")
        srcs.append(s)
    for op in ("sum", "max", "min"):
        dst = np.full((rows, ld), 0xFFD5, dtype=np.uint16)
        orc.treduce(srcs, dst, vr, vc, ld, OPS[op], DT["bf16"])
        mask = np.ones((rows, ld), bool)
        mask[:vr, :vc] = False
        assert np.all(dst[mask] == 0xFFD5)
        assert not np.any(np.isnan(dec(dst[:vr, :vc], "bf16")))


# ---- fp32 Sum: order and error bound ---------------------------------------

def test_rank_order_golden(orc):
    g = golden("treduce_rank_order_f32.json")
    srcs = [np.array([[v]], dtype=np.float32) for v in g["values"]]
    for case in g["cases"]:
        dst = run_treduce(orc, srcs, "f32", "sum", 1, 1, 1, root=case["root"])
        assert dst[0, 0] == np.float32(case["expected_sum"]), case


@pytest.mark.parametrize("nranks", [2, 5, 8, 16])
def test_f32_sum_error_bound(orc, nranks):
    """Recursive summation: |fl(sum) - sum| <= (N-1) 2^-24 sum|x| (first order;
    the second-order term is below 1e-13 relative here)."""
    rng = np.random.default_rng(nranks)
    srcs = [rng.uniform(-1e3, 1e3, size=(1, 4096)).astype(np.float32) for _ in range(nranks)]
    dst = run_treduce(orc, srcs, "f32", "sum", 1, 4096, 4096)
    for j in range(4096):
        xs = [float(s[0, j]) for s in srcs]
        exact = math.fsum(xs)
        bound = (nranks - 1) * 2.0 ** -24 * math.fsum(abs(x) for x in xs) * (1 + 1e-6)
        assert abs(float(dst[0, j]) - exact) <= bound


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("nranks", [2, 8])
def test_16bit_sum_error_bound(orc, dtype, nranks):
    """|out - exact| <= 1/2 ulp of the output type + (N-1) 2^-24 sum|x|:
    binary32 accumulation then one round-to-nearest to the output type."""
    rng = np.random.default_rng(11 + nranks)
    srcs = [enc(rng.standard_normal((1, 8192)), dtype) for _ in range(nranks)]
    dst = run_treduce(orc, srcs, dtype, "sum", 1, 8192, 8192)
    vals = np.stack([dec(s, dtype) for s in srcs])
    exact = vals.sum(axis=0)
    out = dec(dst, dtype)
    bound = 0.5 * ulp16(np.maximum(np.abs(out), np.abs(exact)), dtype) \
        + (nranks - 1) * 2.0 ** -24 * np.abs(vals).sum(axis=0) * (1 + 1e-6)
    assert np.all(np.abs(out - exact) <= bound)


# ---- conversions against library routines ----------------------------------

def _f32_probe_bits():
    rng = np.random.default_rng(5)
    rand = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    hi = np.arange(2 ** 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    struct = (hi[:, None] | lows[None, :]).ravel()
    return np.concatenate([rand, struct])


def test_f32_to_bf16_matches_torch(orc):
    bits = _f32_probe_bits()
    x = bits.view(np.float32)
    got = orc.f32_to_bf16(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


def test_f32_to_f16_matches_numpy(orc):
    bits = _f32_probe_bits()
    # every binary16 value, and the exact midpoints between neighbours (ties)
    h = np.arange(0x7C00, dtype=np.uint16)
    v = h.view(np.float16).astype(np.float64)
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)     # exact in binary32
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0))])
    x = np.concatenate([bits.view(np.float32), near, -near])
    got = orc.f32_to_f16(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


def test_f16_to_f32_matches_numpy(orc):
    h = np.arange(2 ** 16, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_to_f32(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert np.all(np.isnan(got[nan]))


def test_conversion_golden(orc):
    g = golden("conversions.json")
    for x, hx in g["f32_to_f16"]:
        assert orc.f32_to_f16(np.array([x], np.float32))[0] == int(hx, 16), (x, hx)
    for x, hx in g["f32_to_bf16"]:
        assert orc.f32_to_bf16(np.array([x], np.float32))[0] == int(hx, 16), (x, hx)


def test_bf16_widen_exact(orc):
    h = np.arange(2 ** 16, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16_to_f32(h)
    want = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32))
    assert np.array_equal(got.view(np.uint32), h.astype(np.uint32) << 16)  # the encoding's upper half


# ---- reduce_scatter / allgather --------------------------------------------

def _windows(n, rows, cols, ld, dtype):
    base = base_grid(rows, cols)
    out = []
    for r in range(n):
        w = np.full((rows, ld), 0x55, dtype=np.int64)
        w[:, :cols] = base + 100 * r
        out.append(enc(w, dtype) if dtype != "i32" else w.astype(np.int32))
    return out


def test_reduce_scatter_bounds_golden(orc):
    g = golden("reduce_scatter_bounds.json")
    rows, n = g["rows"], g["nranks"]
    cols, ld = 3, 5
    wins = _windows(n, rows, cols, ld, "i32")
    orig = [w.copy() for w in wins]
    assert orc.reduce_scatter(wins, rows, cols, ld, OPS["sum"], DT["i32"]) == 0
    base = base_grid(rows, cols)
    total = n * base + 100 * n * (n - 1) // 2
    b = g["bounds"]
    for r in range(n):
        lo, hi = b[r], b[r + 1]
        np.testing.assert_array_equal(wins[r][lo:hi, :cols], total[lo:hi])
        keep = np.ones(rows, bool)
        keep[lo:hi] = False
        np.testing.assert_array_equal(wins[r][keep], orig[r][keep])   # other rows untouched
        np.testing.assert_array_equal(wins[r][:, cols:], orig[r][:, cols:])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("n,rows", [(4, 10), (4, 3), (8, 64), (3, 7)])
def test_allgather_after_reduce_scatter_is_full_reduction(orc, dtype, n, rows):
    """allgather(reduce_scatter(w)) leaves every window equal to the reduction
    of all windows over the full box (the allreduce identity), bit for bit,
    with Sum in rank order 0..N-1."""
    cols, ld = 6, 8
    rng = np.random.default_rng(rows * n)
    wins = []
    for r in range(n):
        w = np.full((rows, ld), 0x3C, dtype=np.float64)
        w[:, :cols] = rng.integers(-9, 10, size=(rows, cols)) * 0.5
        wins.append(enc(w, dtype) if dtype != "i32" else (w * 2).astype(np.int32))
    orig = [w.copy() for w in wins]
    for op in ("sum", "max", "min"):
        ws = [w.copy() for w in orig]
        full = np.zeros_like(orig[0])
        run_treduce(orc, orig, dtype, op, rows, cols, ld, root=0, dst=full)
        assert orc.reduce_scatter(ws, rows, cols, ld, OPS[op], DT[dtype]) == 0
        assert orc.allgather(ws, rows, cols, ld, DT[dtype]) == 0
        for r in range(n):
            assert np.array_equal(ws[r][:, :cols].view(np.uint8), full[:, :cols].view(np.uint8))
            assert np.array_equal(ws[r][:, cols:], orig[r][:, cols:])
        # closed form on these small half-integers (exact in every type)
        vals = np.stack([dec(o[:, :cols], dtype) for o in orig])
        want = {"sum": vals.sum(0), "max": vals.max(0), "min": vals.min(0)}[op]
        np.testing.assert_array_equal(dec(full[:, :cols], dtype), want)


def test_allgather_copies_owner_chunk(orc):
    n, rows, cols, ld = 4, 10, 5, 7
    wins = [np.full((rows, ld), 1000 * r, dtype=np.int32) + np.arange(rows * ld, dtype=np.int32).reshape(rows, ld)
            for r in range(n)]
    orig = [w.copy() for w in wins]
    assert orc.allgather(wins, rows, cols, ld, DT["i32"]) == 0
    b = golden("reduce_scatter_bounds.json")["bounds"]
    for s in range(n):
        for r in range(n):
            lo, hi = b[r], b[r + 1]
            np.testing.assert_array_equal(wins[s][lo:hi, :cols], orig[r][lo:hi, :cols])
        np.testing.assert_array_equal(wins[s][:, cols:], orig[s][:, cols:])


# ---- all_to_all_v -----------------------------------------------------------

def test_all_to_all_v_golden(orc):
    g = golden("all_to_all_v_clamp.json")
    n, tr, size = g["nranks"], g["target_rows"], g["size"]
    inputs = [np.arange(tr * size, dtype=np.uint16).reshape(tr, size) + 100 * s for s in range(n)]
    inputs = [np.ascontiguousarray(x.astype(np.uint16)) for x in inputs]
    targets = [np.full((tr, size), 0xFFFF, dtype=np.uint16) for _ in range(n)]
    sc = [np.array(c, dtype=np.int32) for c in g["send_counts"]]
    rc = [np.full(n, -7, dtype=np.int32) for _ in range(n)]
    assert orc.all_to_all_v(inputs, targets, sc, rc, tr, size, 2) == 0
    for d in range(n):
        np.testing.assert_array_equal(rc[d], g["expected_recv_counts"][d])
        written = sorted(set(np.nonzero(np.any(targets[d] != 0xFFFF, axis=1))[0].tolist()))
        assert written == g["expected_rows_written"]["target%d" % d]
    mr = tr // n
    # row i of sender s's block for d lands in slot s of target d
    np.testing.assert_array_equal(targets[0][mr + 0], inputs[1][0 * mr + 0])
    np.testing.assert_array_equal(targets[1][0:3], inputs[0][mr:mr + 3])


@pytest.mark.parametrize("n,tr,size", [(3, 12, 5), (4, 17, 3), (5, 20, 8), (1, 4, 2)])
def test_all_to_all_v_tagged_rows(orc, n, tr, size):
    rng = np.random.default_rng(n * 100 + tr)
    mr = tr // n
    inputs = []
    for s in range(n):
        x = rng.integers(0, 2 ** 16, size=(tr, size), dtype=np.uint64).astype(np.uint16)
        for row in range(n * mr):
            x[row, 0], x[row, 1] = s, row // mr
            if size > 2:
                x[row, 2] = row % mr
        inputs.append(np.ascontiguousarray(x))
    targets = [np.full((tr, size), 0xFFFF, dtype=np.uint16) for _ in range(n)]
    sc = [rng.integers(-3, mr + 4, size=n).astype(np.int32) for _ in range(n)]
    rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
    assert orc.all_to_all_v(inputs, targets, sc, rc, tr, size, 2) == 0
    for d in range(n):
        for s in range(n):
            c = min(max(int(sc[s][d]), 0), mr)
            assert rc[d][s] == c
            for i in range(mr):
                row = targets[d][s * mr + i]
                if i < c:
                    assert row[0] == s and row[1] == d and (size <= 2 or row[2] == i)
                    np.testing.assert_array_equal(row, inputs[s][d * mr + i])
                else:
                    assert np.all(row == 0xFFFF)
        assert np.all(targets[d][n * mr:] == 0xFFFF)
