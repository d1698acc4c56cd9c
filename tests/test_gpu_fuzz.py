"""Seeded random configurations of every data entry point against the oracle:
rank counts from 1 to 20 (every rank form and the rank groups beyond
them), ragged shapes, pitches wider than the rows, rows of several tiles, valid boxes from empty to
full, every root, buffers placed off the 16-byte grid (so every vector width
runs), Max / Min / Sum / Prod, and exchange counts that are negative, zero,
within and beyond capacity. Every buffer carries guard bands; results must
match bit for bit (any NaN equal to any NaN for computed floating results).
The staged reduction form is forced on random cases too."""
import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import DevBuf, ORC_DT, bits
from test_gpu_collectives import run_a2av, windows_host
from test_gpu_treduce import PCODE, nan_equal, run_case, values

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16", "i32"]
ELEM_BYTES = {"f32": 4, "i32": 4, "f16": 2, "bf16": 2}
OP4 = {"sum": (P.SUM, oracle.SUM), "max": (P.MAX, oracle.MAX), "min": (P.MIN, oracle.MIN),
       "prod": (P.PROD, oracle.PROD)}


def offset(rng, eb):
    """A buffer offset that keeps element alignment but often breaks 16."""
    o = int(rng.choice([0, 2, 4, 6, 8, 12, 16]))
    return o - o % eb


def shape(rng):
    rows = int(rng.integers(1, 40))
    cols = int(rng.integers(1, 300))
    return rows, cols, cols + int(rng.integers(0, 9))


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_treduce(seed):
    rng = np.random.default_rng(1000 + seed)
    for _ in range(100):
        dtype = DTYPES[int(rng.integers(4))]
        op = ["sum", "max", "min"][int(rng.integers(3))]
        n = int(rng.integers(1, 21))
        rows, cols, ld = shape(rng)
        vr, vc = int(rng.integers(0, rows + 1)), int(rng.integers(0, cols + 1))
        run_case(dtype, op, n, rows, cols, ld, vr, vc, root=int(rng.integers(n)),
                 offset=offset(rng, ELEM_BYTES[dtype]), inplace=bool(rng.random() < 0.2),
                 seed=int(rng.integers(1 << 30)), specials=True)


def wide_shape(rng):
    """Rows wider than one tile (256 vectors), so that the pitched path
    splits every row into several tiles plus a ragged last one."""
    rows = int(rng.integers(1, 12))
    cols = int(rng.integers(1000, 5000))
    return rows, cols, cols + int(rng.integers(1, 9))


@pytest.mark.parametrize("seed", range(2))
def test_fuzz_treduce_wide_rows(seed):
    rng = np.random.default_rng(1500 + seed)
    for _ in range(40):
        dtype = DTYPES[int(rng.integers(4))]
        op = ["sum", "max", "min"][int(rng.integers(3))]
        n = int(rng.integers(1, 21))
        rows, cols, ld = wide_shape(rng)
        vr, vc = int(rng.integers(1, rows + 1)), int(rng.integers(1, cols + 1))
        run_case(dtype, op, n, rows, cols, ld, vr, vc, root=int(rng.integers(n)),
                 offset=offset(rng, ELEM_BYTES[dtype]), inplace=bool(rng.random() < 0.2),
                 seed=int(rng.integers(1 << 30)), specials=True)


@pytest.mark.parametrize("seed", range(4))
def test_fuzz_window_collectives(seed):
    """reduce_scatter then allgather, allreduce, and broadcast on random windows."""
    rng = np.random.default_rng(2000 + seed)
    for i in range(60):
        dtype = DTYPES[int(rng.integers(4))]
        n = int(rng.integers(1, 21))
        rows, cols, ld = wide_shape(rng) if i % 6 == 5 else shape(rng)
        off = offset(rng, ELEM_BYTES[dtype])
        what = ["rs_ag", "allreduce", "broadcast"][int(rng.integers(3))]
        host = windows_host(dtype, n, rows, cols, ld, seed=int(rng.integers(1 << 30)))
        dev = [DevBuf(h, off) for h in host]
        ptrs = [d.ptr for d in dev]
        if what == "rs_ag":
            op = ["sum", "max", "min", "prod"][int(rng.integers(4))]
            P.ptoc_reduce_scatter(ptrs, rows, cols, ld, OP4[op][0], PCODE[dtype])
            P.ptoc_allgather(ptrs, rows, cols, ld, PCODE[dtype])
            assert oracle.reduce_scatter(host, rows, cols, ld, OP4[op][1], ORC_DT[dtype]) == 0
            assert oracle.allgather(host, rows, cols, ld, ORC_DT[dtype]) == 0
        elif what == "allreduce":
            op = ["sum", "max", "min", "prod"][int(rng.integers(4))]
            P.ptoc_allreduce(ptrs, rows, cols, ld, OP4[op][0], PCODE[dtype])
            assert oracle.allreduce(host, rows, cols, ld, OP4[op][1], ORC_DT[dtype]) == 0
        else:
            root = int(rng.integers(n))
            P.ptoc_broadcast(ptrs, rows, cols, ld, PCODE[dtype], root=root)
            assert oracle.broadcast(host, root, rows, cols, ld, ORC_DT[dtype]) == 0
        torch.cuda.synchronize()
        for r in range(n):
            got = dev[r].host()
            assert nan_equal(got, host[r], dtype), "%s %s n=%d %dx%d ld %d off %d window %d" % (
                what, dtype, n, rows, cols, ld, off, r)
            assert dev[r].guards_intact()


@pytest.mark.parametrize("seed", range(4))
def test_fuzz_all_to_all_v(seed):
    rng = np.random.default_rng(3000 + seed)
    for _ in range(48):
        n = int(rng.integers(1, 21))
        tr = int(rng.integers(0, 12 * n + 1))
        size = int(rng.integers(0, 200))
        elem = [np.uint16, np.float32][int(rng.integers(2))]
        mr = tr // n
        lo, hi = -int(rng.integers(0, 4)), mr + int(rng.integers(0, 6))
        run_a2av(n, tr, size, elem, lo, hi, seed=int(rng.integers(1 << 30)),
                 offset=offset(rng, np.dtype(elem).itemsize))


@pytest.mark.parametrize("seed", range(2))
def test_fuzz_all_to_all_v_wide_rows(seed):
    """Rows of 4 to 36 KB: every pair's run spans several tiles, and the
    tiles cross row boundaries."""
    rng = np.random.default_rng(3500 + seed)
    for _ in range(24):
        n = int(rng.integers(1, 17))
        tr = int(rng.integers(n, 6 * n + 1))
        size = int(rng.integers(2000, 9000))
        elem = [np.uint16, np.float32][int(rng.integers(2))]
        mr = tr // n
        run_a2av(n, tr, size, elem, -int(rng.integers(0, 3)), mr + int(rng.integers(0, 3)),
                 seed=int(rng.integers(1 << 30)), offset=offset(rng, np.dtype(elem).itemsize))


@pytest.mark.parametrize("seed", range(2))
def test_fuzz_combine_wide_rows(seed):
    """The combine (kNone and kAdd) on rows of 4 to 36 KB, several tiles per
    pair run."""
    rng = np.random.default_rng(4500 + seed)
    for _ in range(16):
        dtype = DTYPES[int(rng.integers(4))]
        eb = ELEM_BYTES[dtype]
        n = int(rng.integers(1, 17))
        tr = int(rng.integers(n, 6 * n + 1))
        size = int(rng.integers(2000, 9000))
        off = offset(rng, eb)
        mr = tr // n
        ins = [values(rng, dtype, (tr, size)) for _ in range(n)]
        outs = [values(rng, dtype, (tr, size)) for _ in range(n)]
        rc = [rng.integers(-1, mr + 2, size=n).astype(np.int32) for _ in range(n)]
        atomic = [P.ATOMIC_NONE, P.ATOMIC_ADD][int(rng.integers(2))]
        d_in = [DevBuf(x, off) for x in ins]
        d_out = [DevBuf(o, off) for o in outs]
        d_rc = [DevBuf(c) for c in rc]
        P.ptoc_all_to_all_v_combine([d.ptr for d in d_in], [d.ptr for d in d_out], [d.ptr for d in d_rc],
                                    tr, size, atomic, PCODE[dtype])
        torch.cuda.synchronize()
        assert oracle.all_to_all_v_combine(ins, outs, rc, tr, size, atomic, ORC_DT[dtype]) == 0
        for s in range(n):
            assert nan_equal(d_out[s].host(), outs[s], dtype), "combine %s atomic %d output %d" % (dtype, atomic, s)
            assert d_out[s].guards_intact() and d_rc[s].guards_intact()


@pytest.mark.parametrize("seed", range(3))
def test_fuzz_all_to_all_and_combine(seed):
    """The symmetric all_to_all and the combine (kNone and kAdd) on random
    shapes, counts and alignments."""
    rng = np.random.default_rng(4000 + seed)
    for _ in range(48):
        dtype = DTYPES[int(rng.integers(4))]
        eb = ELEM_BYTES[dtype]
        n = int(rng.integers(1, 17))
        tr = int(rng.integers(0, 10 * n + 1))
        size = int(rng.integers(0, 160))
        off = offset(rng, eb)
        mr = tr // n
        ins = [values(rng, dtype, (tr, size)) for _ in range(n)]
        if rng.random() < 0.4:
            tgs = [np.full((tr, size), 0, dtype=ins[0].dtype) for _ in range(n)]
            for t in tgs:
                bits(t)[...] = 0x5A5A if eb == 2 else 0x5A5A5A5A
            d_in = [DevBuf(x, off) for x in ins]
            d_tg = [DevBuf(t, off) for t in tgs]
            P.ptoc_all_to_all([d.ptr for d in d_in], [d.ptr for d in d_tg], tr, size, PCODE[dtype])
            torch.cuda.synchronize()
            assert oracle.all_to_all(ins, tgs, tr, size, eb) == 0
            for d in range(n):
                assert np.array_equal(bits(d_tg[d].host()), bits(tgs[d])), "all_to_all target %d" % d
                assert d_tg[d].guards_intact()
            continue
        outs = [values(rng, dtype, (tr, size)) for _ in range(n)]
        rc = [rng.integers(-2, mr + 4, size=n).astype(np.int32) for _ in range(n)]
        atomic = [P.ATOMIC_NONE, P.ATOMIC_ADD][int(rng.integers(2))]
        d_in = [DevBuf(x, off) for x in ins]
        d_out = [DevBuf(o, off) for o in outs]
        d_rc = [DevBuf(c) for c in rc]
        P.ptoc_all_to_all_v_combine([d.ptr for d in d_in], [d.ptr for d in d_out], [d.ptr for d in d_rc],
                                    tr, size, atomic, PCODE[dtype])
        torch.cuda.synchronize()
        assert oracle.all_to_all_v_combine(ins, outs, rc, tr, size, atomic, ORC_DT[dtype]) == 0
        for s in range(n):
            assert nan_equal(d_out[s].host(), outs[s], dtype), "combine %s atomic %d output %d" % (dtype, atomic, s)
            assert d_out[s].guards_intact() and d_rc[s].guards_intact()


def aligned_pitch(rng, cols, eb):
    """A pitch of at least `cols` elements that is a multiple of 16 bytes (the
    staged form's condition), or any pitch one time in four."""
    ld = cols + int(rng.integers(0, 9))
    if rng.random() < 0.75:
        q = 16 // eb
        ld = (ld + q - 1) // q * q
    return ld


@pytest.mark.parametrize("form", ["bulk", "tma"])
@pytest.mark.parametrize("seed", range(4))
def test_fuzz_staged_form(seed, form, monkeypatch):
    """The staged reduction form, forced (its size rule keeps cases this small
    in registers), on random TREDUCE cases over 1 to 10 ranks, mostly
    16-byte-aligned (2 to 8 ranks on aligned buffers and pitch take the staged
    form, the rest the register form), rows of one or several tiles, and on
    the window reductions; no staged wait gives up. The same with the tensor
    form of TREDUCE."""
    monkeypatch.setenv("PTOC_REDUCE_STAGING", form)
    P.ptoc_wait_faults()
    rng = np.random.default_rng(5000 + seed)
    for i in range(60):
        dtype = DTYPES[int(rng.integers(4))]
        eb = ELEM_BYTES[dtype]
        n = int(rng.integers(1, 11))
        rows, cols, _ = wide_shape(rng) if i % 3 == 0 else shape(rng)
        ld = aligned_pitch(rng, cols, eb)
        off = 0 if rng.random() < 0.8 else offset(rng, eb)
        if i % 4 != 3:
            op = ["sum", "max", "min"][int(rng.integers(3))]
            vr, vc = int(rng.integers(0, rows + 1)), int(rng.integers(0, cols + 1))
            if form == "tma" and rng.random() < 0.6:
                vc -= vc % (16 // eb)           # valid rows of a multiple of 16 bytes: the tensor form applies
            run_case(dtype, op, n, rows, cols, ld, vr, vc, root=int(rng.integers(n)), offset=off,
                     inplace=bool(rng.random() < 0.2), seed=int(rng.integers(1 << 30)), specials=True)
            continue
        op = ["sum", "max", "min", "prod"][int(rng.integers(4))]
        host = windows_host(dtype, n, rows, cols, ld, seed=int(rng.integers(1 << 30)))
        dev = [DevBuf(h, off) for h in host]
        ptrs = [d.ptr for d in dev]
        if rng.random() < 0.5:
            P.ptoc_reduce_scatter(ptrs, rows, cols, ld, OP4[op][0], PCODE[dtype])
            assert oracle.reduce_scatter(host, rows, cols, ld, OP4[op][1], ORC_DT[dtype]) == 0
        else:
            P.ptoc_allreduce(ptrs, rows, cols, ld, OP4[op][0], PCODE[dtype])
            assert oracle.allreduce(host, rows, cols, ld, OP4[op][1], ORC_DT[dtype]) == 0
        torch.cuda.synchronize()
        for r in range(n):
            assert nan_equal(dev[r].host(), host[r], dtype), "%s %s n=%d %dx%d ld %d window %d" % (
                op, dtype, n, rows, cols, ld, r)
            assert dev[r].guards_intact()
    torch.cuda.synchronize()
    assert P.ptoc_wait_faults() == 0
