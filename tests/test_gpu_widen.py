"""allreduce (with Prod), reduce_scatter with Prod, broadcast, symmetric
all_to_all and the all_to_all_v combine on the GPU (through the C ABI) against
the oracle, bit for bit (any NaN equals any NaN for computed floating
results): small odd cases for every element type and both reduction kernels,
then the 8-window fp16 [8192, 4096] and 16-rank bf16 7168-wide shapes at full
size. Every device buffer carries guard bands."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tile_level_collective_gb300 as P
from gpu_util import DevBuf, NP_STORE, ORC_DT, bits, first_diff, oracle_allreduce_threaded, to_dev, to_host
from test_gpu_collectives import windows_host
from test_gpu_treduce import PCODE, nan_equal

pytestmark = pytest.mark.gpu

ORC_OP4 = {"sum": oracle.SUM, "max": oracle.MAX, "min": oracle.MIN, "prod": oracle.PROD}
P_OP4 = {"sum": P.SUM, "max": P.MAX, "min": P.MIN, "prod": P.PROD}

# (n, rows, cols, ld, offset_bytes)
AR_CASES = [
    (1, 4, 9, 9, 0),
    (2, 3, 17, 20, 0),
    (3, 5, 64, 64, 0),         # whole rows: one flat row
    (8, 33, 256, 264, 0),
    (9, 7, 520, 528, 0),       # two groups of ranks
    (5, 6, 100, 100, 4),
    (4, 5, 31, 33, 0),         # odd pitch
    (8, 100, 131, 136, 0),     # row tails written to every window, two tail blocks
    (10, 40, 67, 72, 0),       # two rank groups with row tails
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min", "prod"])
@pytest.mark.parametrize("case", AR_CASES, ids=lambda c: "n%d_%dx%d_ld%d_o%d" % c)
def test_allreduce_small(dtype, op, case):
    n, rows, cols, ld, off = case
    host = windows_host(dtype, n, rows, cols, ld, seed=rows * 7 + n)
    orig = [h.copy() for h in host]
    dev = [DevBuf(h, off) for h in host]
    P.ptoc_allreduce([d.ptr for d in dev], rows, cols, ld, P_OP4[op], PCODE[dtype])
    torch.cuda.synchronize()
    assert oracle.allreduce(host, rows, cols, ld, ORC_OP4[op], ORC_DT[dtype]) == 0
    for r in range(n):
        got = dev[r].host()
        assert nan_equal(got, host[r], dtype), "window %d: %s" % (r, first_diff(got, host[r]))
        assert np.array_equal(bits(got[:, cols:]), bits(orig[r][:, cols:]))
        assert dev[r].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
def test_reduce_scatter_prod(dtype):
    n, rows, cols, ld = 4, 10, 40, 40
    host = windows_host(dtype, n, rows, cols, ld, seed=17)
    dev = [DevBuf(h) for h in host]
    P.ptoc_reduce_scatter([d.ptr for d in dev], rows, cols, ld, P.PROD, PCODE[dtype])
    torch.cuda.synchronize()
    oracle.reduce_scatter(host, rows, cols, ld, oracle.PROD, ORC_DT[dtype])
    for r in range(n):
        assert nan_equal(dev[r].host(), host[r], dtype) and dev[r].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "f16", "i32"])
@pytest.mark.parametrize("case", [(1, 3, 5, 5, 0, 0), (4, 6, 50, 52, 2, 0), (5, 8, 64, 64, 4, 0),
                                  (8, 9, 1000, 1000, 7, 4), (3, 4, 21, 23, 1, 2)],
                         ids=lambda c: "n%d_%dx%d_ld%d_root%d_o%d" % c)
def test_broadcast_small(dtype, case):
    n, rows, cols, ld, root, off = case
    if off == 2 and dtype in ("f32", "i32"):
        off = 4
    host = windows_host(dtype, n, rows, cols, ld, seed=rows + root)
    dev = [DevBuf(h, off) for h in host]
    P.ptoc_broadcast([d.ptr for d in dev], rows, cols, ld, PCODE[dtype], root=root)
    torch.cuda.synchronize()
    oracle.broadcast(host, root, rows, cols, ld, ORC_DT[dtype])
    for r in range(n):
        assert np.array_equal(bits(dev[r].host()), bits(host[r])) and dev[r].guards_intact()


def _rand_rows(rng, tr, size, et):
    x = rng.integers(0, 2 ** 16, size=(tr, size * (np.dtype(et).itemsize // 2)), dtype=np.uint64)
    return np.ascontiguousarray(x.astype(np.uint16).view(et).reshape(tr, size))


@pytest.mark.parametrize("case", [(1, 4, 3, np.uint16, 0), (3, 12, 5, np.uint16, 0), (4, 17, 8, np.uint16, 0),
                                  (5, 20, 7, np.float32, 0), (16, 64, 33, np.uint16, 0),
                                  (8, 800, 1024, np.uint16, 0), (4, 40, 6, np.uint16, 4)],
                         ids=lambda c: str(c))
def test_all_to_all_small(case):
    n, tr, size, et, off = case
    rng = np.random.default_rng(n * 3 + tr)
    inputs = [_rand_rows(rng, tr, size, et) for _ in range(n)]
    targets = [np.full((tr, size), 0, dtype=et) for _ in range(n)]
    for t in targets:
        t.view(np.uint8)[...] = 0xFF
    d_in = [DevBuf(x, off) for x in inputs]
    d_tg = [DevBuf(t, off) for t in targets]
    P.ptoc_all_to_all([d.ptr for d in d_in], [d.ptr for d in d_tg], tr, size,
                      P.BF16 if np.dtype(et).itemsize == 2 else P.F32)
    torch.cuda.synchronize()
    oracle.all_to_all(inputs, targets, tr, size, np.dtype(et).itemsize)
    for d in range(n):
        assert np.array_equal(d_tg[d].host().view(np.uint8), targets[d].view(np.uint8))
        assert d_tg[d].guards_intact()


def _values(rng, dtype, shape):
    v = rng.standard_normal(shape).astype(np.float32) * np.float32(3.0)
    if dtype == "f32":
        return v
    if dtype == "i32":
        return rng.integers(-2 ** 31, 2 ** 31, size=shape, dtype=np.int64).astype(np.int32)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    return synth.f32_to_bf16_bits(v).reshape(shape)


@pytest.mark.parametrize("atomic", ["none", "add"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("case", [(2, 8, 3, 0), (4, 21, 5, 0), (5, 40, 64, 0), (16, 96, 33, 0),
                                  (6, 600, 520, 0), (3, 30, 7, 2)],
                         ids=lambda c: "n%d_tr%d_size%d_o%d" % c)
def test_dispatch_then_combine(atomic, dtype, case):
    """all_to_all_v on the GPU, then the combine on the GPU, against the oracle
    running the same two steps; outputs start from other random values."""
    n, tr, size, off = case
    if off == 2 and dtype in ("f32", "i32"):
        off = 4
    rng = np.random.default_rng(n * 11 + tr)
    mr = tr // n
    inputs = [_values(rng, dtype, (tr, size)) for _ in range(n)]
    outputs = [_values(rng, dtype, (tr, size)) for _ in range(n)]
    targets = [np.zeros((tr, size), dtype=NP_STORE[dtype]) for _ in range(n)]
    sc = [rng.integers(-3, mr + 4, size=n).astype(np.int32) for _ in range(n)]
    rc = [np.full(n, -9, np.int32) for _ in range(n)]
    d_in = [DevBuf(x, off) for x in inputs]
    d_tg = [DevBuf(t, off) for t in targets]
    d_out = [DevBuf(o, off) for o in outputs]
    d_sc = [DevBuf(c) for c in sc]
    d_rc = [DevBuf(c) for c in rc]
    P.ptoc_all_to_all_v([d.ptr for d in d_in], [d.ptr for d in d_tg], [d.ptr for d in d_sc],
                        [d.ptr for d in d_rc], tr, size, PCODE[dtype])
    code = P.ATOMIC_ADD if atomic == "add" else P.ATOMIC_NONE
    P.ptoc_all_to_all_v_combine([d.ptr for d in d_tg], [d.ptr for d in d_out], [d.ptr for d in d_rc],
                                tr, size, code, PCODE[dtype])
    torch.cuda.synchronize()
    eb = np.dtype(NP_STORE[dtype]).itemsize
    assert oracle.all_to_all_v(inputs, targets, sc, rc, tr, size, eb) == 0
    assert oracle.all_to_all_v_combine(targets, outputs, rc, tr, size,
                                       oracle.ATOMIC_ADD if atomic == "add" else oracle.ATOMIC_NONE,
                                       ORC_DT[dtype]) == 0
    for s in range(n):
        got = d_out[s].host()
        assert nan_equal(got, outputs[s], dtype), "output %d: %s" % (s, first_diff(got, outputs[s]))
        assert d_out[s].guards_intact() and d_tg[s].guards_intact()
        assert np.array_equal(d_rc[s].host(), rc[s])


# ---- full-size shapes ----------------------------------------------------------------

def test_allreduce_full_size_f16():
    """8 windows fp16 [8192, 4096], N(0, 1), Sum: every element of every window
    against the oracle, and equal to reduce_scatter + allgather on the GPU."""
    cfg = synth.WINDOWS_F16_N8_8192X4096
    n, rows, cols, ld = cfg["nranks"], cfg["rows"], cfg["cols"], cfg["ld"]
    host = [synth.window(r) for r in range(n)]
    dev = [to_dev(h) for h in host]
    dev2 = [t.clone() for t in dev]
    P.ptoc_allreduce(dev, rows, cols, ld, P.SUM, P.F16)
    P.ptoc_reduce_scatter(dev2, rows, cols, ld, P.SUM, P.F16)
    P.ptoc_allgather(dev2, rows, cols, ld, P.F16)
    assert oracle_allreduce_threaded(host, rows, cols, ld, oracle.SUM, oracle.F16) == 0
    for r in range(n):
        got = to_host(dev[r], np.uint16)
        assert np.array_equal(got, host[r]), "window %d: %s" % (r, first_diff(got, host[r]))
        assert bool(torch.equal(dev[r], dev2[r]))


def test_broadcast_full_size_f16():
    cfg = synth.WINDOWS_F16_N8_8192X4096
    n, rows, cols, ld = cfg["nranks"], cfg["rows"], cfg["cols"], cfg["ld"]
    dev = [to_dev(synth.window(r)) for r in range(n)]
    root_copy = dev[3].clone()
    P.ptoc_broadcast(dev, rows, cols, ld, P.F16, root=3)
    for r in range(n):
        assert bool(torch.equal(dev[r], root_copy))


def test_all_to_all_full_size():
    """16 ranks, bf16 rows of 7168, target_rows 24576 (chunks of 1536 rows),
    tagged rows: every target against the oracle."""
    cfg = synth.DISPATCH_BF16_N16_7168
    n, tr, size = cfg["nranks"], cfg["target_rows"], cfg["size"]
    inputs = [synth.a2av_input(s, n, tr, size) for s in range(n)]
    d_in = [to_dev(x) for x in inputs]
    d_tg = [torch.full((tr, size), -1, dtype=torch.int16, device="cuda") for _ in range(n)]
    P.ptoc_all_to_all(d_in, d_tg, tr, size, P.BF16)
    targets = [np.full((tr, size), 0xFFFF, np.uint16) for _ in range(n)]
    oracle.all_to_all(inputs, targets, tr, size, 2)
    for d in range(n):
        got = to_host(d_tg[d], np.uint16)
        assert np.array_equal(got, targets[d]), "target %d: %s" % (d, first_diff(got, targets[d]))


def test_dispatch_combine_full_size_bf16():
    """The MoE shape: 16 ranks, bf16 rows of 7168, MAX_RECV 1536, counts
    uniform in [0, 2047]. Dispatch, then combine with kAdd into outputs that
    hold other values; every output element against the oracle."""
    cfg = synth.DISPATCH_BF16_N16_7168
    n, tr, size = cfg["nranks"], cfg["target_rows"], cfg["size"]
    inputs = [synth.values(("normal", 0, 1), synth.DT_BF16, 1234 + s, tr * size).reshape(tr, size)
              for s in range(n)]
    outputs = [synth.values(("normal", 0, 1), synth.DT_BF16, 5678 + s, tr * size).reshape(tr, size)
               for s in range(n)]
    sc = [synth.a2av_send_counts(s, n) for s in range(n)]
    d_in = [to_dev(x) for x in inputs]
    d_out = [to_dev(o) for o in outputs]
    d_tg = [torch.zeros((tr, size), dtype=torch.int16, device="cuda") for _ in range(n)]
    d_sc = [to_dev(c) for c in sc]
    d_rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.ptoc_all_to_all_v(d_in, d_tg, d_sc, d_rc, tr, size, P.BF16)
    P.ptoc_all_to_all_v_combine(d_tg, d_out, d_rc, tr, size, P.ATOMIC_ADD, P.BF16)
    torch.cuda.synchronize()
    targets = [np.zeros((tr, size), np.uint16) for _ in range(n)]
    rc = [np.zeros(n, np.int32) for _ in range(n)]
    oracle.all_to_all_v(inputs, targets, sc, rc, tr, size, 2)
    oracle.all_to_all_v_combine(targets, outputs, rc, tr, size, oracle.ATOMIC_ADD, oracle.BF16)
    for s in range(n):
        got = to_host(d_out[s], np.uint16)
        assert np.array_equal(got, outputs[s]), "output %d: %s" % (s, first_diff(got, outputs[s]))
