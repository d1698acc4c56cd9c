"""TREDUCE on the GPU (through the C ABI) against the oracle.

Small and odd shapes first (every dtype and op, 1 to 64 ranks, root 0 and
root != 0, ragged rows, valid boxes inside padding, in place, buffers placed
off the 16-byte grid so every vector width runs), then the three TREDUCE
workloads at full size. The bar is bit-exactness everywhere: integer, Max and
Min results and all_to_all_v are exact by definition, and the kernels keep the
oracle's rank order and binary32 accumulation, so Sum is exact too (the stated
tolerance, 1 ulp of bf16 / f16 and 1e-6 relative for f32, is therefore met
with zero error). Every device buffer carries guard bands that must survive."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tile_level_collective_gb300 as P
from gpu_util import (DevBuf, ELEM, NP_STORE, ORC_DT, ORC_OP, bits, first_diff, oracle_treduce_threaded, to_dev,
                      to_host)

pytestmark = pytest.mark.gpu

PCODE = {"f32": P.F32, "f16": P.F16, "bf16": P.BF16, "i32": P.I32}
SENT = {"f32": 0xFFD5FFD5, "i32": 0x7FD57FD5, "f16": 0xFFD5, "bf16": 0xFFD5}


def values(rng, dtype, shape, specials=False):
    """Random storage-form values; with `specials`, sprinkle signed zeros,
    infinities, subnormals and the largest finite values (no NaN: NaN cases
    are the Max / Min / copy tests below)."""
    if dtype == "i32":
        v = rng.integers(-2 ** 31, 2 ** 31, size=shape, dtype=np.int64).astype(np.int32)
        if specials:
            m = rng.random(shape) < 0.05
            v[m] = rng.choice(np.array([0, -1, 2 ** 31 - 1, -2 ** 31], dtype=np.int32), size=int(m.sum()))
        return v
    x = rng.standard_normal(shape).astype(np.float32) * np.float32(4.0)
    if dtype == "f32":
        out = x
    elif dtype == "f16":
        out = x.astype(np.float16).view(np.uint16)
    else:
        out = synth.f32_to_bf16_bits(x).reshape(shape)
    if specials:
        sp = {"f32": [0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x00000001, 0x807FFFFF, 0x7F7FFFFF],
              "f16": [0x0000, 0x8000, 0x7C00, 0xFC00, 0x0001, 0x83FF, 0x7BFF],
              "bf16": [0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x807F, 0x7F7F]}[dtype]
        m = rng.random(shape) < 0.05
        b = out.view(np.uint32 if dtype == "f32" else np.uint16)
        b[m] = rng.choice(np.array(sp, dtype=b.dtype), size=int(m.sum()))
    return out


def nan_equal(got, want, dtype):
    """Bitwise equality, except that any NaN equals any NaN (payloads of
    computed NaNs are not specified)."""
    if dtype == "i32":
        return np.array_equal(got, want)
    if dtype == "f32":
        g, w = got.view(np.float32), want.view(np.float32)
        gn, wn = np.isnan(g), np.isnan(w)
    else:
        gb, wb = got.view(np.uint16), want.view(np.uint16)
        e = 0x7C00 if dtype == "f16" else 0x7F80
        m = 0x03FF if dtype == "f16" else 0x007F
        gn = ((gb & e) == e) & ((gb & m) != 0)
        wn = ((wb & e) == e) & ((wb & m) != 0)
    return bool(np.array_equal(gn, wn) and np.array_equal(bits(got)[~gn], bits(want)[~wn]))


def run_case(dtype, op, n, rows, cols, ld, vr, vc, root=0, offset=0, inplace=False, seed=0,
             specials=False, host=None):
    rng = np.random.default_rng(seed)
    if host is None:
        host = []
        for _ in range(n):
            h = np.empty((rows, ld), dtype=NP_STORE[dtype])
            bits(h)[...] = 0x7FD5 if ELEM[dtype] == 2 else 0x7FD57FD5   # NaN-patterned padding
            h[:vr, :vc] = values(rng, dtype, (vr, vc), specials)
            host.append(h)
    srcs = [DevBuf(h, offset) for h in host]
    want = host[root].copy() if inplace else np.empty((rows, ld), dtype=NP_STORE[dtype])
    if not inplace:
        bits(want)[...] = SENT[dtype]
    dst = srcs[root] if inplace else DevBuf(want, offset)
    P.ptoc_treduce([s.ptr for s in srcs], dst.ptr, rows, cols, vr, vc, ld, P.OPS[op], PCODE[dtype],
                   root=root)
    torch.cuda.synchronize()
    assert oracle.treduce(host, want, vr, vc, ld, ORC_OP[op], ORC_DT[dtype], root=root) == 0
    got = dst.host()
    assert nan_equal(got, want, dtype), first_diff(got, want)
    for s in srcs:
        assert s.guards_intact()
    assert dst.guards_intact()
    if not inplace:
        for r, s in enumerate(srcs):
            assert np.array_equal(bits(s.host()), bits(host[r])), "a source was modified"


# (n, rows, cols, ld, vr, vc, root, offset_bytes)
SMALL = [
    (1, 3, 5, 5, 3, 5, 0, 0),
    (2, 1, 1, 1, 1, 1, 1, 0),
    (2, 1, 7, 7, 1, 7, 0, 0),
    (3, 3, 33, 40, 3, 33, 2, 0),
    (4, 17, 100, 128, 13, 97, 1, 0),
    (8, 64, 256, 256, 64, 256, 0, 0),
    (8, 5, 1030, 1030, 5, 1030, 3, 0),
    (9, 4, 8200, 8200, 3, 8199, 8, 0),          # group of 8 plus one; 9 tiles per row
    (16, 9, 300, 304, 9, 300, 5, 0),
    (17, 2, 129, 129, 2, 129, 16, 0),
    (64, 3, 70, 72, 3, 69, 33, 0),
    (4, 6, 50, 52, 6, 50, 0, 4),                # 4-byte aligned buffers
    (4, 6, 50, 52, 6, 50, 2, 8),                # 8-byte aligned buffers
    (5, 7, 31, 33, 7, 31, 4, 0),                # odd pitch: narrow vectors
    (5, 300, 515, 520, 300, 515, 2, 0),         # 900 row-tail elements: four tail blocks
    (11, 120, 259, 264, 120, 259, 7, 0),        # two rank groups, tails over two tail blocks
    (12, 5, 67, 72, 5, 67, 3, 4),               # 9-16 ranks on 4-byte-aligned buffers
    (20, 4, 130, 136, 4, 129, 11, 8),           # over 16 ranks on 8-byte-aligned buffers
    (16, 6, 520, 520, 6, 517, 15, 0),           # 16 ranks, 16-byte data narrowed to 8-byte vectors
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "n%d_%dx%d_ld%d_v%dx%d_r%d_o%d" % c)
def test_small_shapes(dtype, op, case):
    n, rows, cols, ld, vr, vc, root, off = case
    run_case(dtype, op, n, rows, cols, ld, vr, vc, root=root, offset=off, seed=hash(case) % 1000,
             specials=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_two_byte_aligned_16bit(dtype, op):
    """Buffers only 2-byte aligned: the element-wise path."""
    run_case(dtype, op, 3, 5, 37, 37, 5, 37, root=1, offset=2, seed=5)
    run_case(dtype, op, 3, 1, 1001, 1001, 1, 1001, root=0, offset=6, seed=6)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_in_place_on_root(dtype, op):
    run_case(dtype, op, 4, 12, 70, 72, 11, 66, root=2, inplace=True, seed=3)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_single_rank_copies_bits(dtype, op):
    """N = 1 is a bit copy (TREDUCE article §4.3), NaN payloads included."""
    rng = np.random.default_rng(1)
    w = 2 if ELEM[dtype] == 2 else 4
    h = rng.integers(0, 2 ** (8 * w), size=(9, 40), dtype=np.uint64).astype(
        np.uint16 if w == 2 else np.uint32).view(NP_STORE[dtype])
    run_case(dtype, op, 1, 9, 40, 40, 9, 40, host=[np.ascontiguousarray(h)])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_max_min_nan_and_signed_zero(dtype):
    """Max / Min select inputs bit for bit: a NaN never replaces the
    accumulator, a NaN root stays, +0 / -0 ties keep the earlier operand."""
    if dtype == "f32":
        nan, pz, nz, one = 0x7FC01234, 0, 0x80000000, 0x3F800000
        st = np.uint32
    elif dtype == "f16":
        nan, pz, nz, one = 0x7E12, 0, 0x8000, 0x3C00
        st = np.uint16
    else:
        nan, pz, nz, one = 0x7FC3, 0, 0x8000, 0x3F80
        st = np.uint16
    a = np.array([[pz, nz, one, nan] * 8], dtype=st).view(NP_STORE[dtype])
    b = np.array([[nz, pz, nan, one] * 8], dtype=st).view(NP_STORE[dtype])
    c = np.array([[nz, nz, one, nan] * 8], dtype=st).view(NP_STORE[dtype])
    for op in ("max", "min"):
        for root in range(3):
            run_case(dtype, op, 3, 1, 32, 32, 1, 32, root=root, host=[a.copy(), b.copy(), c.copy()])


def test_empty_region_leaves_dst():
    host = [np.ones((4, 8), np.float32) for _ in range(2)]
    srcs = [DevBuf(h) for h in host]
    d = np.full((4, 8), -1.0, np.float32)
    dst = DevBuf(d)
    for vr, vc in ((0, 8), (4, 0)):
        P.ptoc_treduce([s.ptr for s in srcs], dst.ptr, 4, 8, vr, vc, 8, P.SUM, P.F32)
    torch.cuda.synchronize()
    assert np.array_equal(dst.host(), d) and dst.guards_intact()


def test_stream_ordering_on_a_side_stream():
    """Work is enqueued on the given stream and ordered with it."""
    s = torch.cuda.Stream()
    host = [np.full((64, 64), float(r + 1), np.float32) for r in range(3)]
    srcs = [to_dev(h) for h in host]
    dst = torch.zeros(64, 64, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        srcs[0].mul_(2.0)                           # queued before the reduce on s
        P.treduce(srcs, dst, op="sum", stream=s)
    s.synchronize()
    assert torch.all(dst == 2.0 + 2.0 + 3.0)


# ---- full-size workloads --------------------------------------------------------

def _upload(w):
    host = [w.slice(r) for r in range(w.nranks)]
    return host, [to_dev(h) for h in host]


def test_treduce_f32_n4_256_full():
    """4 ranks, f32 256 x 256, U[-1, 1], Sum: every element against the oracle."""
    w = synth.treduce_f32_n4_256()
    host, dev = _upload(w)
    dst = torch.empty(w.rows, w.ld, dtype=torch.float32, device="cuda")
    P.ptoc_treduce(dev, dst, w.rows, w.cols, w.valid_rows, w.valid_cols, w.ld, P.SUM, P.F32)
    want = np.zeros((w.rows, w.ld), np.float32)
    oracle.treduce(host, want, w.valid_rows, w.valid_cols, w.ld, oracle.SUM, oracle.F32)
    got = to_host(dst, np.float32)
    assert np.array_equal(bits(got), bits(want)), first_diff(got, want)


def test_treduce_bf16_n8_4096_valid4000_full():
    """8 ranks, bf16 [4096, 4096], valid 4000 x 4000 inside NaN-sentinel
    padding, N(0, 1); Sum, Max, Min: every element of dst (valid box and the
    untouched 0xFFD5 padding) against the oracle."""
    w = synth.treduce_bf16_n8_4096_valid4000()
    host, dev = _upload(w)
    for op in w.ops:
        want = np.full((w.rows, w.ld), w.dst_pad, dtype=np.uint16)
        dst = to_dev(want)
        P.ptoc_treduce([t for t in dev], dst, w.rows, w.cols, w.valid_rows, w.valid_cols, w.ld,
                       P.OPS[op], P.BF16)
        assert oracle.treduce(host, want, w.valid_rows, w.valid_cols, w.ld, ORC_OP[op], oracle.BF16) == 0
        got = to_host(dst, np.uint16)
        assert np.array_equal(got, want), op + ": " + first_diff(got, want)
        assert np.all(got[w.valid_rows:, :] == w.dst_pad) and np.all(got[:, w.valid_cols:] == w.dst_pad)


def test_treduce_f32_sum_n8_16384x8192_full():
    """8 ranks, f32 [16384, 8192] (4 GiB of inputs), U[-1e3, 1e3], Sum:
    every one of the 134,217,728 elements against the oracle, bit for bit (the
    oracle runs on row slices in host threads). As a second check, independent
    of both, every element lies within the recursive-summation bound
    (N-1) * 2^-24 * sum|x| of the binary64 sum."""
    w = synth.treduce_f32_n8_16384x8192()
    host, dev = _upload(w)
    dst = torch.empty(w.rows, w.ld, dtype=torch.float32, device="cuda")
    P.ptoc_treduce(dev, dst, w.rows, w.cols, w.valid_rows, w.valid_cols, w.ld, P.SUM, P.F32)
    torch.cuda.synchronize()
    want = np.zeros((w.rows, w.ld), np.float32)
    assert oracle_treduce_threaded(host, want, w.valid_rows, w.valid_cols, w.ld, oracle.SUM, oracle.F32) == 0
    got = to_host(dst, np.float32)
    assert got.size == 16384 * 8192
    assert np.array_equal(bits(got), bits(want)), first_diff(got, want)
    exact = torch.zeros(w.rows, w.ld, dtype=torch.float64, device="cuda")
    mag = torch.zeros_like(exact)
    for t in dev:
        exact += t.double()
        mag += t.double().abs()
    err = (dst.double() - exact).abs()
    assert bool(torch.all(err <= (w.nranks - 1) * 2.0 ** -24 * mag * (1 + 1e-6) + 1e-300))


def test_treduce_i32_max_n8_16384x8192_full():
    """8 ranks, int32 [16384, 8192], U[-2^30, 2^30], Max: every one of the
    134,217,728 elements against the oracle, bit for bit."""
    w = synth.treduce_i32_n8_16384x8192()
    host, dev = _upload(w)
    dst = torch.empty(w.rows, w.ld, dtype=torch.int32, device="cuda")
    P.ptoc_treduce(dev, dst, w.rows, w.cols, w.valid_rows, w.valid_cols, w.ld, P.MAX, P.I32)
    torch.cuda.synchronize()
    want = np.zeros((w.rows, w.ld), np.int32)
    assert oracle_treduce_threaded(host, want, w.valid_rows, w.valid_cols, w.ld, oracle.MAX, oracle.I32) == 0
    got = to_host(dst, np.int32)
    assert got.size == 16384 * 8192
    assert np.array_equal(got, want), first_diff(got, want)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_aligned_data_group_forms(dtype, op):
    """16-byte-aligned data: more than one group of eight ranks (the kernel's
    multi-group form, with ragged rows and row tails), one group on full rows,
    and the in-place form."""
    run_case(dtype, op, 11, 7, 520, 528, 6, 517, root=4, seed=12, specials=True)
    run_case(dtype, op, 8, 33, 256, 256, 33, 256, root=0, seed=13)       # flat, full rows
    run_case(dtype, op, 2, 3, 64, 64, 3, 64, root=1, seed=14, inplace=True)
