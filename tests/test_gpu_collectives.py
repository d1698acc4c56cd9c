"""reduce_scatter, allgather and all_to_all_v on the GPU (through the C ABI)
against the oracle, bit for bit: small and odd cases (rows not divisible by N,
rows < N, pitch > cols, buffers off the 16-byte grid, counts below 0 and above
MAX_RECV), then the 8-window fp16 reduce_scatter + allgather workload and the
16-rank MoE-dispatch all_to_all_v workload at full size."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tile_level_collective_gb300 as P
from gpu_util import DevBuf, NP_STORE, ORC_DT, ORC_OP, bits, first_diff, to_dev, to_host
from test_gpu_treduce import PCODE, nan_equal, values

pytestmark = pytest.mark.gpu


def windows_host(dtype, n, rows, cols, ld, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        h = np.empty((rows, ld), dtype=NP_STORE[dtype])
        bits(h)[...] = 0x5A5A if h.itemsize == 2 else 0x5A5A5A5A
        h[:, :cols] = values(rng, dtype, (rows, cols), specials=True)
        out.append(h)
    return out


# (n, rows, cols, ld, offset_bytes)
RS_CASES = [
    (1, 5, 7, 7, 0),
    (2, 3, 9, 12, 0),
    (3, 2, 5, 5, 0),          # rows < N: rank 0 owns no rows
    (4, 10, 33, 40, 0),
    (8, 64, 256, 256, 0),
    (5, 17, 1030, 1032, 4),
    (8, 9, 8200, 8200, 8),
    (6, 7, 31, 33, 0),        # odd pitch
    (8, 100, 131, 136, 0),    # row tails of every owner, over two tail blocks
    (9, 90, 131, 136, 0),     # two rank groups with row tails
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("case", RS_CASES, ids=lambda c: "n%d_%dx%d_ld%d_o%d" % c)
def test_reduce_scatter_then_allgather(dtype, op, case):
    n, rows, cols, ld, off = case
    host = windows_host(dtype, n, rows, cols, ld, seed=rows * 31 + n)
    orig = [h.copy() for h in host]
    dev = [DevBuf(h, off) for h in host]
    ptrs = [d.ptr for d in dev]
    P.ptoc_reduce_scatter(ptrs, rows, cols, ld, P.OPS[op], PCODE[dtype])
    torch.cuda.synchronize()
    assert oracle.reduce_scatter(host, rows, cols, ld, ORC_OP[op], ORC_DT[dtype]) == 0
    for r in range(n):
        got = dev[r].host()
        assert nan_equal(got, host[r], dtype), "RS window %d: %s" % (r, first_diff(got, host[r]))
        assert dev[r].guards_intact()
    P.ptoc_allgather(ptrs, rows, cols, ld, PCODE[dtype])
    torch.cuda.synchronize()
    assert oracle.allgather(host, rows, cols, ld, ORC_DT[dtype]) == 0
    full = np.empty_like(orig[0])
    bits(full)[...] = 0
    oracle.treduce(orig, full, rows, cols, ld, ORC_OP[op], ORC_DT[dtype], root=0)
    for r in range(n):
        got = dev[r].host()
        assert nan_equal(got, host[r], dtype), "AG window %d: %s" % (r, first_diff(got, host[r]))
        # allgather after reduce_scatter is the full reduction; padding kept
        assert nan_equal(got[:, :cols], full[:, :cols], dtype)
        assert np.array_equal(bits(got[:, cols:]), bits(orig[r][:, cols:]))
        assert dev[r].guards_intact()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_two_byte_aligned_windows(dtype):
    n, rows, cols, ld = 3, 8, 21, 23
    host = windows_host(dtype, n, rows, cols, ld, seed=9)
    dev = [DevBuf(h, 2) for h in host]
    P.ptoc_reduce_scatter([d.ptr for d in dev], rows, cols, ld, P.SUM, PCODE[dtype])
    P.ptoc_allgather([d.ptr for d in dev], rows, cols, ld, PCODE[dtype])
    torch.cuda.synchronize()
    oracle.reduce_scatter(host, rows, cols, ld, oracle.SUM, ORC_DT[dtype])
    oracle.allgather(host, rows, cols, ld, ORC_DT[dtype])
    for r in range(n):
        assert nan_equal(dev[r].host(), host[r], dtype) and dev[r].guards_intact()


# ---- all_to_all_v -------------------------------------------------------------

def run_a2av(n, tr, size, elem_np, count_lo, count_hi, seed, offset=0):
    rng = np.random.default_rng(seed)
    mr = tr // n
    inputs = []
    for s in range(n):
        x = rng.integers(0, 2 ** 16, size=(tr, size * (elem_np().itemsize // 2)), dtype=np.uint64)
        x = x.astype(np.uint16).view(elem_np).reshape(tr, size)
        inputs.append(np.ascontiguousarray(x))
    sc = [rng.integers(count_lo, count_hi + 1, size=n).astype(np.int32) for _ in range(n)]
    targets = [np.full((tr, size), 0, dtype=elem_np) for _ in range(n)]
    for t in targets:
        t.view(np.uint8)[...] = 0xFF
    rc = [np.full(n, -7, dtype=np.int32) for _ in range(n)]
    d_in = [DevBuf(x, offset) for x in inputs]
    d_tg = [DevBuf(t, offset) for t in targets]
    d_sc = [DevBuf(c) for c in sc]
    d_rc = [DevBuf(c) for c in rc]
    dt = P.BF16 if elem_np().itemsize == 2 else P.F32
    P.ptoc_all_to_all_v([d.ptr for d in d_in], [d.ptr for d in d_tg], [d.ptr for d in d_sc],
                        [d.ptr for d in d_rc], tr, size, dt)
    torch.cuda.synchronize()
    assert oracle.all_to_all_v(inputs, targets, sc, rc, tr, size, elem_np().itemsize) == 0
    for d in range(n):
        assert np.array_equal(d_rc[d].host(), rc[d]), (d, d_rc[d].host(), rc[d])
        got = d_tg[d].host()
        assert np.array_equal(got.view(np.uint8), targets[d].view(np.uint8)), "target %d" % d
        assert d_tg[d].guards_intact() and d_rc[d].guards_intact()
        assert np.array_equal(d_sc[d].host(), sc[d])
    return mr


@pytest.mark.parametrize("case", [
    # n, target_rows, size, elem type, count range, offset
    (1, 4, 3, np.uint16, -2, 6, 0),
    (2, 7, 4, np.uint16, -1, 5, 0),
    (3, 12, 5, np.uint16, -3, 7, 0),       # odd size: 2-byte rows
    (4, 17, 8, np.uint16, 0, 6, 0),
    (5, 20, 7, np.float32, -2, 6, 0),
    (16, 64, 33, np.uint16, -3, 8, 0),
    (8, 800, 1024, np.uint16, 0, 140, 0),  # several tiles per pair
    (4, 40, 6, np.uint16, 0, 12, 4),       # 4-byte aligned buffers
    (3, 9, 0, np.uint16, -1, 5, 0),        # zero-width rows: counts only
    (4, 3, 8, np.uint16, 0, 3, 0),         # target_rows < N: MAX_RECV = 0
    (64, 320, 24, np.uint16, -2, 7, 0),    # the rank cap: 4096 pairs
], ids=lambda c: str(c))
def test_all_to_all_v_small(case):
    n, tr, size, et, lo, hi, off = case
    run_a2av(n, tr, size, et, lo, hi, seed=n * 7 + tr, offset=off)


# ---- full-size workloads -----------------------------------------------------------

def test_reduce_scatter_allgather_f16_n8_8192x4096_full():
    """8 windows fp16 [8192, 4096], N(0, 1): reduce_scatter (Sum, 1024-row
    chunks) then allgather, every element of every window against the oracle;
    and the gathered windows equal a TREDUCE of saved copies of the inputs."""
    cfg = synth.WINDOWS_F16_N8_8192X4096
    n, rows, cols, ld = cfg["nranks"], cfg["rows"], cfg["cols"], cfg["ld"]
    host = [synth.window(r) for r in range(n)]
    dev = [to_dev(h) for h in host]
    saved = [t.clone() for t in dev]
    P.ptoc_reduce_scatter(dev, rows, cols, ld, P.SUM, P.F16)
    oracle.reduce_scatter(host, rows, cols, ld, oracle.SUM, oracle.F16)
    for r in range(n):
        got = to_host(dev[r], np.uint16)
        assert np.array_equal(got, host[r]), "RS window %d: %s" % (r, first_diff(got, host[r]))
    P.ptoc_allgather(dev, rows, cols, ld, P.F16)
    oracle.allgather(host, rows, cols, ld, oracle.F16)
    full = torch.empty_like(saved[0])
    P.ptoc_treduce(saved, full, rows, cols, rows, cols, ld, P.SUM, P.F16)
    for r in range(n):
        got = to_host(dev[r], np.uint16)
        assert np.array_equal(got, host[r]), "AG window %d: %s" % (r, first_diff(got, host[r]))
        assert bool(torch.equal(dev[r], full))


@pytest.mark.parametrize("count_div", [1, 64])
def test_all_to_all_v_bf16_n16_7168_full(count_div):
    """16 ranks, bf16 rows of 7168, target_rows 24576 (MAX_RECV 1536),
    send_counts uniform in [0, 2047] (about a quarter clamp), tagged input rows,
    targets prefilled with 0xFFFF: every target window and every count against
    the oracle. With the counts divided by 64 it is the sparse exchange
    (about 1 % of capacity) that the benchmark also times."""
    cfg = synth.DISPATCH_BF16_N16_7168
    n, tr, size = cfg["nranks"], cfg["target_rows"], cfg["size"]
    mr = tr // n
    inputs = [synth.a2av_input(s, n, tr, size) for s in range(n)]
    sc = [synth.a2av_send_counts(s, n) // count_div for s in range(n)]
    if count_div == 1:
        assert sum(int((c > mr).sum()) for c in sc) > 0      # the clamp is exercised
    d_in = [to_dev(x) for x in inputs]
    d_tg = [torch.full((tr, size), -1, dtype=torch.int16, device="cuda") for _ in range(n)]
    d_sc = [to_dev(c) for c in sc]
    d_rc = [torch.full((n,), -7, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.ptoc_all_to_all_v(d_in, d_tg, d_sc, d_rc, tr, size, P.BF16)
    torch.cuda.synchronize()
    targets = [np.full((tr, size), cfg["sentinel"], dtype=np.uint16) for _ in range(n)]
    rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
    assert oracle.all_to_all_v(inputs, targets, sc, rc, tr, size, 2) == 0
    del inputs
    for d in range(n):
        assert np.array_equal(d_rc[d].cpu().numpy(), rc[d])
        got = to_host(d_tg[d], np.uint16)
        assert np.array_equal(got, targets[d]), "target %d: %s" % (d, first_diff(got, targets[d]))
        # placement by tag: slot s row i carries (s, d, i)
        for s in range(n):
            c = int(rc[d][s])
            if c:
                blk = got[s * mr:s * mr + c, :3]
                assert np.all(blk[:, 0] == s) and np.all(blk[:, 1] == d)
                assert np.array_equal(blk[:, 2], np.arange(c, dtype=np.uint16))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_nine_ranks(dtype):
    """Nine windows: the kernel's multi-group form in scatter mode."""
    n, rows, cols, ld = 9, 20, 136, 136
    host = windows_host(dtype, n, rows, cols, ld, seed=21)
    dev = [DevBuf(h) for h in host]
    P.ptoc_reduce_scatter([d.ptr for d in dev], rows, cols, ld, P.SUM, PCODE[dtype])
    torch.cuda.synchronize()
    oracle.reduce_scatter(host, rows, cols, ld, oracle.SUM, ORC_DT[dtype])
    for r in range(n):
        assert nan_equal(dev[r].host(), host[r], dtype) and dev[r].guards_intact()


@pytest.mark.parametrize("unroll", ["4", "8", "16"])
def test_all_to_all_v_unrolls(unroll, monkeypatch):
    """The exchange kernel at each of its tile sizes (PTOC_A2AV_UNROLL)."""
    monkeypatch.setenv("PTOC_A2AV_UNROLL", unroll)
    run_a2av(6, 600, 520, np.uint16, -5, 110, seed=33)
    run_a2av(16, 3200, 1024, np.uint16, -40, 260, seed=34)
    run_a2av(3, 30, 8, np.float32, -2, 12, seed=35)
