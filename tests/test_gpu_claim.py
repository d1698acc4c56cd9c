"""The claiming exchange kernel (all_to_all_v and the combine, whose counts live
on the device): one wave of blocks takes the live tiles from a zeroed 4-byte
counter that each call allocates in stream order. Covered here:
- sparse counts (nothing, one pair, everything at capacity);
- calls whose kernels overlap on several streams, and calls from several host
  threads (each call has its own counter);
- calls with a synchronization between them (the library pool's path);
- replay of a captured graph (the graph memory node path).
Every result is compared with the oracle on the same host data."""
import threading

import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def make(n, tr, size, counts, seed):
    rng = np.random.default_rng(seed)
    ins = [rng.integers(0, 2 ** 16, size=(tr, size), dtype=np.uint64).astype(np.uint16) for _ in range(n)]
    sc = [np.asarray(c, dtype=np.int32) for c in counts]
    return ins, sc


def expect(ins, sc, tr, size):
    n = len(ins)
    th = [np.full((tr, size), 0xFFFF, np.uint16) for _ in range(n)]
    rh = [np.zeros(n, np.int32) for _ in range(n)]
    assert oracle.all_to_all_v(ins, th, sc, rh, tr, size, 2) == 0
    return th, rh


def run_a2av(ins, sc, tr, size, stream=None):
    n = len(ins)
    d_in = [to_dev(h) for h in ins]
    d_sc = [to_dev(c) for c in sc]
    d_tg = [torch.full((tr, size), -1, dtype=torch.int16, device="cuda") for _ in range(n)]
    d_rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.ptoc_all_to_all_v(d_in, d_tg, d_sc, d_rc, tr, size, P.BF16, stream=stream)
    return d_in, d_sc, d_tg, d_rc


PATTERNS = ["none", "one_pair", "capacity", "above_capacity", "diagonal"]


@pytest.mark.parametrize("pattern", PATTERNS)
def test_sparse_and_full_counts(pattern):
    n, tr, size = 8, 8 * 37, 300
    mr = tr // n
    counts = np.zeros((n, n), np.int32)
    if pattern == "one_pair":
        counts[5, 2] = 29
    elif pattern == "capacity":
        counts[:] = mr
    elif pattern == "above_capacity":
        counts[:] = mr + 1000
    elif pattern == "diagonal":
        counts[np.arange(n), np.arange(n)] = mr - 1
    ins, sc = make(n, tr, size, counts, seed=PATTERNS.index(pattern))
    _, _, d_tg, d_rc = run_a2av(ins, sc, tr, size)
    torch.cuda.synchronize()
    th, rh = expect(ins, sc, tr, size)
    for d in range(n):
        assert np.array_equal(to_host(d_tg[d], np.uint16), th[d]), "target %d" % d
        assert np.array_equal(d_rc[d].cpu().numpy(), rh[d])


def test_combine_sparse_counts():
    """The combine (kAdd) with most recv counts zero and one at capacity."""
    n, tr, size = 6, 6 * 20, 96
    mr = tr // n
    rc = np.zeros((n, n), np.int32)
    rc[1, 4] = mr
    rc[3, 3] = 7
    rng = np.random.default_rng(5)
    wins = [rng.integers(-1000, 1000, size=(tr, size)).astype(np.int32) for _ in range(n)]
    outs = [rng.integers(-1000, 1000, size=(tr, size)).astype(np.int32) for _ in range(n)]
    rcs = [rc[d].copy() for d in range(n)]
    d_w = [to_dev(w) for w in wins]
    d_o = [to_dev(o) for o in outs]
    d_rc = [to_dev(r) for r in rcs]
    P.ptoc_all_to_all_v_combine(d_w, d_o, d_rc, tr, size, P.ATOMIC_ADD, P.I32)
    torch.cuda.synchronize()
    assert oracle.all_to_all_v_combine(wins, outs, rcs, tr, size, oracle.ATOMIC_ADD, oracle.I32) == 0
    for d in range(n):
        assert np.array_equal(to_host(d_o[d], np.int32), outs[d])


def test_overlapping_calls_on_streams():
    """Calls on four streams with no synchronization between them: their
    kernels may run at the same time, each with its own counter."""
    n, tr, size = 5, 5 * 64, 520
    rng = np.random.default_rng(11)
    cases = []
    streams = [torch.cuda.Stream() for _ in range(4)]
    for k, st in enumerate(streams):
        ins, sc = make(n, tr, size, rng.integers(-3, 70, size=(n, n)), seed=20 + k)
        with torch.cuda.stream(st):
            bufs = run_a2av(ins, sc, tr, size, stream=st)
        cases.append((ins, sc, bufs))
    torch.cuda.synchronize()
    for ins, sc, (_, _, d_tg, d_rc) in cases:
        th, rh = expect(ins, sc, tr, size)
        for d in range(n):
            assert np.array_equal(to_host(d_tg[d], np.uint16), th[d])
            assert np.array_equal(d_rc[d].cpu().numpy(), rh[d])


def test_host_threads():
    errors = []

    def worker(tid):
        try:
            n, tr, size = 4 + tid % 3, 48 * (4 + tid % 3), 200 + 8 * tid
            rng = np.random.default_rng(300 + tid)
            st = torch.cuda.Stream()
            for it in range(6):
                ins, sc = make(n, tr, size, rng.integers(-5, 60, size=(n, n)), seed=1000 * tid + it)
                with torch.cuda.stream(st):
                    _, _, d_tg, d_rc = run_a2av(ins, sc, tr, size, stream=st)
                st.synchronize()
                th, rh = expect(ins, sc, tr, size)
                for d in range(n):
                    if not np.array_equal(to_host(d_tg[d], np.uint16), th[d]) or \
                            not np.array_equal(d_rc[d].cpu().numpy(), rh[d]):
                        errors.append("thread %d iteration %d rank %d" % (tid, it, d))
                        return
        except Exception as e:  # reported to the main thread
            errors.append("thread %d: %r" % (tid, e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(6)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_synchronized_repeats():
    """A synchronization after every call (the pool keeps its memory mapped;
    each call still gets a zeroed counter)."""
    n, tr, size = 8, 8 * 30, 128
    rng = np.random.default_rng(77)
    for it in range(8):
        ins, sc = make(n, tr, size, rng.integers(-2, 40, size=(n, n)), seed=500 + it)
        _, _, d_tg, d_rc = run_a2av(ins, sc, tr, size)
        torch.cuda.synchronize()
        th, rh = expect(ins, sc, tr, size)
        for d in range(n):
            assert np.array_equal(to_host(d_tg[d], np.uint16), th[d])
            assert np.array_equal(d_rc[d].cpu().numpy(), rh[d])


def test_graph_replay_of_dispatch_and_combine():
    """all_to_all_v then the kAdd combine captured once and replayed with new
    counts and data: each replay allocates and zeroes its own counters."""
    n, tr, size = 4, 4 * 50, 72
    rng = np.random.default_rng(9)
    d_in = [torch.zeros(tr, size, dtype=torch.int32, device="cuda") for _ in range(n)]
    d_tg = [torch.zeros(tr, size, dtype=torch.int32, device="cuda") for _ in range(n)]
    d_out = [torch.zeros(tr, size, dtype=torch.int32, device="cuda") for _ in range(n)]
    d_sc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
    d_rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]

    def step():
        P.ptoc_all_to_all_v(d_in, d_tg, d_sc, d_rc, tr, size, P.I32)
        P.ptoc_all_to_all_v_combine(d_tg, d_out, d_rc, tr, size, P.ATOMIC_ADD, P.I32)

    step()                               # first calls outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for it in range(4):
        ins = [rng.integers(-100, 100, size=(tr, size)).astype(np.int32) for _ in range(n)]
        outs = [rng.integers(-100, 100, size=(tr, size)).astype(np.int32) for _ in range(n)]
        tgs = [np.zeros((tr, size), np.int32) for _ in range(n)]
        sc = [rng.integers(-4, 60, size=n).astype(np.int32) for _ in range(n)]
        for dst, src in zip(d_in + d_out + d_tg + d_sc, ins + outs + tgs + sc):
            dst.copy_(torch.from_numpy(src).cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        rc = [np.zeros(n, np.int32) for _ in range(n)]
        assert oracle.all_to_all_v(ins, tgs, sc, rc, tr, size, 4) == 0
        assert oracle.all_to_all_v_combine(tgs, outs, rc, tr, size, oracle.ATOMIC_ADD, oracle.I32) == 0
        for d in range(n):
            assert np.array_equal(to_host(d_tg[d], np.int32), tgs[d]), "replay %d target %d" % (it, d)
            assert np.array_equal(d_rc[d].cpu().numpy(), rc[d])
            assert np.array_equal(to_host(d_out[d], np.int32), outs[d]), "replay %d output %d" % (it, d)
