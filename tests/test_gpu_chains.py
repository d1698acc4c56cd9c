"""Dependent calls back to back on one stream, no host synchronisation in
between: each call reads what the previous one wrote. With programmatic
dependent launch (the default) a kernel may start while the previous one
finishes; its griddepcontrol.wait must still order every read after the
producer's writes. Checked bit for bit against the oracle running the same
chain, with the overlap on and off."""
import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pdl", ["1", "0"])
def test_dependent_chain(pdl, monkeypatch):
    monkeypatch.setenv("PTOC_PDL", pdl)
    n, rows, cols = 4, 512, 2048
    rng = np.random.default_rng(2)
    hs = [rng.integers(-1000, 1000, size=(rows, cols)).astype(np.int32) for _ in range(n)]
    srcs = [to_dev(h) for h in hs]
    d1 = torch.empty(rows, cols, dtype=torch.int32, device="cuda")
    d2 = torch.empty_like(d1)
    wins = [torch.empty_like(d1) for _ in range(n)]
    tr, size = 256, 64
    for it in range(5):
        # TREDUCE -> TREDUCE on its output -> copy into windows -> RS -> AG ->
        # allreduce -> all_to_all_v from the windows -> combine back
        P.ptoc_treduce(srcs, d1, rows, cols, rows, cols, cols, P.SUM, P.I32)
        P.ptoc_treduce([d1, srcs[it % n]], d2, rows, cols, rows, cols, cols, P.MAX, P.I32)
        for w in wins:
            P.ptoc_treduce([d2], w, rows, cols, rows, cols, cols, P.SUM, P.I32)    # one rank: a copy
        P.ptoc_reduce_scatter(wins, rows, cols, cols, P.MIN, P.I32)
        P.ptoc_allgather(wins, rows, cols, cols, P.I32)
        P.ptoc_allreduce(wins, rows, cols, cols, P.SUM, P.I32)
        ins = [w.view(-1)[: tr * size].view(tr, size) for w in wins]
        tgs = [torch.zeros(tr, size, dtype=torch.int32, device="cuda") for _ in range(n)]
        sc = [to_dev(np.full(n, 40 + s, np.int32)) for s in range(n)]
        rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
        P.ptoc_all_to_all_v(ins, tgs, sc, rc, tr, size, P.I32)
        outs = [torch.ones(tr, size, dtype=torch.int32, device="cuda") for _ in range(n)]
        P.ptoc_all_to_all_v_combine(tgs, outs, rc, tr, size, P.ATOMIC_ADD, P.I32)
        torch.cuda.synchronize()

        o1 = np.zeros((rows, cols), np.int32)
        oracle.treduce(hs, o1, rows, cols, cols, oracle.SUM, oracle.I32)
        o2 = np.zeros_like(o1)
        oracle.treduce([o1, hs[it % n]], o2, rows, cols, cols, oracle.MAX, oracle.I32)
        ow = [o2.copy() for _ in range(n)]
        oracle.reduce_scatter(ow, rows, cols, cols, oracle.MIN, oracle.I32)
        oracle.allgather(ow, rows, cols, cols, oracle.I32)
        oracle.allreduce(ow, rows, cols, cols, oracle.SUM, oracle.I32)
        assert np.array_equal(to_host(d2, np.int32), o2)
        for w, o in zip(wins, ow):
            assert np.array_equal(to_host(w, np.int32), o)
        oi = [np.ascontiguousarray(o.reshape(-1)[: tr * size].reshape(tr, size)) for o in ow]
        ot = [np.zeros((tr, size), np.int32) for _ in range(n)]
        orc_ = [np.zeros(n, np.int32) for _ in range(n)]
        oracle.all_to_all_v(oi, ot, [np.full(n, 40 + s, np.int32) for s in range(n)], orc_, tr, size, 4)
        oo = [np.ones((tr, size), np.int32) for _ in range(n)]
        oracle.all_to_all_v_combine(ot, oo, orc_, tr, size, oracle.ATOMIC_ADD, oracle.I32)
        for t, o in zip(outs, oo):
            assert np.array_equal(to_host(t, np.int32), o)


@pytest.mark.parametrize("prefetch", ["1", "0"])
def test_first_wave_prefetch_of_rows_written_last(prefetch, monkeypatch):
    """The register form's first wave asks L2 for its first tiles before it
    waits for the previous kernel. Here the next call's sources are the rows
    the previous call writes in its last waves (the tail of a 64 MiB result),
    and every iteration writes new values there, so a prefetch that served a
    stale line would show. Bit for bit against the oracle, prefetch on and
    off, programmatic dependent launch on."""
    monkeypatch.setenv("PTOC_PDL", "1")
    monkeypatch.setenv("PTOC_L2_PREFETCH", prefetch)
    n, rows, cols, tail = 4, 4096, 4096, 256
    rng = np.random.default_rng(9)
    hs = [rng.integers(-(1 << 28), 1 << 28, size=(rows, cols)).astype(np.int32) for _ in range(n)]
    srcs = [to_dev(h) for h in hs]
    d1 = torch.empty(rows, cols, dtype=torch.int32, device="cuda")
    d2 = torch.empty(tail, cols, dtype=torch.int32, device="cuda")
    d3 = torch.empty_like(d2)
    d1_tail = d1[rows - tail:]
    for it in range(6):
        a, b = it % n, (it + 1) % n
        P.ptoc_treduce([srcs[a], srcs[b]], d1, rows, cols, rows, cols, cols, P.SUM, P.I32)
        P.ptoc_treduce([d1_tail, srcs[2][:tail]], d2, tail, cols, tail, cols, cols, P.MAX, P.I32)
        P.ptoc_treduce([d2, d1_tail], d3, tail, cols, tail, cols, cols, P.SUM, P.I32)
        torch.cuda.synchronize()
        o1 = np.zeros((tail, cols), np.int32)
        oracle.treduce([hs[a][rows - tail:], hs[b][rows - tail:]], o1, tail, cols, cols, oracle.SUM, oracle.I32)
        o2 = np.zeros_like(o1)
        oracle.treduce([o1, hs[2][:tail]], o2, tail, cols, cols, oracle.MAX, oracle.I32)
        o3 = np.zeros_like(o1)
        oracle.treduce([o2, o1], o3, tail, cols, cols, oracle.SUM, oracle.I32)
        assert np.array_equal(to_host(d1_tail, np.int32), o1), "iteration %d: d1 tail" % it
        assert np.array_equal(to_host(d2, np.int32), o2), "iteration %d: d2" % it
        assert np.array_equal(to_host(d3, np.int32), o3), "iteration %d: d3" % it
