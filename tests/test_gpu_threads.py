"""Several host threads call the library at once, each on its own stream and
buffers (ctypes releases the GIL during the calls, so the library's host code
runs concurrently: its only state is per-device caches kept in atomics).
Every result is checked against the oracle."""
import threading

import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def worker(tid, errors):
    try:
        rng = np.random.default_rng(100 + tid)
        stream = torch.cuda.Stream()
        n, rows, cols = 3 + tid % 4, 64 + 8 * tid, 300 + tid
        hs = [rng.integers(-50, 50, size=(rows, cols)).astype(np.int32) for _ in range(n)]
        with torch.cuda.stream(stream):
            srcs = [to_dev(h) for h in hs]
            dst = torch.empty(rows, cols, dtype=torch.int32, device="cuda")
            wins = [s.clone() for s in srcs]
        for it in range(20):
            op = [P.SUM, P.MAX, P.MIN][it % 3]
            P.ptoc_treduce(srcs, dst, rows, cols, rows, cols, cols, op, P.I32, stream=stream, root=it % n)
            P.ptoc_allreduce(wins, rows, cols, cols, P.MAX, P.I32, stream=stream)
            stream.synchronize()
            want = np.zeros((rows, cols), np.int32)
            oracle.treduce(hs, want, rows, cols, cols, [oracle.SUM, oracle.MAX, oracle.MIN][it % 3],
                           oracle.I32, root=it % n)
            if not np.array_equal(to_host(dst, np.int32), want):
                errors.append("thread %d iteration %d: treduce differs" % (tid, it))
                return
        ow = [h.copy() for h in hs]
        oracle.allreduce(ow, rows, cols, cols, oracle.MAX, oracle.I32)
        for w, o in zip(wins, ow):
            if not np.array_equal(to_host(w, np.int32), o):
                errors.append("thread %d: allreduce differs" % tid)
                return
    except Exception as e:  # reported to the main thread
        errors.append("thread %d: %r" % (tid, e))


@pytest.mark.parametrize("form", ["regs", "bulk", "tma"])
def test_concurrent_host_threads(form, monkeypatch):
    """With PTOC_REDUCE_STAGING=bulk the 16-byte-aligned cases (threads 0 and
    4) run the staged form, concurrently with the others' register form."""
    monkeypatch.setenv("PTOC_REDUCE_STAGING", form)
    P.ptoc_wait_faults()
    errors = []
    threads = [threading.Thread(target=worker, args=(t, errors)) for t in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert P.ptoc_wait_faults() == 0
