"""The host variant of the credit barrier ("Distributed Operators (N6)",
Barrier-signal protocol): ranks are Python threads (the call releases the GIL)
or separate processes sharing one mapping. A complete call leaves every cell
at zero whatever the interleaving and can be repeated; a rank that never
arrives makes the others give up in generation 1 and leaves exactly the
credits the oracle's step machine leaves; bad arguments are refused. No GPU
is used."""
import multiprocessing as mp
import threading
from multiprocessing import shared_memory

import numpy as np
import pytest

import oracle
import tile_level_collective_gb300 as P


def windows(sig):
    """Row p of the [N, N] int32 array is rank p's window."""
    n = sig.shape[0]
    return [sig.ctypes.data + 4 * n * p for p in range(n)]


def run_threads(sig, ranks, generations, timeout_ns):
    status = np.full(sig.shape[0], -1, np.int32)
    win = windows(sig)

    def rank_main(r):
        P.ptoc_credit_barrier_host(win, r, generations, timeout_ns, status.ctypes.data + 4 * r)

    ts = [threading.Thread(target=rank_main, args=(r,)) for r in ranks]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=120)
        assert not t.is_alive()
    return status


@pytest.mark.parametrize("n", [1, 2, 3, 8, 24])
@pytest.mark.parametrize("g", [0, 1, 7, 100])
def test_threads_complete_calls_self_clear(n, g):
    sig = np.zeros((n, n), np.int32)
    for _ in range(3):                        # reusable: each call starts and ends at zero
        st = run_threads(sig, range(n), g, 20 * 10 ** 9)
        assert np.all(st == 0)
        assert np.all(sig == 0)


@pytest.mark.parametrize("n,missing", [(2, [0]), (3, [2]), (8, [1, 6]), (16, [15])])
def test_threads_absent_ranks_leave_the_oracles_credits(n, missing):
    present = np.ones(n, np.int32)
    present[missing] = 0
    sig = np.zeros((n, n), np.int32)
    st = run_threads(sig, [r for r in range(n) if present[r]], 3, 100 * 10 ** 6)
    want_sig = np.zeros((n, n), np.int32)
    want_st = oracle.credit_barrier(n, 3, present, want_sig)
    assert np.array_equal(sig, want_sig)
    for r in range(n):
        if present[r]:
            assert st[r] == want_st[r] == 1   # gave up waiting in generation 1
    sig[...] = 0                              # the host-side reset, then a complete call
    assert np.all(run_threads(sig, range(n), 3, 20 * 10 ** 9) == 0) and np.all(sig == 0)


def _process_rank(name, n, rank, generations, timeout_ns, skip):
    shm = shared_memory.SharedMemory(name=name)
    try:
        cells = np.ndarray((n * n + n,), np.int32, buffer=shm.buf)
        if rank in skip:
            return                            # this rank never arrives
        base = cells.ctypes.data
        win = [base + 4 * n * p for p in range(n)]
        P.ptoc_credit_barrier_host(win, rank, generations, timeout_ns, base + 4 * (n * n + rank))
    finally:
        del cells
        shm.close()


def run_processes(n, generations, timeout_ns, skip=()):
    shm = shared_memory.SharedMemory(create=True, size=4 * (n * n + n))
    try:
        cells = np.ndarray((n * n + n,), np.int32, buffer=shm.buf)
        cells[:] = 0
        cells[n * n:] = -1
        ctx = mp.get_context("spawn")
        ps = [ctx.Process(target=_process_rank, args=(shm.name, n, r, generations, timeout_ns, tuple(skip)))
              for r in range(n)]
        for p in ps:
            p.start()
        for p in ps:
            p.join(timeout=120)
            assert p.exitcode == 0
        sig = cells[:n * n].reshape(n, n).copy()
        st = cells[n * n:].copy()
        del cells
        return sig, st
    finally:
        shm.close()
        shm.unlink()


def test_processes_complete_and_absent():
    """Ranks as processes on a shared mapping: a complete call self-clears;
    with rank 2 absent the other two give up and leave the oracle's credits."""
    n = 3
    sig, st = run_processes(n, 20, 20 * 10 ** 9)
    assert np.all(st == 0) and np.all(sig == 0)
    sig, st = run_processes(n, 4, 200 * 10 ** 6, skip=(2,))
    want_sig = np.zeros((n, n), np.int32)
    want_st = oracle.credit_barrier(n, 4, np.array([1, 1, 0]), want_sig)
    assert np.array_equal(sig, want_sig)
    assert st[0] == want_st[0] == 1 and st[1] == want_st[1] == 1 and st[2] == -1


def test_host_barrier_rejects():
    sig = np.zeros((4, 4), np.int32)
    win = windows(sig)
    out = np.zeros(2, np.int32)
    ST = out.ctypes.data
    B = P.ptoc_credit_barrier_host
    assert B(win, 4, 1, 10 ** 9, ST, check=False) == P.ERR_INVALID_ARG        # rank out of range
    assert B(win, -1, 1, 10 ** 9, ST, check=False) == P.ERR_INVALID_ARG
    assert B(win, 0, -1, 10 ** 9, ST, check=False) == P.ERR_INVALID_ARG       # generations
    assert B(win, 0, 1, 0, ST, check=False) == P.ERR_INVALID_ARG              # timeout
    assert B(win, 0, 1, 61 * 10 ** 9, ST, check=False) == P.ERR_INVALID_ARG
    assert B(win, 0, 1, 10 ** 9, 0, check=False) == P.ERR_INVALID_ARG         # status
    assert B(win, 0, 1, 10 ** 9, ST + 2, check=False) == P.ERR_INVALID_ARG
    assert B([win[0], 0, win[2], win[3]], 0, 1, 10 ** 9, ST, check=False) == P.ERR_INVALID_ARG
    assert B([win[0], win[0] + 2, win[2], win[3]], 0, 1, 10 ** 9, ST, check=False) == P.ERR_INVALID_ARG
    assert B([win[0], win[0] + 4, win[2], win[3]], 0, 1, 10 ** 9, ST, check=False) == P.ERR_ALIAS
    assert B(win, 0, 1, 10 ** 9, win[3] + 4, check=False) == P.ERR_ALIAS      # status over a window
    assert np.all(sig == 0) and np.all(out == 0)                               # nothing ran


def test_threads_random_presence_against_the_oracle():
    """Seeded random rank counts, generations and presence patterns: the
    statuses and the cells the threads leave equal the oracle's (with a rank
    absent every present rank gives up in generation 1, whatever the
    interleaving; with all present everything clears)."""
    rng = np.random.default_rng(11)
    for _ in range(24):
        n = int(rng.integers(1, 13))
        g = int(rng.integers(1, 6))
        present = (rng.random(n) < 0.8).astype(np.int32)
        if not present.any():
            present[int(rng.integers(n))] = 1
        sig = np.zeros((n, n), np.int32)
        timeout = 20 * 10 ** 9 if present.all() else 30 * 10 ** 6
        st = run_threads(sig, [r for r in range(n) if present[r]], g, timeout)
        want_sig = np.zeros((n, n), np.int32)
        want_st = oracle.credit_barrier(n, g, present, want_sig)
        assert np.array_equal(sig, want_sig), (n, g, present)
        for r in range(n):
            if present[r]:
                assert st[r] == want_st[r], (n, g, present, r)
