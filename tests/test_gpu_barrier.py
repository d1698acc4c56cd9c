"""The credit barrier on the GPU (through the C ABI) against the oracle's run
of the same protocol. Complete calls leave every signal window at zero and can
be repeated; ranks that are not launched make the others give up after the
(short) timeout with status = the generation they waited in, leaving exactly
the credits the oracle predicts; ptoc_signal_reset recovers. No wait here can
hang: every wait in the kernel has a deadline and an iteration cap."""
import time

import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import DevBuf

pytestmark = pytest.mark.gpu

TIMEOUT_NS = 200_000_000          # 0.2 s


def windows(n):
    return [DevBuf(np.zeros(n, np.int32)) for _ in range(n)]


def read(ws):
    return np.stack([w.host() for w in ws])


@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 64])
@pytest.mark.parametrize("g", [0, 1, 3, 50])
def test_complete_calls_self_clear(n, g):
    ws = windows(n)
    status = DevBuf(np.full(n, -5, np.int32))
    for _ in range(3):
        P.ptoc_credit_barrier([w.ptr for w in ws], list(range(n)), g, TIMEOUT_NS, status.ptr)
        torch.cuda.synchronize()
        assert np.all(status.host() == 0)
        assert np.all(read(ws) == 0)
    sig = np.zeros((n, n), np.int32)
    assert np.all(oracle.credit_barrier(n, g, np.ones(n), sig) == 0) and np.all(sig == 0)
    assert all(w.guards_intact() for w in ws) and status.guards_intact()


def test_many_generations_local_order_shuffled():
    n, g = 16, 1000
    ws = windows(n)
    ranks = list(np.random.default_rng(3).permutation(n))
    status = DevBuf(np.full(n, -5, np.int32))
    P.ptoc_credit_barrier([w.ptr for w in ws], ranks, g, 5 * TIMEOUT_NS, status.ptr)
    torch.cuda.synchronize()
    assert np.all(status.host() == 0) and np.all(read(ws) == 0)


@pytest.mark.parametrize("n,missing", [(2, [1]), (4, [3]), (8, [1, 6]), (16, [0])])
def test_absent_ranks_time_out_and_leak_credits(n, missing):
    ws = windows(n)
    local = [r for r in range(n) if r not in missing]
    status = DevBuf(np.full(len(local), -5, np.int32))
    t0 = time.time()
    P.ptoc_credit_barrier([w.ptr for w in ws], local, 3, TIMEOUT_NS, status.ptr)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    present = np.array([0 if r in missing else 1 for r in range(n)], np.int32)
    sig = np.zeros((n, n), np.int32)
    want_status = oracle.credit_barrier(n, 3, present, sig)
    assert status.host().tolist() == [int(want_status[r]) for r in local]
    assert np.array_equal(read(ws), sig)
    assert TIMEOUT_NS / 1e9 * 0.9 <= elapsed < 10.0
    # recovery: reset, then a complete call
    P.ptoc_signal_reset([w.ptr for w in ws])
    status2 = DevBuf(np.full(n, -5, np.int32))
    P.ptoc_credit_barrier([w.ptr for w in ws], list(range(n)), 3, TIMEOUT_NS, status2.ptr)
    torch.cuda.synchronize()
    assert np.all(status2.host() == 0) and np.all(read(ws) == 0)
    assert all(w.guards_intact() for w in ws)
