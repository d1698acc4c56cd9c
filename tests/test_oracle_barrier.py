"""Pins for the oracle's credit barrier against what the page states: a
complete call leaves the signal all-zero (self-clearing) and reusable, a rank
that never arrives makes the others time out and leaks credits (hand-worked
golden file), and Eq waits can hang where Ge waits complete."""
import numpy as np
import pytest

from conftest import golden


@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 64])
@pytest.mark.parametrize("g", [0, 1, 2, 7])
def test_complete_call_self_clears(orc, n, g):
    sig = np.zeros((n, n), np.int32)
    for _ in range(3):                       # reusable: every call starts and ends at zero
        st = orc.credit_barrier(n, g, np.ones(n), sig)
        assert np.all(st == 0)
        assert np.all(sig == 0)


def test_missing_rank_golden(orc):
    c = golden("credit_barrier_missing_rank.json")
    sig = np.zeros((c["nranks"], c["nranks"]), np.int32)
    st = orc.credit_barrier(c["nranks"], c["generations"], c["present"], sig)
    assert st.tolist() == c["expected_status"]
    assert sig.tolist() == c["expected_signal"]


@pytest.mark.parametrize("n,missing", [(2, [0]), (4, [3]), (8, [1, 6]), (16, [15])])
def test_missing_ranks_leak_one_credit_per_present_pair(orc, n, missing):
    present = np.ones(n, np.int32)
    present[missing] = 0
    sig = np.zeros((n, n), np.int32)
    st = orc.credit_barrier(n, 3, present, sig)
    want = np.zeros((n, n), np.int32)
    for s in range(n):
        if present[s]:
            want[:, s] = 1
            want[s, s] = 0
    assert np.array_equal(sig, want)
    assert all(st[r] == (1 if present[r] else -1) for r in range(n))
    sig[...] = 0                             # the host-side reset
    assert np.all(orc.credit_barrier(n, 3, np.ones(n), sig) == 0) and np.all(sig == 0)


def test_equality_wait_can_hang_where_ge_completes(orc):
    """The page: a fast peer can advance a cell past the value a waiter looks
    for before it polls, so an equality wait may never unblock. Under the
    oracle's scheduler, 3 ranks and 2 generations: rank 2 passes generation 1
    and notifies for generation 2 before rank 0 polls generation 1."""
    sig = np.zeros((3, 3), np.int32)
    st = orc.credit_barrier(3, 2, np.ones(3), sig, wait_eq=True)
    assert np.any(st > 0)                    # somebody hangs with Eq
    sig = np.zeros((3, 3), np.int32)
    assert np.all(orc.credit_barrier(3, 2, np.ones(3), sig) == 0) and np.all(sig == 0)
