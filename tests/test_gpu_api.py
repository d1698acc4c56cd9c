"""Every Python convenience over torch tensors on the GPU, against the oracle
on the same host data (the conveniences derive rows, cols and the pitch from
the tensors and run on torch's current stream)."""
import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P

pytestmark = pytest.mark.gpu


def host_i32(rng, n, rows, cols):
    return [rng.integers(-1000, 1000, size=(rows, cols)).astype(np.int32) for _ in range(n)]


def dev(hs):
    return [torch.from_numpy(h.copy()).cuda() for h in hs]


def test_treduce_and_window_conveniences():
    rng = np.random.default_rng(4)
    n, rows, cols = 5, 30, 100
    hs = host_i32(rng, n, rows, cols)
    out = torch.zeros(rows, cols, dtype=torch.int32, device="cuda")
    P.treduce(dev(hs), out, op="max", valid_rows=21, valid_cols=77, root=2)
    want = np.zeros((rows, cols), np.int32)
    assert oracle.treduce(hs, want, 21, 77, cols, oracle.MAX, oracle.I32, root=2) == 0
    assert np.array_equal(out.cpu().numpy(), want)

    w = dev(hs)
    P.reduce_scatter(w, op="sum")
    P.allgather(w)
    hw = [h.copy() for h in hs]
    assert oracle.reduce_scatter(hw, rows, cols, cols, oracle.SUM, oracle.I32) == 0
    assert oracle.allgather(hw, rows, cols, cols, oracle.I32) == 0
    for a, b in zip(w, hw):
        assert np.array_equal(a.cpu().numpy(), b)

    w = dev(hs)
    P.allreduce(w, op="prod")
    hw = [h.copy() for h in hs]
    assert oracle.allreduce(hw, rows, cols, cols, oracle.PROD, oracle.I32) == 0
    for a, b in zip(w, hw):
        assert np.array_equal(a.cpu().numpy(), b)

    w = dev(hs)
    P.broadcast(w, root=3)
    hw = [h.copy() for h in hs]
    assert oracle.broadcast(hw, 3, rows, cols, cols, oracle.I32) == 0
    for a, b in zip(w, hw):
        assert np.array_equal(a.cpu().numpy(), b)


@pytest.mark.parametrize("noalloc", [False, True])
def test_exchange_conveniences(noalloc):
    rng = np.random.default_rng(5)
    n, tr, size = 4, 4 * 12, 33
    mr = tr // n
    ins = host_i32(rng, n, tr, size)
    sc = [rng.integers(-2, mr + 3, size=n).astype(np.int32) for _ in range(n)]
    d_in = dev(ins)
    d_tg = [torch.full((tr, size), -9, dtype=torch.int32, device="cuda") for _ in range(n)]
    d_sc = dev(sc)
    d_rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.all_to_all_v(d_in, d_tg, d_sc, d_rc, noalloc=noalloc)
    th = [np.full((tr, size), -9, np.int32) for _ in range(n)]
    rh = [np.zeros(n, np.int32) for _ in range(n)]
    assert oracle.all_to_all_v(ins, th, sc, rh, tr, size, 4) == 0
    for d in range(n):
        assert np.array_equal(d_tg[d].cpu().numpy(), th[d])
        assert np.array_equal(d_rc[d].cpu().numpy(), rh[d])

    outs = host_i32(rng, n, tr, size)
    d_out = dev(outs)
    P.all_to_all_v_combine(d_tg, d_out, d_rc, atomic="add")
    assert oracle.all_to_all_v_combine(th, outs, rh, tr, size, oracle.ATOMIC_ADD, oracle.I32) == 0
    for s in range(n):
        assert np.array_equal(d_out[s].cpu().numpy(), outs[s])

    d_tg2 = [torch.full((tr, size), -9, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.all_to_all(d_in, d_tg2)
    th2 = [np.full((tr, size), -9, np.int32) for _ in range(n)]
    assert oracle.all_to_all(ins, th2, tr, size, 4) == 0
    for d in range(n):
        assert np.array_equal(d_tg2[d].cpu().numpy(), th2[d])
