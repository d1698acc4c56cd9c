"""Maximum sizes: slices of more than 2^31 elements (64-bit offsets
everywhere), in the flat path (whole rows) and the 2-D path (valid box inside
a wider pitch), and an all_to_all_v whose pair runs pass 2^31 bytes. Inputs
are made on the device from a closed-form integer formula; the oracle receives
the same formula evaluated on the host (numpy, in row chunks on host threads),
and every element of every result, padding included, must equal the
oracle's, bit for bit."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import oracle_treduce_threaded

pytestmark = pytest.mark.gpu

A, B = 2654435761, 40503          # the formula: x_r[k] = (A*k + B*r) mod 2^31 - 2^30
THREADS = os.cpu_count() or 1


def device_slice(numel, r):
    out = torch.empty(numel, dtype=torch.int32, device="cuda")
    chunk = 1 << 28
    for s in range(0, numel, chunk):
        k = torch.arange(s, min(s + chunk, numel), dtype=torch.int64, device="cuda")
        out[s:s + k.numel()] = ((k * A + B * r) % (1 << 31) - (1 << 30)).to(torch.int32)
        del k
    return out


def host_values(ks, r):
    ks = np.asarray(ks, dtype=np.int64)
    return ((ks * A + B * r) % (1 << 31) - (1 << 30)).astype(np.int32)


def host_rows(r, a, b, ld):
    """Rows [a, b) of rank r's slice as int32 [b - a, ld], from the formula,
    computed in pieces on host threads (numpy releases the interpreter lock)."""
    out = np.empty((b - a) * ld, dtype=np.int32)
    n = out.size
    bounds = [n * t // THREADS for t in range(THREADS + 1)]

    def part(t):
        step = 1 << 22                  # bounded temporaries per thread
        for lo in range(bounds[t], bounds[t + 1], step):
            hi = min(bounds[t + 1], lo + step)
            out[lo:hi] = host_values(np.arange(a * ld + lo, a * ld + hi, dtype=np.int64), r)

    with ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(part, range(THREADS)))
    return out.reshape(b - a, ld)


@pytest.mark.parametrize("layout", ["flat", "2d"])
def test_more_than_2_31_elements(layout):
    """Sum and Max over 3 ranks, root 1: every element of both results (the
    valid box and the padding around it, which keeps its fill) against the
    oracle, compared in chunks of rows."""
    n = 3
    if layout == "flat":
        rows, cols, ld = 1 << 16, 1 << 15 | 8, 1 << 15 | 8      # 2^31 + 2^19 elements, whole rows
        vr, vc = rows, cols
    else:
        rows, cols, ld = 40000, 54000, 54016                   # 2.16e9 elements, valid box narrower
        vr, vc = rows - 3, cols - 5
    numel = rows * ld
    assert numel > 2 ** 31
    srcs = [device_slice(numel, r) for r in range(n)]
    ops = ((P.SUM, oracle.SUM), (P.MAX, oracle.MAX))
    dsts = []
    for op, _ in ops:
        d = torch.full((numel,), 7, dtype=torch.int32, device="cuda")
        P.ptoc_treduce(srcs, d, rows, cols, vr, vc, ld, op, P.I32, root=1)
        dsts.append(d)
    torch.cuda.synchronize()
    # spot check: the host formula is the one the device evaluated
    ks = np.array([0, ld - 1, numel // 2, numel - 1], dtype=np.int64)
    for r in range(n):
        assert np.array_equal(srcs[r][torch.from_numpy(ks).cuda()].cpu().numpy(), host_values(ks, r))
    del srcs
    torch.cuda.empty_cache()
    chunk = max(1, (1 << 27) // ld)
    compared = 0
    for a in range(0, rows, chunk):
        b = min(rows, a + chunk)
        hs = [host_rows(r, a, b, ld) for r in range(n)]
        vrows = max(0, min(vr, b) - a)
        for (op, ocode), d in zip(ops, dsts):
            want = np.full((b - a, ld), 7, dtype=np.int32)
            if vrows:
                assert oracle_treduce_threaded([h[:vrows] for h in hs], want[:vrows], vrows, vc, ld, ocode,
                                               oracle.I32, root=1) == 0
            got = d.view(rows, ld)[a:b].cpu().numpy()
            assert np.array_equal(got, want), "op %d rows %d..%d: %d elements differ" % (
                op, a, b - 1, int((got != want).sum()))
        compared += (b - a) * ld
    assert compared == numel
    del dsts
    torch.cuda.empty_cache()


def test_all_to_all_v_runs_past_2_gib():
    """2 ranks of 32 KiB rows, MAX_RECV 80,000: each full pair run is 2.6 GB,
    so byte offsets inside a run pass 2^31. Every row of both targets (and
    the recv counts) against the oracle's all_to_all_v over the same inputs,
    computed from the formula on the host."""
    n, size, mr = 2, 8192, 80_000                  # int32 elements: 32 KiB rows
    tr = n * mr
    counts = np.array([[mr, mr - 1], [5, mr + 1000]], dtype=np.int32)   # last one clamps to mr
    ins = [device_slice(tr * size, r).view(tr, size) for r in range(n)]
    tgs = [torch.full((tr, size), -7, dtype=torch.int32, device="cuda") for _ in range(n)]
    sc = [torch.from_numpy(counts[s].copy()).cuda() for s in range(n)]
    rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.ptoc_all_to_all_v(ins, tgs, sc, rc, tr, size, P.I32)
    torch.cuda.synchronize()
    del ins
    torch.cuda.empty_cache()
    h_in = [host_rows(r, 0, tr, size) for r in range(n)]
    h_tg = [np.full((tr, size), -7, dtype=np.int32) for _ in range(n)]
    h_rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
    assert oracle.all_to_all_v(h_in, h_tg, [c.copy() for c in counts], h_rc, tr, size, 4) == 0
    del h_in
    for d in range(n):
        assert np.array_equal(rc[d].cpu().numpy(), h_rc[d])
        step = 1 << 14
        for a in range(0, tr, step):
            got = tgs[d][a:a + step].cpu().numpy()
            assert np.array_equal(got, h_tg[d][a:a + step]), "target %d rows %d.." % (d, a)
    del tgs
    torch.cuda.empty_cache()
