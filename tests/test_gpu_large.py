"""Maximum sizes: slices of more than 2^31 elements (64-bit offsets
everywhere), in the flat path (whole rows) and the 2-D path (valid box inside
a wider pitch). Inputs are made on the device from a closed-form integer
formula; the oracle receives the same formula evaluated on the host at
sampled positions (the first and last elements, row ends, random points) and
its result there must equal the GPU's, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P

pytestmark = pytest.mark.gpu

A, B = 2654435761, 40503          # the formula: x_r[k] = (A*k + B*r) mod 2^31 - 2^30


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


@pytest.mark.parametrize("layout", ["flat", "2d"])
def test_more_than_2_31_elements(layout):
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
    dst = torch.full((numel,), 7, dtype=torch.int32, device="cuda")
    for op, ocode in ((P.SUM, oracle.SUM), (P.MAX, oracle.MAX)):
        P.ptoc_treduce(srcs, dst, rows, cols, vr, vc, ld, op, P.I32, root=1)
        torch.cuda.synchronize()
        rng = np.random.default_rng(9)
        ii = np.concatenate([[0, 0, vr - 1, vr - 1, vr // 2], rng.integers(0, vr, 4000)])
        jj = np.concatenate([[0, vc - 1, 0, vc - 1, vc // 2], rng.integers(0, vc, 4000)])
        ks = ii.astype(np.int64) * ld + jj
        got = dst[torch.from_numpy(ks).cuda()].cpu().numpy().reshape(1, -1)
        sv = [host_values(ks, r).reshape(1, -1) for r in range(n)]
        want = np.zeros_like(sv[0])
        assert oracle.treduce(sv, want, 1, want.size, want.size, ocode, oracle.I32, root=1) == 0
        assert np.array_equal(got, want)
        if layout == "2d":
            # the padding (columns vc..ld and rows vr..rows) keeps its fill
            pad_k = np.array([vc, ld - 1, (vr - 1) * ld + vc, vr * ld, numel - 1], dtype=np.int64)
            assert np.all(dst[torch.from_numpy(pad_k).cuda()].cpu().numpy() == 7)
    del srcs, dst
    torch.cuda.empty_cache()


def test_all_to_all_v_runs_past_2_gib():
    """2 ranks of 32 KiB rows, MAX_RECV 80,000: each full pair run is 2.6 GB,
    so byte offsets inside a run pass 2^31. The exchange is a bit copy, so the
    expected target rows are the definition itself: target d row s*MR + i is
    input s row d*MR + i for i < the clamped count, and untouched rows keep
    their fill. Checked on sampled rows, every run's first and last row, and
    the first row past each run."""
    n, size, mr = 2, 8192, 80_000                  # int32 elements: 32 KiB rows
    tr = n * mr
    counts = np.array([[mr, mr - 1], [5, mr + 1000]], dtype=np.int32)   # last one clamps to mr
    ins = [device_slice(tr * size, r).view(tr, size) for r in range(n)]
    tgs = [torch.full((tr, size), -7, dtype=torch.int32, device="cuda") for _ in range(n)]
    sc = [torch.from_numpy(counts[s].copy()).cuda() for s in range(n)]
    rc = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)]
    P.ptoc_all_to_all_v(ins, tgs, sc, rc, tr, size, P.I32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    for d in range(n):
        assert rc[d].cpu().tolist() == [int(min(max(counts[s][d], 0), mr)) for s in range(n)]
        for s in range(n):
            c = int(min(max(counts[s][d], 0), mr))
            rows = {0, c - 1, c, mr - 1} | set(rng.integers(0, mr, size=40).tolist())
            for i in sorted(x for x in rows if 0 <= x < mr):
                got = tgs[d][s * mr + i]
                if i < c:
                    assert torch.equal(got, ins[s][d * mr + i]), (d, s, i)
                else:
                    assert bool((got == -7).all()), (d, s, i)
    del ins, tgs
    torch.cuda.empty_cache()
