"""ptoc_all_to_all_v_noalloc: the all_to_all_v exchange with its tile counter
in a fixed block of library device memory instead of a per-call allocation.
Two calls in a row on one stream must give exactly what ptoc_all_to_all_v
gives on the same inputs (and what the oracle gives). Collected last, and
independent of the tests before it: every call zeroes the counter itself."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tile_level_collective_gb300 as P
from gpu_util import to_dev, to_host


def test_noalloc_symbol_is_exported():
    assert hasattr(ctypes.CDLL(P.LIB_PATH), "ptoc_all_to_all_v_noalloc")


def test_noalloc_rejects_like_all_to_all_v():
    """Bad arguments fail before any CUDA call (fake addresses, no launch)."""
    A, MB = 0x7F0000000000, 1 << 20
    ins = [A + r * 64 * MB for r in range(4)]
    tgs = [A + (8 + r) * 64 * MB for r in range(4)]
    sc = [A + 16 * 64 * MB + 256 * r for r in range(4)]
    rc = [A + 17 * 64 * MB + 256 * r for r in range(4)]
    f = P.ptoc_all_to_all_v_noalloc
    assert f(ins, tgs[:3], sc, rc, 64, 16, P.BF16, stream=0, check=False) == P.ERR_INVALID_ARG
    assert f(ins, [A] + tgs[1:], sc, rc, 64, 16, P.BF16, stream=0, check=False) == P.ERR_ALIAS
    assert f(ins, tgs, sc, rc, -1, 16, P.BF16, stream=0, check=False) == P.ERR_INVALID_ARG
    # past the kernel's int32 tile index: 64 ranks of 1 TiB windows
    n, size, mr = 64, 8192, 1 << 20
    B, S = 0x100000000000, 1 << 41
    big_in = [B + r * S for r in range(n)]
    big_tg = [B + (n + r) * S for r in range(n)]
    big_sc = [B + 2 * n * S + 256 * r for r in range(n)]
    big_rc = [B + 2 * n * S + (1 << 20) + 256 * r for r in range(n)]
    assert f(big_in, big_tg, big_sc, big_rc, mr * n, size, P.BF16, stream=0, check=False) == P.ERR_UNSUPPORTED


@pytest.mark.gpu
def test_two_calls_in_a_row_match_all_to_all_v():
    n, tr, size = 8, 8 * 48, 520
    rng = np.random.default_rng(2024)
    cases = []
    for k in range(2):
        ins = [rng.integers(0, 2 ** 16, size=(tr, size), dtype=np.uint64).astype(np.uint16) for _ in range(n)]
        sc = [rng.integers(-5, 70, size=n).astype(np.int32) for _ in range(n)]
        cases.append((ins, sc))

    def buffers(ins, sc):
        return ([to_dev(h) for h in ins], [to_dev(c) for c in sc],
                [torch.full((tr, size), -1, dtype=torch.int16, device="cuda") for _ in range(n)],
                [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(n)])

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ref = [buffers(*c) for c in cases]
        got = [buffers(*c) for c in cases]
    torch.cuda.synchronize()
    for d_in, d_sc, d_tg, d_rc in ref:
        P.ptoc_all_to_all_v(d_in, d_tg, d_sc, d_rc, tr, size, P.BF16, stream=stream)
    # two calls back to back on one stream: the second zeroes the shared
    # counter after the first kernel, in stream order
    for d_in, d_sc, d_tg, d_rc in got:
        P.ptoc_all_to_all_v_noalloc(d_in, d_tg, d_sc, d_rc, tr, size, P.BF16, stream=stream)
    stream.synchronize()
    for (ins, sc), r, g in zip(cases, ref, got):
        th = [np.full((tr, size), 0xFFFF, np.uint16) for _ in range(n)]
        rh = [np.zeros(n, np.int32) for _ in range(n)]
        assert oracle.all_to_all_v(ins, th, sc, rh, tr, size, 2) == 0
        for d in range(n):
            assert np.array_equal(to_host(g[2][d], np.uint16), to_host(r[2][d], np.uint16)), "target %d" % d
            assert np.array_equal(g[3][d].cpu().numpy(), r[3][d].cpu().numpy()), "recv_counts %d" % d
            assert np.array_equal(to_host(g[2][d], np.uint16), th[d])
            assert np.array_equal(g[3][d].cpu().numpy(), rh[d])
