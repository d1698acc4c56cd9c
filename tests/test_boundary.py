"""The C ABI without a GPU: the library loads, exports every function
include/ptoc.h declares, and rejects bad arguments with the documented status
before any CUDA call. Every case here breaks at least one rule (or is empty),
so no case can reach a kernel launch, with or without a GPU.
Device addresses below are fake and never dereferenced."""
import ctypes
import os
import re

import pytest

import tile_level_collective_gb300 as P
from conftest import ROOT

A = 0x7F0000000000          # fake, 4 KiB-aligned device addresses
MB = 1 << 20


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ptoc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ptoc_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    assert declared_functions() == ["ptoc_all_to_all", "ptoc_all_to_all_v", "ptoc_all_to_all_v_combine",
                                    "ptoc_all_to_all_v_noalloc", "ptoc_allgather", "ptoc_allreduce", "ptoc_broadcast",
                                    "ptoc_credit_barrier", "ptoc_credit_barrier_host", "ptoc_reduce_scatter",
                                    "ptoc_signal_reset",
                                    "ptoc_status_string", "ptoc_treduce", "ptoc_wait_faults"]


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(P.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_wait_faults_refuses_a_null_output():
    lib = ctypes.CDLL(P.LIB_PATH)
    lib.ptoc_wait_faults.argtypes = [ctypes.c_void_p]
    assert lib.ptoc_wait_faults(None) == P.ERR_INVALID_ARG


def test_status_strings():
    assert P.ptoc_status_string(P.OK) == "PTOC_OK"
    assert P.ptoc_status_string(P.ERR_ALIAS) == "PTOC_ERR_ALIAS"
    assert P.ptoc_status_string(P.ERR_UNSUPPORTED) == "PTOC_ERR_UNSUPPORTED"
    assert P.ptoc_status_string(99) == "PTOC_ERR_UNKNOWN"


def srcs(n, stride=64 * MB, base=A):
    return [base + r * stride for r in range(n)]


DST = A + 200 * 64 * MB


def tr(tensors=None, dst=DST, rows=8, cols=8, vr=8, vc=8, ld=8, op=P.SUM, dt=P.F32, root=0):
    tensors = srcs(4) if tensors is None else tensors
    return P.ptoc_treduce(tensors, dst, rows, cols, vr, vc, ld, op, dt, stream=0, root=root, check=False)


@pytest.mark.parametrize("kw,status", [
    (dict(tensors=[]), P.ERR_INVALID_ARG),                       # nranks 0
    (dict(tensors=srcs(65, stride=MB)), P.ERR_INVALID_ARG),      # nranks > 64
    (dict(root=-1), P.ERR_INVALID_ARG),                          # root outside [0, N)
    (dict(root=4), P.ERR_INVALID_ARG),
    (dict(tensors=[A, 0, A + 2 * 64 * MB, A + 3 * 64 * MB]), P.ERR_INVALID_ARG),  # null slice
    (dict(dst=0), P.ERR_INVALID_ARG),
    (dict(dt=7), P.ERR_INVALID_ARG),
    (dict(op=P.PROD), P.ERR_UNSUPPORTED),                        # reserved ABI value
    (dict(op=9), P.ERR_INVALID_ARG),
    (dict(rows=-1), P.ERR_INVALID_ARG),
    (dict(vr=9), P.ERR_INVALID_ARG),                             # valid > physical
    (dict(vc=9), P.ERR_INVALID_ARG),
    (dict(cols=9, vc=8, ld=8), P.ERR_INVALID_ARG),               # cols > ld
    (dict(ld=-3), P.ERR_INVALID_ARG),
    (dict(dst=DST + 2), P.ERR_INVALID_ARG),                      # f32 dst not 4-byte aligned
    (dict(tensors=[A + 1, A + 64 * MB]), P.ERR_INVALID_ARG),     # misaligned source
    (dict(rows=2 ** 40, cols=2 ** 40, vr=1, vc=1, ld=2 ** 40), P.ERR_INVALID_ARG),  # size overflow
    (dict(dst=A + 64 * MB + 16), P.ERR_ALIAS),                   # dst overlaps rank 1
    (dict(dst=A + 64 * MB, root=0), P.ERR_ALIAS),                # dst == a non-root slice
])
def test_treduce_rejects(kw, status):
    assert tr(**kw) == status


def test_treduce_empty_region_is_ok_without_launch():
    assert tr(vr=0) == P.OK
    assert tr(vc=0) == P.OK
    assert tr(rows=0, cols=0, vr=0, vc=0, ld=0) == P.OK


def test_treduce_raises_ptoc_error():
    with pytest.raises(P.PtocError) as e:
        P.ptoc_treduce(srcs(2), DST, 4, 4, 4, 4, 4, P.PROD, P.F32, stream=0)
    assert e.value.status == P.ERR_UNSUPPORTED


def test_reduce_scatter_and_allgather_reject():
    w = srcs(4)
    overl = [A, A + 100, A + 2 * 64 * MB, A + 3 * 64 * MB]
    assert P.ptoc_reduce_scatter(overl, 64, 64, 64, P.SUM, P.F32, stream=0, check=False) == P.ERR_ALIAS
    assert P.ptoc_reduce_scatter(w, 64, 64, 64, 7, P.F32, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_reduce_scatter(w, 64, 65, 64, P.SUM, P.F32, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_reduce_scatter(w, 64, 64, 64, P.SUM, 5, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_reduce_scatter([], 64, 64, 64, P.SUM, P.F32, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_reduce_scatter(w, 0, 64, 64, P.SUM, P.F32, stream=0, check=False) == P.OK
    assert P.ptoc_allgather(overl, 64, 64, 64, P.F16, stream=0, check=False) == P.ERR_ALIAS
    assert P.ptoc_allgather([A + 1, A + 64 * MB], 4, 4, 4, P.F16, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_allgather(w, 64, 0, 64, P.F16, stream=0, check=False) == P.OK
    assert P.ptoc_allgather([A], 64, 64, 64, P.F16, stream=0, check=False) == P.OK   # one rank: nothing to move


A2AV_CALL = {"call": P.ptoc_all_to_all_v}


def a2av(inputs=None, targets=None, sc=None, rc=None, tr_=64, size=16, dt=P.BF16):
    n = 4
    inputs = srcs(n) if inputs is None else inputs
    targets = srcs(n, base=A + 8 * 64 * MB) if targets is None else targets
    sc = [A + 16 * 64 * MB + 256 * r for r in range(n)] if sc is None else sc
    rc = [A + 17 * 64 * MB + 256 * r for r in range(n)] if rc is None else rc
    return A2AV_CALL["call"](inputs, targets, sc, rc, tr_, size, dt, stream=0, check=False)


@pytest.mark.parametrize("call", ["ptoc_all_to_all_v", "ptoc_all_to_all_v_noalloc"])
def test_all_to_all_v_rejects(call, monkeypatch):
    """The same checks guard the allocating and the no-allocation entry point."""
    monkeypatch.setitem(A2AV_CALL, "call", getattr(P, call))
    assert a2av(targets=srcs(3, base=A + 8 * 64 * MB)) == P.ERR_INVALID_ARG        # N mismatch
    assert a2av(sc=[A + 16 * 64 * MB, 0, A + 16 * 64 * MB + 512, A + 16 * 64 * MB + 768]) == P.ERR_INVALID_ARG
    assert a2av(rc=[A + 17 * 64 * MB + 2, A + 17 * 64 * MB + 256, A + 17 * 64 * MB + 512,
                    A + 17 * 64 * MB + 768]) == P.ERR_INVALID_ARG                  # counts misaligned
    assert a2av(tr_=-1) == P.ERR_INVALID_ARG
    assert a2av(size=-1) == P.ERR_INVALID_ARG
    assert a2av(dt=11) == P.ERR_INVALID_ARG
    # outputs overlapping anything
    assert a2av(targets=[A] + srcs(3, base=A + 9 * 64 * MB)) == P.ERR_ALIAS                 # target = input
    assert a2av(targets=[A + 8 * 64 * MB, A + 8 * 64 * MB + 64] + srcs(2, base=A + 10 * 64 * MB)) == P.ERR_ALIAS
    assert a2av(rc=[A + 16 * 64 * MB + 4] + [A + 17 * 64 * MB + 256 * r for r in range(1, 4)]) == P.ERR_ALIAS
    assert a2av(rc=[A + 8 * 64 * MB + 8] + [A + 17 * 64 * MB + 256 * r for r in range(1, 4)]) == P.ERR_ALIAS


def test_allreduce_and_broadcast_reject():
    w = srcs(4)
    overl = [A, A + 100, A + 2 * 64 * MB, A + 3 * 64 * MB]
    assert P.ptoc_allreduce(overl, 64, 64, 64, P.SUM, P.F32, stream=0, check=False) == P.ERR_ALIAS
    assert P.ptoc_allreduce(w, 64, 64, 64, 7, P.F32, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_allreduce(w, 64, 65, 64, P.PROD, P.F32, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_allreduce(w, 0, 64, 64, P.PROD, P.F32, stream=0, check=False) == P.OK
    assert P.ptoc_allreduce([A], 64, 64, 64, P.PROD, P.F32, stream=0, check=False) == P.OK    # one rank
    assert P.ptoc_reduce_scatter(w, 0, 64, 64, P.PROD, P.F32, stream=0, check=False) == P.OK  # Prod allowed
    assert P.ptoc_broadcast(w, 64, 64, 64, P.F32, stream=0, root=4, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_broadcast(w, 64, 64, 64, P.F32, stream=0, root=-1, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_broadcast(overl, 64, 64, 64, P.F32, stream=0, root=0, check=False) == P.ERR_ALIAS
    assert P.ptoc_broadcast(w, 64, 0, 64, P.F32, stream=0, root=1, check=False) == P.OK


def test_all_to_all_and_combine_reject():
    ins, tgs = srcs(4), srcs(4, base=A + 8 * 64 * MB)
    assert P.ptoc_all_to_all(ins, tgs[:3], 64, 16, P.BF16, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_all_to_all(ins, [A] + tgs[1:], 64, 16, P.BF16, stream=0, check=False) == P.ERR_ALIAS
    assert P.ptoc_all_to_all(ins, tgs, -1, 16, P.BF16, stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_all_to_all(ins, tgs, 3, 16, P.BF16, stream=0, check=False) == P.OK      # chunk 0
    rc = [A + 17 * 64 * MB + 256 * r for r in range(4)]
    C = P.ptoc_all_to_all_v_combine
    assert C(ins, tgs, rc, 64, 16, 2, P.BF16, stream=0, check=False) == P.ERR_INVALID_ARG  # atomic
    assert C(ins, tgs, rc, 64, 16, P.ATOMIC_ADD, 9, stream=0, check=False) == P.ERR_INVALID_ARG
    assert C(ins, [A + 64 * MB] + tgs[1:], rc, 64, 16, P.ATOMIC_ADD, P.BF16, stream=0,
             check=False) == P.ERR_ALIAS                                                   # output = window
    assert C(ins, [rc[0] - 8] + tgs[1:], rc, 64, 16, P.ATOMIC_ADD, P.BF16, stream=0,
             check=False) == P.ERR_ALIAS                                                   # output over counts
    assert C(ins, tgs, [rc[0] + 2] + rc[1:], 64, 16, P.ATOMIC_NONE, P.BF16, stream=0,
             check=False) == P.ERR_INVALID_ARG                                             # misaligned counts
    assert C(ins, tgs, rc, 3, 16, P.ATOMIC_ADD, P.BF16, stream=0, check=False) == P.OK     # MAX_RECV 0


def test_credit_barrier_rejects():
    sig = [A + 512 * r for r in range(4)]
    ST = A + 64 * MB
    B = P.ptoc_credit_barrier
    assert B(sig, [], 1, 10 ** 9, ST, stream=0, check=False) == P.ERR_INVALID_ARG         # no local rank
    assert B(sig, [0, 4], 1, 10 ** 9, ST, stream=0, check=False) == P.ERR_INVALID_ARG     # rank out of range
    assert B(sig, [1, 1], 1, 10 ** 9, ST, stream=0, check=False) == P.ERR_INVALID_ARG     # duplicate
    assert B(sig, [0], -1, 10 ** 9, ST, stream=0, check=False) == P.ERR_INVALID_ARG       # generations
    assert B(sig, [0], 1, 0, ST, stream=0, check=False) == P.ERR_INVALID_ARG              # timeout
    assert B(sig, [0], 1, 61 * 10 ** 9, ST, stream=0, check=False) == P.ERR_INVALID_ARG
    assert B(sig, [0], 1, 10 ** 9, 0, stream=0, check=False) == P.ERR_INVALID_ARG         # status
    assert B(sig, [0], 1, 10 ** 9, ST + 2, stream=0, check=False) == P.ERR_INVALID_ARG
    assert B([A, A + 8, A + 1024, A + 2048], [0], 1, 10 ** 9, ST, stream=0, check=False) == P.ERR_ALIAS
    assert B(sig, [0, 1], 1, 10 ** 9, sig[2] + 4, stream=0, check=False) == P.ERR_ALIAS  # status over a window
    assert P.ptoc_signal_reset([A, 0], stream=0, check=False) == P.ERR_INVALID_ARG
    assert P.ptoc_signal_reset([A + 2], stream=0, check=False) == P.ERR_INVALID_ARG


def test_device_count_exchanges_reject_int32_tile_overflow():
    """64 ranks, 8192-wide bf16 rows, MAX_RECV = 2^20: 4096 pairs x 2^19 tiles
    of 32 KiB is past the int32 tile index of the claiming kernel, so the call
    returns UNSUPPORTED before any CUDA call (fake, disjoint 1 TiB windows)."""
    n, size, mr = 64, 8192, 1 << 20
    tr_ = mr * n
    B, S = 0x100000000000, 1 << 41
    ins = [B + r * S for r in range(n)]
    tgs = [B + (n + r) * S for r in range(n)]
    sc = [B + 2 * n * S + 256 * r for r in range(n)]
    rc = [B + 2 * n * S + (1 << 20) + 256 * r for r in range(n)]
    assert P.ptoc_all_to_all_v(ins, tgs, sc, rc, tr_, size, P.BF16, stream=0, check=False) == P.ERR_UNSUPPORTED
    assert P.ptoc_all_to_all_v_noalloc(ins, tgs, sc, rc, tr_, size, P.BF16, stream=0,
                                       check=False) == P.ERR_UNSUPPORTED
    assert P.ptoc_all_to_all_v_combine(ins, tgs, rc, tr_, size, P.ATOMIC_ADD, P.BF16, stream=0,
                                       check=False) == P.ERR_UNSUPPORTED


def test_package_refuses_to_import_without_the_library(tmp_path):
    """No fallback path: a copy of the binding without libptoc.so beside it
    raises ImportError at import, naming the missing library."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "tile_level_collective_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "tile_level_collective_gb300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import tile_level_collective_gb300"], cwd=tmp_path,
                       capture_output=True, text=True, env=dict(os.environ, PYTHONPATH=str(tmp_path)))
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libptoc.so is not built" in r.stderr
