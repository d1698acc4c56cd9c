"""Helpers of the GPU parity tests: guard-banded device buffers (so an
out-of-bounds write shows up as a changed guard byte), host <-> device copies
of raw encodings, and the oracle's dtype codes."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

GUARD = 512                    # bytes of sentinel on each side of every buffer
GUARD_BYTE = 0xA5

ORC_DT = {"f32": oracle.F32, "f16": oracle.F16, "bf16": oracle.BF16, "i32": oracle.I32}
ORC_OP = {"sum": oracle.SUM, "max": oracle.MAX, "min": oracle.MIN}
TORCH_T = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i32": torch.int32}
NP_STORE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "i32": np.int32}
ELEM = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}


class DevBuf:
    """A device buffer holding `host` (numpy, storage form), placed `offset`
    bytes past a 512-byte boundary, with GUARD sentinel bytes around it."""

    def __init__(self, host, offset=0):
        host = np.ascontiguousarray(host)
        self.shape, self.np_dtype = host.shape, host.dtype
        self.nbytes = host.nbytes
        self.offset = offset
        self.raw = torch.full((GUARD + offset + self.nbytes + GUARD,), GUARD_BYTE,
                              dtype=torch.uint8, device="cuda")
        self.raw[GUARD + offset:GUARD + offset + self.nbytes] = \
            torch.from_numpy(host.reshape(-1).view(np.uint8).copy()).cuda()

    @property
    def ptr(self):
        return self.raw.data_ptr() + GUARD + self.offset

    def host(self):
        b = self.raw[GUARD + self.offset:GUARD + self.offset + self.nbytes].cpu().numpy()
        return b.view(self.np_dtype).reshape(self.shape)

    def guards_intact(self):
        r = self.raw.cpu().numpy()
        lo = r[:GUARD + self.offset]
        hi = r[GUARD + self.offset + self.nbytes:]
        return bool(np.all(lo == GUARD_BYTE) and np.all(hi == GUARD_BYTE))


def to_dev(host):
    """numpy storage array -> contiguous device tensor with the same bytes."""
    host = np.ascontiguousarray(host)
    if host.dtype == np.uint16:
        return torch.from_numpy(host.view(np.int16)).cuda()
    return torch.from_numpy(host).cuda()


def to_host(t, np_dtype):
    a = t.cpu()
    if np_dtype == np.uint16:
        return a.view(torch.int16).numpy().view(np.uint16)
    return a.numpy()


def bits(a):
    a = np.asarray(a)
    return a.view(np.uint16 if a.itemsize == 2 else np.uint32)


def first_diff(got, want):
    d = np.argwhere(bits(got) != bits(want))
    return "%d elements differ, first at %s: got %s want %s" % (
        len(d), d[:3].tolist(), [hex(int(bits(got)[tuple(i)])) for i in d[:3]],
        [hex(int(bits(want)[tuple(i)])) for i in d[:3]]) if len(d) else "equal"


def oracle_treduce_threaded(srcs, dst, valid_rows, valid_cols, ld, op, dtype, threads=None, root=0):
    """oracle.treduce over contiguous row slices of the valid box, one host
    thread each (ctypes releases the interpreter lock during a call). Each
    element's result depends only on that element of every source, so the
    split run writes exactly what one call writes (checked on the CPU in
    test_oracle_split.py). Returns the first non-zero return code, else 0."""
    threads = threads or os.cpu_count() or 1
    bounds = [valid_rows * t // threads for t in range(threads + 1)]

    def part(t):
        a, b = bounds[t], bounds[t + 1]
        if b <= a:
            return 0
        return oracle.treduce([s[a:b] for s in srcs], dst[a:b], b - a, valid_cols, ld, op, dtype, root)

    with ThreadPoolExecutor(threads) as ex:
        rcs = list(ex.map(part, range(threads)))
    return next((rc for rc in rcs if rc != 0), 0)


def oracle_allreduce_threaded(windows, rows, cols, ld, op, dtype, threads=None):
    """oracle.allreduce over contiguous row slices of every window, one host
    thread each (allreduce acts row by row, so the split run writes exactly
    what one call writes; checked on the CPU in test_oracle_split.py)."""
    threads = threads or os.cpu_count() or 1
    bounds = [rows * t // threads for t in range(threads + 1)]

    def part(t):
        a, b = bounds[t], bounds[t + 1]
        if b <= a:
            return 0
        return oracle.allreduce([w[a:b] for w in windows], b - a, cols, ld, op, dtype)

    with ThreadPoolExecutor(threads) as ex:
        rcs = list(ex.map(part, range(threads)))
    return next((rc for rc in rcs if rc != 0), 0)
