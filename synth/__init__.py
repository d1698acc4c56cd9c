"""Seeded synthetic inputs for the TREDUCE / window-collective workloads.

Shared by the tests, the smoke check and the benchmark, for both the CUDA
library and the oracle. It holds none of the reduction or data-movement
arithmetic: it turns (seed, element counter) into values (``synth.c``, a
counter-based SplitMix64 stream) and lays them out in the workloads' shapes.
Conversions of generated binary32 values to bfloat16 / float16 are done by
library routines (torch for bfloat16, numpy for float16), both round to
nearest even.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

RAW64, UNIF_F32, NORM_F32, UNIF_I32, BITS16 = range(5)
BASE_SEED = 1234
_lib = None


def build(force=False):
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.synth_fill.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                 ctypes.c_double, ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_void_p, ctypes.c_int]
        L.synth_fill.restype = ctypes.c_int
        _lib = L
    return _lib


_OUT_TYPE = {RAW64: np.uint64, UNIF_F32: np.float32, NORM_F32: np.float32,
             UNIF_I32: np.int32, BITS16: np.uint16}


def fill(kind, seed, n, start=0, lo=0.0, hi=0.0, lo_i=0, hi_i=0, out=None):
    """Elements start .. start+n-1 of stream `seed`, of the given kind."""
    if out is None:
        out = np.empty(int(n), dtype=_OUT_TYPE[kind])
    assert out.dtype == _OUT_TYPE[kind] and out.size == n and out.flags.c_contiguous
    rc = _L().synth_fill(kind, seed & (2**64 - 1), start, int(n), float(lo), float(hi),
                         int(lo_i), int(hi_i), out.ctypes.data, os.cpu_count() or 1)
    if rc != 0:
        raise ValueError("synth_fill rejected its arguments")
    return out


def at(kind, seed, counters, lo=0.0, hi=0.0, lo_i=0, hi_i=0):
    """Values at arbitrary counters (for sampled checks): one fill per counter."""
    counters = np.asarray(counters, dtype=np.int64).ravel()
    out = np.empty(counters.size, dtype=_OUT_TYPE[kind])
    for idx, k in enumerate(counters):
        out[idx] = fill(kind, seed, 1, start=int(k), lo=lo, hi=hi, lo_i=lo_i, hi_i=hi_i)[0]
    return out


def f32_to_bf16_bits(x):
    """binary32 -> bfloat16 encodings (torch's RNE conversion)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_to_f16_bits(x):
    """binary32 -> float16 encodings (numpy's RNE conversion)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


# --------------------------------------------------------------------------
# Workload recipes. A rank slice is a row-major [rows, ld] buffer whose valid
# box [valid_rows, valid_cols] holds the generated values, element (i, j)
# taking counter i*valid_cols + j of the rank's stream (seed BASE_SEED + r);
# everything outside the box holds the padding sentinel.
# --------------------------------------------------------------------------

DT_F32, DT_F16, DT_BF16, DT_I32 = "f32", "f16", "bf16", "i32"
STORAGE = {DT_F32: np.float32, DT_F16: np.uint16, DT_BF16: np.uint16, DT_I32: np.int32}


def values(dist, dtype, seed, n, start=0):
    """n generated values in storage form (raw encodings for 16-bit types)."""
    kind, lo, hi = dist
    if kind == "uniform":
        if dtype == DT_I32:
            return fill(UNIF_I32, seed, n, start, lo_i=lo, hi_i=hi)
        v = fill(UNIF_F32, seed, n, start, lo=lo, hi=hi)
    elif kind == "normal":
        if (lo, hi) != (0, 1):
            raise ValueError("only the standard normal N(0, 1) is generated")
        v = fill(NORM_F32, seed, n, start)
    else:
        raise ValueError(kind)
    if dtype == DT_F32:
        return v
    if dtype == DT_BF16:
        return f32_to_bf16_bits(v)
    if dtype == DT_F16:
        return f32_to_f16_bits(v)
    raise ValueError(dtype)


def values_at(dist, dtype, seed, counters):
    counters = np.asarray(counters, dtype=np.int64).ravel()
    return np.concatenate([values(dist, dtype, seed, 1, int(k)) for k in counters]) \
        if counters.size else np.empty(0, dtype=STORAGE[dtype])


def rank_slice(dist, dtype, rank, rows, ld, valid_rows, valid_cols, pad_bits=None,
               base_seed=BASE_SEED):
    """One rank's [rows, ld] slice (numpy, storage form)."""
    st = STORAGE[dtype]
    out = np.empty((rows, ld), dtype=st)
    if pad_bits is not None and (valid_rows < rows or valid_cols < ld):
        out.view(np.uint16 if out.itemsize == 2 else np.uint32)[...] = pad_bits
    elif valid_rows < rows or valid_cols < ld:
        out[...] = 0
    v = values(dist, dtype, base_seed + rank, valid_rows * valid_cols)
    out[:valid_rows, :valid_cols] = v.reshape(valid_rows, valid_cols)
    return out


class TreduceWorkload:
    """A TREDUCE case: N rank slices of [rows, ld], valid box, op list."""

    def __init__(self, name, nranks, dtype, rows, cols, ld, valid_rows, valid_cols,
                 dist, ops, root=0, src_pad=None, dst_pad=None):
        self.name, self.nranks, self.dtype = name, nranks, dtype
        self.rows, self.cols, self.ld = rows, cols, ld
        self.valid_rows, self.valid_cols = valid_rows, valid_cols
        self.dist, self.ops, self.root = dist, ops, root
        self.src_pad, self.dst_pad = src_pad, dst_pad

    @property
    def elem_bytes(self):
        return np.dtype(STORAGE[self.dtype]).itemsize

    def algorithmic_bytes(self):
        """(N + 1) * bytes per element * valid elements: N reads and 1 write."""
        return (self.nranks + 1) * self.elem_bytes * self.valid_rows * self.valid_cols

    def slice(self, r):
        return rank_slice(self.dist, self.dtype, r, self.rows, self.ld,
                          self.valid_rows, self.valid_cols, self.src_pad)

    def sample(self, r, ii, jj):
        """Values of rank r at valid-box positions (ii, jj), storage form."""
        k = np.asarray(ii, dtype=np.int64) * self.valid_cols + np.asarray(jj, dtype=np.int64)
        return values_at(self.dist, self.dtype, BASE_SEED + r, k)


# The benchmark workloads: shapes, distributions and sentinels.
def treduce_f32_n4_256():
    return TreduceWorkload("treduce_sum_n4_f32_256x256", 4, DT_F32, 256, 256, 256, 256, 256,
                           ("uniform", -1.0, 1.0), ["sum"])


def treduce_bf16_n8_4096_valid4000():
    return TreduceWorkload("treduce_n8_bf16_4096x4096_valid4000", 8, DT_BF16, 4096, 4096, 4096,
                           4000, 4000, ("normal", 0, 1), ["sum", "max", "min"],
                           src_pad=0x7FD5, dst_pad=0xFFD5)


def treduce_f32_n8_16384x8192():
    return TreduceWorkload("treduce_sum_n8_f32_16384x8192", 8, DT_F32, 16384, 8192, 8192,
                           16384, 8192, ("uniform", -1e3, 1e3), ["sum"])


def treduce_i32_n8_16384x8192():
    return TreduceWorkload("treduce_max_n8_i32_16384x8192", 8, DT_I32, 16384, 8192, 8192,
                           16384, 8192, ("uniform", -2**30, 2**30), ["max"])


WINDOWS_F16_N8_8192X4096 = dict(nranks=8, rows=8192, cols=4096, ld=4096, dtype=DT_F16, dist=("normal", 0, 1))


def window(r, cfg=WINDOWS_F16_N8_8192X4096):
    return rank_slice(cfg["dist"], cfg["dtype"], r, cfg["rows"], cfg["ld"], cfg["rows"], cfg["cols"])


# all_to_all_v: N=16 ranks, bf16 rows of 7168, target_rows 24576 (MAX_RECV 1536).
DISPATCH_BF16_N16_7168 = dict(nranks=16, size=7168, target_rows=24576, count_hi=2047, sentinel=0xFFFF)
COUNT_STREAM_START = 1 << 40   # counts use the sender's stream, far from its row data


def a2av_send_counts(s, nranks, hi=DISPATCH_BF16_N16_7168["count_hi"], lo=0):
    """send_counts of sender s: nranks ints uniform in [lo, hi]."""
    return fill(UNIF_I32, BASE_SEED + s, nranks, start=COUNT_STREAM_START, lo_i=lo, hi_i=hi)


def a2av_tag(s, d, i):
    """The three tag elements of input row (d*MAX_RECV + i) of sender s."""
    return np.array([s & 0xFFFF, d & 0xFFFF, i & 0xFFFF], dtype=np.uint16)


def a2av_input(s, nranks, target_rows, size):
    """Sender s's input [target_rows, size] (uint16 encodings): element (row, c)
    is bit-pattern counter row*size + c of stream BASE_SEED + s, except the first
    three elements of each row, which carry the (s, d, i) tag of that row."""
    x = fill(BITS16, BASE_SEED + s, target_rows * size).reshape(target_rows, size)
    mr = target_rows // nranks
    if size >= 3 and mr > 0:
        rows = np.arange(nranks * mr)
        x[: nranks * mr, 0] = s
        x[: nranks * mr, 1] = rows // mr
        x[: nranks * mr, 2] = rows % mr
    return x


def a2av_input_row(s, row, nranks, target_rows, size):
    """One row of a2av_input(s, ...) computed on its own (for sampled checks)."""
    x = fill(BITS16, BASE_SEED + s, size, start=row * size)
    mr = target_rows // nranks
    if size >= 3 and mr > 0 and row < nranks * mr:
        x[0], x[1], x[2] = s, row // mr, row % mr
    return x
