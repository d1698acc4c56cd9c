"""Oracle for the TREDUCE / window-collective hot path (ctypes wrapper).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The
product path (``tile_level_collective_gb300``) never imports it and shares no
code with it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, compiled with
``-ffp-contract=off`` and no fast-math). This module only builds that file with
gcc, loads it and passes numpy buffers to it. Element types are given as the
oracle's own codes below; 16-bit floating types travel as ``uint16`` arrays
holding the raw encodings.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# ReduceOp values (TREDUCE article, section 1.3; Prod appended by the
# Distributed Operators page's ABI enums).
SUM, MAX, MIN, PROD = 0, 1, 2, 3
# AtomicType values (Distributed Operators page, ABI enums).
ATOMIC_NONE, ATOMIC_ADD = 0, 1
# The oracle's element-type codes.
F32, F16, BF16, I32 = 0, 1, 2, 3
ELEM_BYTES = {F32: 4, F16: 2, BF16: 2, I32: 4}
NUMPY_TYPE = {F32: np.float32, F16: np.uint16, BF16: np.uint16, I32: np.int32}

_lib = None


def compile_source(src, out):
    """gcc with the oracle's flags: src (C file) -> out (shared library)."""
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(os.path.abspath(out)))
    os.close(fd)
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    try:
        subprocess.check_call(cmd)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def build(force=False):
    """Compile oracle.c into liboracle.so beside it (gcc, plain flags)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    return compile_source(_SRC, _LIB)


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB)
    return _lib


def load(path):
    """Load an oracle build and declare its functions (the tests also load
    deliberately broken copies, to show that the pins catch them)."""
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.oracle_treduce.argtypes = [ctypes.POINTER(vp), i32, i32, vp, i64, i64, i64, i32, i32]
    L.oracle_treduce_sum_native_acc.argtypes = [ctypes.POINTER(vp), i32, i32, vp, i64, i64, i64, i32]
    L.oracle_treduce_sum_native_acc.restype = ctypes.c_int
    L.oracle_reduce_scatter.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i64, i32, i32]
    L.oracle_allgather.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i64, i32]
    L.oracle_all_to_all_v.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp),
                                      ctypes.POINTER(vp), ctypes.POINTER(vp),
                                      i32, i64, i64, i32]
    L.oracle_allreduce.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i64, i32, i32]
    L.oracle_broadcast.argtypes = [ctypes.POINTER(vp), i32, i32, i64, i64, i64, i32]
    L.oracle_all_to_all.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, i64, i64, i32]
    L.oracle_all_to_all_v_combine.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp),
                                              ctypes.POINTER(vp), i32, i64, i64, i32, i32]
    L.oracle_credit_barrier.argtypes = [i32, i32, vp, vp, vp, i32]
    for name in ("oracle_treduce", "oracle_reduce_scatter", "oracle_allgather",
                 "oracle_all_to_all_v", "oracle_allreduce", "oracle_broadcast",
                 "oracle_all_to_all", "oracle_all_to_all_v_combine", "oracle_credit_barrier"):
        getattr(L, name).restype = ctypes.c_int
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_f16.restype = ctypes.c_uint16
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_f32.restype = ctypes.c_float
    for name in ("oracle_f32_to_bf16_array", "oracle_f32_to_f16_array",
                 "oracle_f16_to_f32_array", "oracle_bf16_to_f32_array"):
        getattr(L, name).argtypes = [vp, vp, i64]
        getattr(L, name).restype = None
    return L


def _ptrs(arrays):
    for a in arrays:
        if not a.flags.c_contiguous:
            raise ValueError("oracle buffers must be C-contiguous")
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def treduce(srcs, dst, valid_rows, valid_cols, ld, op, dtype, root=0):
    """dst[i*ld+j] = reduction over srcs in the page's rank order; see oracle.c."""
    return lib().oracle_treduce(_ptrs(srcs), len(srcs), root, dst.ctypes.data,
                                valid_rows, valid_cols, ld, op, dtype)


def treduce_sum_native_acc(srcs, dst, valid_rows, valid_cols, ld, dtype, root=0):
    """TREDUCE Sum with every partial sum rounded to the destination type (the
    accumulator tile in the destination type); see oracle.c."""
    return lib().oracle_treduce_sum_native_acc(_ptrs(srcs), len(srcs), root, dst.ctypes.data,
                                               valid_rows, valid_cols, ld, dtype)


def reduce_scatter(windows, rows, cols, ld, op, dtype):
    return lib().oracle_reduce_scatter(_ptrs(windows), len(windows), rows, cols, ld, op, dtype)


def allgather(windows, rows, cols, ld, dtype):
    return lib().oracle_allgather(_ptrs(windows), len(windows), rows, cols, ld, dtype)


def all_to_all_v(inputs, targets, send_counts, recv_counts, target_rows, size, elem_size):
    n = len(inputs)
    assert len(targets) == n and len(send_counts) == n and len(recv_counts) == n
    for c in list(send_counts) + list(recv_counts):
        assert c.dtype == np.int32
    return lib().oracle_all_to_all_v(_ptrs(inputs), _ptrs(targets), _ptrs(send_counts),
                                     _ptrs(recv_counts), n, target_rows, size, elem_size)


def allreduce(windows, rows, cols, ld, op, dtype):
    return lib().oracle_allreduce(_ptrs(windows), len(windows), rows, cols, ld, op, dtype)


def broadcast(windows, root, rows, cols, ld, dtype):
    return lib().oracle_broadcast(_ptrs(windows), len(windows), root, rows, cols, ld, dtype)


def all_to_all(inputs, targets, target_rows, size, elem_size):
    assert len(targets) == len(inputs)
    return lib().oracle_all_to_all(_ptrs(inputs), _ptrs(targets), len(inputs), target_rows, size,
                                   elem_size)


def all_to_all_v_combine(windows, outputs, recv_counts, target_rows, size, atomic, dtype):
    n = len(windows)
    assert len(outputs) == n and len(recv_counts) == n
    return lib().oracle_all_to_all_v_combine(_ptrs(windows), _ptrs(outputs), _ptrs(recv_counts), n,
                                             target_rows, size, atomic, dtype)


def credit_barrier(nranks, generations, present, signal, wait_eq=False):
    """Runs the credit barrier on `signal` (int32 [N, N], row r = rank r's
    window) in place; returns the per-rank status array."""
    present = np.ascontiguousarray(present, dtype=np.int32)
    assert signal.dtype == np.int32 and signal.shape == (nranks, nranks) and signal.flags.c_contiguous
    status = np.zeros(nranks, dtype=np.int32)
    rc = lib().oracle_credit_barrier(nranks, generations, present.ctypes.data, signal.ctypes.data,
                                     status.ctypes.data, 1 if wait_eq else 0)
    assert rc == 0
    return status


def f32_to_bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f32_to_f16(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f16_to_f32(h):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, dtype=np.float32)
    lib().oracle_f16_to_f32_array(h.ctypes.data, y.ctypes.data, h.size)
    return y


def bf16_to_f32(h):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, dtype=np.float32)
    lib().oracle_bf16_to_f32_array(h.ctypes.data, y.ctypes.data, h.size)
    return y
