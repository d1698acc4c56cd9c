"""GB300 tile-level collective library: Python binding of libptoc.so.

This module only marshals arguments into the C ABI declared in
``include/ptoc.h``; every step of every operation runs in the library's CUDA
kernels. PyTorch is used for device memory and streams (``data_ptr()`` and
``cuda_stream``), never for the computation.

Entry points carry the C names:

    ptoc_treduce(tensors, dst, rows, cols, valid_rows, valid_cols, ld, op, dtype,
                 stream=None, root=0)
    ptoc_reduce_scatter(windows, rows, cols, ld, op, dtype, stream=None)
    ptoc_allgather(windows, rows, cols, ld, dtype, stream=None)
    ptoc_all_to_all_v(inputs, targets, send_counts, recv_counts, target_rows,
                      size, dtype, stream=None)
    ptoc_all_to_all_v_noalloc(inputs, targets, send_counts, recv_counts,
                              target_rows, size, dtype, stream=None)
    ptoc_allreduce(windows, rows, cols, ld, op, dtype, stream=None)
    ptoc_broadcast(windows, rows, cols, ld, dtype, stream=None, root=0)
    ptoc_all_to_all(inputs, targets, target_rows, size, dtype, stream=None)
    ptoc_all_to_all_v_combine(windows, outputs, recv_counts, target_rows, size,
                              atomic, dtype, stream=None)
    ptoc_credit_barrier(signals, local_ranks, generations, timeout_ns, status,
                        stream=None)
    ptoc_credit_barrier_host(signals, rank, generations, timeout_ns, status)
    ptoc_signal_reset(signals, stream=None)
    ptoc_wait_faults()   (returns the count)

Buffers are torch tensors or raw device addresses (ints). ``stream=None``
means torch's current stream. A non-OK status raises :class:`PtocError`
(nothing was launched); pass ``check=False`` to get the status instead.
``treduce``, ``reduce_scatter``, ``allgather``, ``allreduce``, ``broadcast``,
``all_to_all_v`` (``noalloc=True`` selects the no-allocation call),
``all_to_all`` and ``all_to_all_v_combine`` are shape-inferring conveniences
over the same calls; they refuse (ValueError) tensors whose layouts the C calls
cannot describe.

The package refuses to import when libptoc.so has not been built: there is no
fallback path.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libptoc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libptoc.so is not built (expected at %s); build it with "
        "`python tile_level_collective_gb300/_build.py` or __graft_entry__.build()" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

# ---- ABI constants (mirror include/ptoc.h) ---------------------------------
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIAS, ERR_CUDA = 0, 1, 2, 3, 4
SUM, MAX, MIN, PROD = 0, 1, 2, 3
F32, F16, BF16, I32 = 0, 1, 2, 3
ATOMIC_NONE, ATOMIC_ADD = 0, 1
MAX_RANKS = 64

OPS = {"sum": SUM, "max": MAX, "min": MIN, "prod": PROD}


class ptoc_group(ctypes.Structure):
    _fields_ = [("tensors", ctypes.POINTER(ctypes.c_void_p)),
                ("nranks", ctypes.c_int32),
                ("root", ctypes.c_int32)]


_vp, _i64 = ctypes.c_void_p, ctypes.c_int64
_G = ctypes.POINTER(ptoc_group)
_lib.ptoc_treduce.argtypes = [_G, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]
_lib.ptoc_reduce_scatter.argtypes = [_G, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]
_lib.ptoc_allgather.argtypes = [_G, _i64, _i64, _i64, ctypes.c_int, _vp]
_lib.ptoc_all_to_all_v.argtypes = [_G, _G, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i64, _i64,
                                   ctypes.c_int, _vp]
_lib.ptoc_all_to_all_v_noalloc.argtypes = _lib.ptoc_all_to_all_v.argtypes
_lib.ptoc_allreduce.argtypes = [_G, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]
_lib.ptoc_broadcast.argtypes = [_G, _i64, _i64, _i64, ctypes.c_int, _vp]
_lib.ptoc_all_to_all.argtypes = [_G, _G, _i64, _i64, ctypes.c_int, _vp]
_lib.ptoc_all_to_all_v_combine.argtypes = [_G, _G, ctypes.POINTER(_vp), _i64, _i64, ctypes.c_int,
                                           ctypes.c_int, _vp]
_lib.ptoc_credit_barrier.argtypes = [_G, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32,
                                     _i64, _vp, _vp]
_lib.ptoc_credit_barrier_host.argtypes = [_G, ctypes.c_int32, ctypes.c_int32, _i64, _vp]
_lib.ptoc_signal_reset.argtypes = [_G, _vp]
for _f in ("ptoc_treduce", "ptoc_reduce_scatter", "ptoc_allgather", "ptoc_all_to_all_v", "ptoc_all_to_all_v_noalloc",
           "ptoc_allreduce", "ptoc_broadcast", "ptoc_all_to_all", "ptoc_all_to_all_v_combine",
           "ptoc_credit_barrier", "ptoc_credit_barrier_host", "ptoc_signal_reset"):
    getattr(_lib, _f).restype = ctypes.c_int
_lib.ptoc_wait_faults.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
_lib.ptoc_wait_faults.restype = ctypes.c_int
_lib.ptoc_status_string.argtypes = [ctypes.c_int]
_lib.ptoc_status_string.restype = ctypes.c_char_p


class PtocError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s failed: %s" % (where, ptoc_status_string(status)))


def ptoc_status_string(status):
    return _lib.ptoc_status_string(int(status)).decode()


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()          # a torch tensor
    return x.ctypes.data             # a numpy array (host memory: the host credit barrier)


def _stream(stream):
    if stream is None:
        import torch
        if torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr_array(items):
    return (ctypes.c_void_p * max(len(items), 1))(*[_addr(t) for t in items])


def _group(tensors, root=0):
    arr = _ptr_array(tensors)
    g = ptoc_group(ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), len(tensors), root)
    return g, arr


def _done(status, where, check):
    if check and status != OK:
        raise PtocError(status, where)
    return status


def ptoc_treduce(tensors, dst, rows, cols, valid_rows, valid_cols, ld, op, dtype,
                 stream=None, root=0, check=True):
    g, keep = _group(tensors, root)
    st = _lib.ptoc_treduce(ctypes.byref(g), _addr(dst), rows, cols, valid_rows, valid_cols, ld,
                           int(op), int(dtype), _stream(stream))
    return _done(st, "ptoc_treduce", check)


def ptoc_reduce_scatter(windows, rows, cols, ld, op, dtype, stream=None, check=True):
    g, keep = _group(windows)
    st = _lib.ptoc_reduce_scatter(ctypes.byref(g), rows, cols, ld, int(op), int(dtype), _stream(stream))
    return _done(st, "ptoc_reduce_scatter", check)


def ptoc_allgather(windows, rows, cols, ld, dtype, stream=None, check=True):
    g, keep = _group(windows)
    st = _lib.ptoc_allgather(ctypes.byref(g), rows, cols, ld, int(dtype), _stream(stream))
    return _done(st, "ptoc_allgather", check)


def ptoc_all_to_all_v(inputs, targets, send_counts, recv_counts, target_rows, size, dtype,
                      stream=None, check=True):
    gi, k1 = _group(inputs)
    gt, k2 = _group(targets)
    sc = _ptr_array(send_counts)
    rc = _ptr_array(recv_counts)
    st = _lib.ptoc_all_to_all_v(ctypes.byref(gi), ctypes.byref(gt), sc, rc, target_rows, size,
                                int(dtype), _stream(stream))
    return _done(st, "ptoc_all_to_all_v", check)


def ptoc_all_to_all_v_noalloc(inputs, targets, send_counts, recv_counts, target_rows, size, dtype,
                              stream=None, check=True):
    gi, k1 = _group(inputs)
    gt, k2 = _group(targets)
    sc = _ptr_array(send_counts)
    rc = _ptr_array(recv_counts)
    st = _lib.ptoc_all_to_all_v_noalloc(ctypes.byref(gi), ctypes.byref(gt), sc, rc, target_rows, size,
                                        int(dtype), _stream(stream))
    return _done(st, "ptoc_all_to_all_v_noalloc", check)


def ptoc_allreduce(windows, rows, cols, ld, op, dtype, stream=None, check=True):
    g, keep = _group(windows)
    st = _lib.ptoc_allreduce(ctypes.byref(g), rows, cols, ld, int(op), int(dtype), _stream(stream))
    return _done(st, "ptoc_allreduce", check)


def ptoc_broadcast(windows, rows, cols, ld, dtype, stream=None, root=0, check=True):
    g, keep = _group(windows, root)
    st = _lib.ptoc_broadcast(ctypes.byref(g), rows, cols, ld, int(dtype), _stream(stream))
    return _done(st, "ptoc_broadcast", check)


def ptoc_all_to_all(inputs, targets, target_rows, size, dtype, stream=None, check=True):
    gi, k1 = _group(inputs)
    gt, k2 = _group(targets)
    st = _lib.ptoc_all_to_all(ctypes.byref(gi), ctypes.byref(gt), target_rows, size, int(dtype),
                              _stream(stream))
    return _done(st, "ptoc_all_to_all", check)


def ptoc_all_to_all_v_combine(windows, outputs, recv_counts, target_rows, size, atomic, dtype,
                              stream=None, check=True):
    gw, k1 = _group(windows)
    go, k2 = _group(outputs)
    rc = _ptr_array(recv_counts)
    st = _lib.ptoc_all_to_all_v_combine(ctypes.byref(gw), ctypes.byref(go), rc, target_rows, size,
                                        int(atomic), int(dtype), _stream(stream))
    return _done(st, "ptoc_all_to_all_v_combine", check)


def ptoc_credit_barrier(signals, local_ranks, generations, timeout_ns, status, stream=None, check=True):
    g, keep = _group(signals)
    ranks = (ctypes.c_int32 * max(len(local_ranks), 1))(*[int(r) for r in local_ranks])
    st = _lib.ptoc_credit_barrier(ctypes.byref(g), ranks, len(local_ranks), int(generations),
                                  int(timeout_ns), _addr(status), _stream(stream))
    return _done(st, "ptoc_credit_barrier", check)


def ptoc_credit_barrier_host(signals, rank, generations, timeout_ns, status, check=True):
    """Rank `rank`'s part of one host credit-barrier call, on the calling
    thread. `signals` and `status` are HOST memory: addresses (ints), CPU
    tensors or numpy arrays.
    ctypes releases the GIL for the call, so ranks on Python threads run
    concurrently."""
    g, keep = _group(signals)
    st = _lib.ptoc_credit_barrier_host(ctypes.byref(g), int(rank), int(generations), int(timeout_ns),
                                       _addr(status))
    return _done(st, "ptoc_credit_barrier_host", check)


def ptoc_signal_reset(signals, stream=None, check=True):
    g, keep = _group(signals)
    st = _lib.ptoc_signal_reset(ctypes.byref(g), _stream(stream))
    return _done(st, "ptoc_signal_reset", check)


def ptoc_wait_faults(check=True):
    """The count of staged-reduction waits that gave up on the current device
    since the previous call (the count then restarts at zero)."""
    n = ctypes.c_uint32(0)
    st = _lib.ptoc_wait_faults(ctypes.byref(n))
    _done(st, "ptoc_wait_faults", check)
    return int(n.value) if st == OK else st


# ---- shape-inferring conveniences over torch tensors ------------------------

def dtype_code(t):
    import torch
    m = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16, torch.int32: I32}
    if t.dtype not in m:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return m[t.dtype]


def _rows_cols_ld(t):
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.stride(1) != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    return t.shape[0], t.shape[1], t.stride(0)


def _same_layout(tensors, what, contiguous=False):
    """Every tensor 2-D with the first one's shape, row pitch, dtype and device
    (and packed rows when `contiguous`): the C calls take one description."""
    t0 = tensors[0]
    rows, cols, ld = _rows_cols_ld(t0)
    if contiguous and ld != cols:
        raise ValueError("%s: rows must be packed (stride(0) == shape[1])" % what)
    for t in tensors[1:]:
        if t.dim() != 2 or tuple(t.shape) != tuple(t0.shape) or t.stride() != t0.stride() \
                or t.dtype != t0.dtype or t.device != t0.device:
            raise ValueError("%s: every tensor needs the same shape, strides, dtype and device" % what)
    return rows, cols, ld


def treduce(tensors, dst, op="sum", valid_rows=None, valid_cols=None, root=0, stream=None):
    """dst = reduction of 2-D tensors over their valid box (default: all)."""
    _same_layout(list(tensors) + [dst], "treduce")
    rows, cols, ld = _rows_cols_ld(dst)
    vr = rows if valid_rows is None else valid_rows
    vc = cols if valid_cols is None else valid_cols
    return ptoc_treduce(tensors, dst, rows, cols, vr, vc, ld, OPS[op] if isinstance(op, str) else op,
                        dtype_code(dst), stream=stream, root=root)


def reduce_scatter(windows, op="sum", stream=None):
    rows, cols, ld = _same_layout(windows, "reduce_scatter")
    return ptoc_reduce_scatter(windows, rows, cols, ld, OPS[op] if isinstance(op, str) else op,
                               dtype_code(windows[0]), stream=stream)


def allgather(windows, stream=None):
    rows, cols, ld = _same_layout(windows, "allgather")
    return ptoc_allgather(windows, rows, cols, ld, dtype_code(windows[0]), stream=stream)


def all_to_all_v(inputs, targets, send_counts, recv_counts, stream=None, noalloc=False):
    """noalloc=True: ptoc_all_to_all_v_noalloc (no allocation; one call in
    flight at a time)."""
    tr, size, _ = _same_layout(list(inputs) + list(targets), "all_to_all_v", contiguous=True)
    f = ptoc_all_to_all_v_noalloc if noalloc else ptoc_all_to_all_v
    return f(inputs, targets, send_counts, recv_counts, tr, size, dtype_code(targets[0]), stream=stream)


def allreduce(windows, op="sum", stream=None):
    rows, cols, ld = _same_layout(windows, "allreduce")
    return ptoc_allreduce(windows, rows, cols, ld, OPS[op] if isinstance(op, str) else op,
                          dtype_code(windows[0]), stream=stream)


def broadcast(windows, root=0, stream=None):
    rows, cols, ld = _same_layout(windows, "broadcast")
    return ptoc_broadcast(windows, rows, cols, ld, dtype_code(windows[0]), stream=stream, root=root)


def all_to_all(inputs, targets, stream=None):
    tr, size, _ = _same_layout(list(inputs) + list(targets), "all_to_all", contiguous=True)
    return ptoc_all_to_all(inputs, targets, tr, size, dtype_code(targets[0]), stream=stream)


def all_to_all_v_combine(windows, outputs, recv_counts, atomic="none", stream=None):
    tr, size, _ = _same_layout(list(windows) + list(outputs), "all_to_all_v_combine", contiguous=True)
    a = {"none": ATOMIC_NONE, "add": ATOMIC_ADD}[atomic] if isinstance(atomic, str) else atomic
    return ptoc_all_to_all_v_combine(windows, outputs, recv_counts, tr, size, a,
                                     dtype_code(outputs[0]), stream=stream)
