"""Benchmark of the TREDUCE / window-collective hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Default workload: TREDUCE over 8 ranks of [16384, 8192] 4-byte elements, the
largest TREDUCE case: f32 Sum over U[-1e3, 1e3] inputs and the int32 Max
variant over U[-2^30, 2^30] inputs, each over its own sources (8 x 512 MiB);
one step = the two launches. Metric: effective HBM GB/s = (N + 1) *
bytes/elem * valid elements per launch, summed over the step, divided by the
step's device time. Inputs are generated on the host by the seeded generator
and resident in HBM before timing; before every step L2 is flushed outside the
timed events (a 256 MiB buffer is written, then read back, which leaves L2
cold and clean: no dirty flush lines for the timed kernels to write back), and
each launch reads 4 GiB besides, far more than L2. The K-step block is timed
again, back to back, until the timed region spans half a second, so that the
clock record samples it; every timed step counts. Other workloads (the bf16
4096 x 4096 case with its 4000 x 4000 valid box as `--workload treduce`, and
the parity configurations) can be timed with --workload for the per-kernel
evidence. After the timed steps the CPU-baseline leg times the oracle on a
bounded sample of the workload and then, untimed, compares the resident run's
results with the oracle's (cpu_baseline.parity, bit for bit; every element
for the TREDUCE workloads).

--impl reference times the CPU oracle on the host's CPU cores (the only
other implementation there is), on a bounded sample of the same workload per
step. Multi-GPU (torchrun): every rank runs an independent replica (the path
has no cross-GPU exchange); value is the total over ranks / max time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TREDUCE effective HBM GB/s (N reads + 1 write) and % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


L2_NOTE = ("flushed before every step, outside the timed events: a 256 MiB buffer is written, then "
           "read back (cold, clean L2)")


class L2Flush:
    """Leaves L2 cold and clean: writes a buffer twice the size of L2, then
    reads the same buffer back. Measured on GB300: a write alone leaves dirty
    lines that the next kernel must write back, and a read of another buffer
    does not clear them either; reading the written buffer back does, and the
    kernels that follow then take their ncu cold-cache durations."""

    def __init__(self, dev):
        import torch
        self.a = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.words = self.a.view(torch.int32)
        self.sink = torch.empty((), dtype=torch.int32, device=dev)

    def __call__(self, k=0):
        import torch
        self.a.fill_(k & 0xFF)
        torch.amax(self.words, dim=0, out=self.sink)
# The device-code sources of each workload's dominant kernel: a recorded ncu
# traffic figure stays valid while these hash the same (a change of launch
# configuration in ptoc_api.cu calls for a new capture too).
_CSRC = "tile_level_collective_gb300/csrc/"
_COMMON = [_CSRC + "ptoc_internal.h", _CSRC + "reduce_impl.cuh"]
REDUCE_SOURCES = _COMMON + [_CSRC + f for f in ("reduce_forms.cuh", "reduce_f32.cu", "reduce_f16.cu",
                                                "reduce_bf16.cu", "reduce_i32.cu")]
MOVE_SOURCES = _COMMON + [_CSRC + "movement.cu"]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class Workload:
    """One benchmark workload: host inputs, device buffers, the launches of a
    step and its algorithmic bytes."""
    # Launches of different kernels in one step are timed one by one (events
    # between them); launches of one kernel family are timed as a step (events
    # around it), so they run back to back as a caller's calls do.
    per_launch_timing = False
    name = ""
    dtype_compute = "f32"
    storage = ""
    kernel = ""
    pipelined_e2e = False
    e2e_inplace = False
    sources = REDUCE_SOURCES      # of the dominant kernel

    def config(self):
        raise NotImplementedError

    def prepare(self):
        """Called before every step, outside the timed events (restores the
        inputs of in-place workloads)."""


# The library's choice between its two reduction forms (mirrors the rule in
# ptoc_api.cu, for the kernel label of the bench line only): launches of 2 to
# 8 ranks on 16-byte-aligned data that move at least 1.5 GiB take the staged
# form unless PTOC_REDUCE_STAGING forces one.
STAGED_MIN_BYTES = 3 << 29


def reduce_form(nbytes, nranks):
    forced = os.environ.get("PTOC_REDUCE_STAGING")
    if not 2 <= nranks <= 8:
        return "regs"
    if forced in ("bulk", "regs"):
        return forced
    return "bulk" if nbytes >= STAGED_MIN_BYTES else "regs"


def reduce_kernel_label(nbytes, nranks, what):
    if reduce_form(nbytes, nranks) == "bulk":
        return "reduce_staged_kernel<%s> (sources staged in shared memory by bulk copies, one block per tile)" % what
    return "reduce_kernel<%s> (sources loaded into registers, one block per tile)" % what


class TreduceBench(Workload):
    def __init__(self, w, storage):
        self.w, self.storage = w, storage
        self.name = w.name
        self.kernel = reduce_kernel_label(w.algorithmic_bytes(), w.nranks, "%s, %s" % (storage, "/".join(w.ops)))
        self.dtype_compute = "i32" if storage == "i32" else "f32"

    def bytes_per_launch(self):
        return self.w.algorithmic_bytes()

    def launches_per_step(self):
        return len(self.w.ops)

    def bytes_per_step(self):
        return self.bytes_per_launch() * self.launches_per_step()

    def setup_host(self):
        import numpy as np
        self.host = [np.ascontiguousarray(self.w.slice(r)) for r in range(self.w.nranks)]

    def setup_device(self, dev):
        import numpy as np
        import torch
        w = self.w
        self.dev = [_to_dev(h, dev) for h in self.host]
        pad = w.dst_pad if w.dst_pad is not None else 0
        self.dst_init = np.empty((w.rows, w.ld), dtype=self.host[0].dtype)
        self.dst_init.view(np.uint16 if self.dst_init.itemsize == 2 else np.uint32)[...] = pad
        self.dsts = [_to_dev(self.dst_init, dev) for _ in w.ops]

    def launch(self, i, srcs=None, dst=None):
        import tile_level_collective_gb300 as P
        w = self.w
        code = {"f32": P.F32, "f16": P.F16, "bf16": P.BF16, "i32": P.I32}[self.storage]
        P.ptoc_treduce(srcs or self.dev, dst if dst is not None else self.dsts[i], w.rows, w.cols,
                       w.valid_rows, w.valid_cols, w.ld, P.OPS[w.ops[i]], code)

    # e2e: every step uploads its inputs from pinned host memory and reads its
    # results back; double-buffered on three streams, so step k's upload
    # overlaps step k-1's compute and download (a caller streaming batches).
    pipelined_e2e = True

    def setup_e2e(self, dev):
        import torch
        self.pinned = [_pin(h) for h in self.host]
        self.e2e_in = [[torch.empty_like(t) for t in self.dev] for _ in range(2)]
        # fresh destinations (the pad pattern), so the check below sees only
        # what the pipelined calls wrote
        self.e2e_out = [[_to_dev(self.dst_init, dev) for _ in self.w.ops] for _ in range(2)]
        self.out_pinned = [[torch.empty(_nbytes(self.dst_init), dtype=torch.uint8).pin_memory()
                            for _ in self.w.ops] for _ in range(2)]

    def e2e_upload(self, b):
        for d, h in zip(self.e2e_in[b], self.pinned):
            d.view(-1).view(torch_uint8()).copy_(h, non_blocking=True)

    def e2e_compute(self, b):
        for i in range(self.launches_per_step()):
            self.launch(i, srcs=self.e2e_in[b], dst=self.e2e_out[b][i])

    def e2e_download(self, b):
        for o, d in zip(self.out_pinned[b], self.e2e_out[b]):
            o.copy_(d.view(-1).view(torch_uint8()), non_blocking=True)

    def e2e_verify(self, b):
        """The downloaded results equal the resident run's bytes (same inputs)."""
        for o, d in zip(self.out_pinned[b], self.dsts):
            if not bool((o == d.view(-1).view(torch_uint8()).cpu()).all()):
                raise RuntimeError("pipelined end-to-end result differs from the resident result")

    def h2d_bytes(self):
        return sum(_nbytes(h) for h in self.host)

    def d2h_bytes(self):
        return _nbytes(self.dst_init) * len(self.w.ops)

    def config(self):
        w = self.w
        return {"workload": w.name, "op": "TREDUCE", "nranks": w.nranks, "storage_dtype": self.storage,
                "shape": [w.rows, w.cols], "ld": w.ld, "valid": [w.valid_rows, w.valid_cols],
                "ops": w.ops, "root": w.root, "values": ("normal(0,1)" if w.dist[0] == "normal" else "%s[%s, %s]" % w.dist),
                "seed": "1234 + rank (SplitMix64, counter-based)",
                "step": "%d TREDUCE launches (%s)" % (len(w.ops), ", ".join(w.ops)),
                "bytes_per_step": self.bytes_per_step(),
                "l2": L2_NOTE}

    # oracle on a bounded sample: the first `rows` rows of the valid box
    def oracle_sample(self, rows):
        import oracle
        w = self.w
        rows = max(1, min(rows, w.valid_rows))
        import numpy as np
        out = np.empty((rows, w.ld), dtype=self.host[0].dtype)
        code = {"f32": oracle.F32, "bf16": oracle.BF16, "f16": oracle.F16, "i32": oracle.I32}[self.storage]
        ops = {"sum": oracle.SUM, "max": oracle.MAX, "min": oracle.MIN}
        t0 = time.perf_counter()
        for op in w.ops:
            oracle.treduce(self.host, out, rows, w.valid_cols, w.ld, ops[op], code)
        dt = time.perf_counter() - t0
        nbytes = (w.nranks + 1) * w.elem_bytes * rows * w.valid_cols * len(w.ops)
        return nbytes, dt, "rows 0..%d of the %dx%d valid box, ops %s" % (
            rows - 1, w.valid_rows, w.valid_cols, "+".join(w.ops))

    def oracle_rows_per_second(self):
        nb, dt, _ = self.oracle_sample(8)
        return 8.0 / max(dt, 1e-9)

    def oracle_parity(self, rows):
        """The resident run's results on the first `rows` rows against the
        oracle on the same host inputs, bit for bit: every valid element, and
        the padding of those rows still holding its sentinel."""
        import numpy as np
        import oracle
        w = self.w
        rows = max(1, min(rows, w.valid_rows))
        code = {"f32": oracle.F32, "bf16": oracle.BF16, "f16": oracle.F16, "i32": oracle.I32}[self.storage]
        ops = {"sum": oracle.SUM, "max": oracle.MAX, "min": oracle.MIN}
        bad = []
        for i, op in enumerate(w.ops):
            want = self.dst_init[:rows].copy()
            oracle.treduce([h[:rows] for h in self.host], want, rows, w.valid_cols, w.ld, ops[op], code)
            got = np.ascontiguousarray(self.dsts[i][:rows].cpu().numpy()).view(want.dtype)
            if not np.array_equal(got.view(np.uint8), want.view(np.uint8)):
                bad.append(op)
        return {"rows": "0..%d of %d" % (rows - 1, w.valid_rows), "ops": list(w.ops),
                "result": "bit-exact" if not bad else "MISMATCH in " + ", ".join(bad)}

    def max_rows(self):
        return self.w.valid_rows

    def oracle_parity_all(self, threads=None):
        """Every element of the resident run's results against the oracle on
        the same host inputs, bit for bit: the whole valid box of every op,
        and the padding around it still holding its sentinel. The oracle runs
        on contiguous row slices, one host thread each (a split run equals
        one call, byte for byte)."""
        import numpy as np
        w = self.w
        threads = threads or os.cpu_count() or 1
        bad = []
        for i, op in enumerate(w.ops):
            want = self.oracle_rows_threaded(0, w.valid_rows, op, threads)
            got = np.ascontiguousarray(self.dsts[i].cpu().numpy()).view(want.dtype)
            if not np.array_equal(got.view(np.uint8), want.view(np.uint8)):
                bad.append(op)
        return {"rows": "all %d of %d (every element, padding included)" % (w.valid_rows, w.rows),
                "ops": list(w.ops), "result": "bit-exact" if not bad else "MISMATCH in " + ", ".join(bad)}

    def oracle_rows_threaded(self, lo, hi, op, threads):
        """The oracle's full dst (padding as initialised) for valid rows
        [lo, hi) of one op, split into `threads` contiguous row slices on as
        many host threads; rows outside [lo, hi) keep the padding."""
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        w = self.w
        out = self.dst_init.copy()
        code = {"f32": oracle.F32, "bf16": oracle.BF16, "f16": oracle.F16, "i32": oracle.I32}[self.storage]
        code_op = {"sum": oracle.SUM, "max": oracle.MAX, "min": oracle.MIN}[op]
        n = hi - lo
        bounds = [lo + n * t // threads for t in range(threads + 1)]

        def part(t):
            a, b = bounds[t], bounds[t + 1]
            if b > a:
                oracle.treduce([h[a:b] for h in self.host], out[a:b], b - a, w.valid_cols, w.ld, code_op, code)

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(part, range(threads)))
        return out

    def oracle_sample_threaded(self, rows, threads):
        """The same oracle call on `rows` rows, the rows split into `threads`
        contiguous slices run on as many host threads (ctypes releases the
        interpreter lock during the call)."""
        import numpy as np
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        w = self.w
        rows = max(threads, min(rows, w.valid_rows))
        out = np.empty((rows, w.ld), dtype=self.host[0].dtype)
        code = {"f32": oracle.F32, "bf16": oracle.BF16, "f16": oracle.F16, "i32": oracle.I32}[self.storage]
        ops = {"sum": oracle.SUM, "max": oracle.MAX, "min": oracle.MIN}
        bounds = [rows * t // threads for t in range(threads + 1)]

        def part(t):
            lo, hi = bounds[t], bounds[t + 1]
            for op in w.ops:
                oracle.treduce([h[lo:hi] for h in self.host], out[lo:hi], hi - lo, w.valid_cols, w.ld,
                               ops[op], code)

        with ThreadPoolExecutor(threads) as ex:
            t0 = time.perf_counter()
            list(ex.map(part, range(threads)))
            dt = time.perf_counter() - t0
        nbytes = (w.nranks + 1) * w.elem_bytes * rows * w.valid_cols * len(w.ops)
        return nbytes, dt, out


class TreducePairBench(Workload):
    """The two TREDUCE launches of one 8-rank [16384, 8192] case: f32 Sum over
    U[-1e3, 1e3] inputs and the int32 Max variant over U[-2^30, 2^30] inputs
    (each with its own 8 x 512 MiB of sources and its own dst), one launch of
    each per step. Every figure is the sum over the two parts."""
    pipelined_e2e = True

    def __init__(self, parts):
        self.parts = parts
        w = parts[0].w
        assert all(p.w.algorithmic_bytes() == w.algorithmic_bytes() and len(p.w.ops) == 1 for p in parts)
        self.name = "treduce_n8_16384x8192_f32sum_i32max"
        self.kernel = " and ".join(p.kernel for p in parts)
        self.dtype_compute = "+".join(p.dtype_compute for p in parts)

    def bytes_per_launch(self):
        return self.parts[0].bytes_per_launch()

    def launches_per_step(self):
        return len(self.parts)

    def bytes_per_step(self):
        return sum(p.bytes_per_step() for p in self.parts)

    def max_rows(self):
        return self.parts[0].w.valid_rows

    def setup_host(self):
        for p in self.parts:
            p.setup_host()

    def setup_device(self, dev):
        for p in self.parts:
            p.setup_device(dev)

    def launch(self, i, srcs=None, dst=None):
        self.parts[i].launch(0, srcs, dst)

    def setup_e2e(self, dev):
        for p in self.parts:
            p.setup_e2e(dev)

    def e2e_upload(self, b):
        for p in self.parts:
            p.e2e_upload(b)

    def e2e_compute(self, b):
        for p in self.parts:
            p.e2e_compute(b)

    def e2e_download(self, b):
        for p in self.parts:
            p.e2e_download(b)

    def e2e_verify(self, b):
        for p in self.parts:
            p.e2e_verify(b)

    def h2d_bytes(self):
        return sum(p.h2d_bytes() for p in self.parts)

    def d2h_bytes(self):
        return sum(p.d2h_bytes() for p in self.parts)

    def config(self):
        w = self.parts[0].w
        return {"workload": self.name, "op": "TREDUCE", "nranks": w.nranks,
                "storage_dtype": "+".join(p.storage for p in self.parts),
                "shape": [w.rows, w.cols], "ld": w.ld, "valid": [w.valid_rows, w.valid_cols],
                "ops": ["%s %s" % (p.storage, p.w.ops[0]) for p in self.parts], "root": w.root,
                "values": "; ".join("%s %s[%s, %s]" % ((p.storage,) + tuple(p.w.dist)) for p in self.parts),
                "seed": "1234 + rank (SplitMix64, counter-based)",
                "step": "%d TREDUCE launches (%s), each over its own 8 sources" % (
                    len(self.parts), ", ".join("%s %s" % (p.storage, p.w.ops[0]) for p in self.parts)),
                "bytes_per_step": self.bytes_per_step(),
                "l2": L2_NOTE + "; each launch also reads 4 GiB, 33x L2"}

    def oracle_sample(self, rows):
        nb_tot, dt_tot, descs = 0, 0.0, []
        for p in self.parts:
            nb, dt, desc = p.oracle_sample(rows)
            nb_tot, dt_tot = nb_tot + nb, dt_tot + dt
            descs.append("%s: %s" % (p.storage, desc))
        return nb_tot, dt_tot, "; ".join(descs)

    def oracle_rows_per_second(self):
        return 1.0 / sum(1.0 / p.oracle_rows_per_second() for p in self.parts)

    def oracle_parity(self, rows):
        return self.oracle_parity_all()

    def oracle_parity_all(self, threads=None):
        res = [p.oracle_parity_all(threads) for p in self.parts]
        bad = [p.storage + " " + r["result"] for p, r in zip(self.parts, res) if r["result"] != "bit-exact"]
        return {"rows": res[0]["rows"], "ops": ["%s %s" % (p.storage, p.w.ops[0]) for p in self.parts],
                "result": "bit-exact" if not bad else "; ".join(bad)}

    def oracle_sample_threaded(self, rows, threads):
        nb_tot, dt_tot, outs = 0, 0.0, []
        for p in self.parts:
            nb, dt, out = p.oracle_sample_threaded(rows, threads)
            nb_tot, dt_tot = nb_tot + nb, dt_tot + dt
            outs.append(out)
        return nb_tot, dt_tot, outs


class RsAgBench(Workload):
    """reduce_scatter (Sum) then allgather over 8 fp16 windows [8192, 4096]."""

    def __init__(self):
        import synth
        self.cfg = synth.WINDOWS_F16_N8_8192X4096
        self.name = "reduce_scatter_allgather_n8_f16_8192x4096"
        self.per_launch_timing = True
        self.storage = "f16"
        self.kernel = "reduce_kernel<f16> (owner-window mode) + gather_kernel"

    def bytes_per_launch_list(self):
        c = self.cfg
        elems = c["rows"] * c["cols"]
        return [(c["nranks"] + 1) * 2 * elems, c["nranks"] * 2 * elems]

    def launches_per_step(self):
        return 2

    def bytes_per_step(self):
        return sum(self.bytes_per_launch_list())

    def bytes_per_launch(self):
        return self.bytes_per_launch_list()[0]

    def setup_host(self):
        import synth
        self.host = [synth.window(r, self.cfg) for r in range(self.cfg["nranks"])]

    def setup_device(self, dev):
        self.dev = [_to_dev(h, dev) for h in self.host]
        self.saved = [t.clone() for t in self.dev]

    def prepare(self):
        for t, s in zip(self.dev, self.saved):
            t.copy_(s)

    def launch(self, i, srcs=None, dst=None):
        import tile_level_collective_gb300 as P
        c = self.cfg
        wins = srcs or self.dev
        if i == 0:
            P.ptoc_reduce_scatter(wins, c["rows"], c["cols"], c["ld"], P.SUM, P.F16)
        else:
            P.ptoc_allgather(wins, c["rows"], c["cols"], c["ld"], P.F16)

    # e2e: windows uploaded, reduced and gathered in place, read back
    pipelined_e2e = True
    e2e_inplace = True

    def setup_e2e(self, dev):
        import torch
        self.pinned = [_pin(h) for h in self.host]
        self.e2e_win = [[torch.empty_like(t) for t in self.dev] for _ in range(2)]
        self.out_pinned = [_pinned_like(self.dev) for _ in range(2)]

    def e2e_upload(self, b):
        _upload(self.e2e_win[b], self.pinned)

    def e2e_compute(self, b):
        self.launch(0, srcs=self.e2e_win[b])
        self.launch(1, srcs=self.e2e_win[b])

    def e2e_download(self, b):
        _download(self.out_pinned[b], self.e2e_win[b])

    def e2e_verify(self, b):
        _check_same(self.out_pinned[b], self.dev, "window")

    def h2d_bytes(self):
        return sum(_nbytes(h) for h in self.host)

    def d2h_bytes(self):
        return sum(_nbytes(h) for h in self.host)

    def config(self):
        c = self.cfg
        return {"workload": self.name, "op": "reduce_scatter+allgather", "nranks": c["nranks"],
                "storage_dtype": "f16", "shape": [c["rows"], c["cols"]], "ld": c["ld"],
                "values": "normal(0,1)", "step": "reduce_scatter (Sum) then allgather",
                "bytes_per_step": self.bytes_per_step(),
                "l2": L2_NOTE}

    def oracle_sample(self, rows):
        import numpy as np
        import oracle
        c = self.cfg
        n = c["nranks"]
        rows = max(n, min(rows, c["rows"]))
        wins = [h[:rows].copy() for h in self.host]          # the oracle works in place
        t0 = time.perf_counter()
        oracle.reduce_scatter(wins, rows, c["cols"], c["ld"], oracle.SUM, oracle.F16)
        oracle.allgather(wins, rows, c["cols"], c["ld"], oracle.F16)
        dt = time.perf_counter() - t0
        nb = (2 * n + 1) * 2 * rows * c["cols"]
        return nb, dt, "reduce_scatter+allgather over rows 0..%d of the 8 windows" % (rows - 1)

    def oracle_parity(self, rows):
        """After reduce_scatter and allgather every window holds, in each row,
        the rank-ordered reduction of that row whatever the chunk bounds, so
        the oracle's pass over the first rows gives the full-size values
        there."""
        import numpy as np
        import oracle
        c = self.cfg
        rows = max(c["nranks"], min(rows, c["rows"]))
        wins = [h[:rows].copy() for h in self.host]          # the oracle works in place
        oracle.reduce_scatter(wins, rows, c["cols"], c["ld"], oracle.SUM, oracle.F16)
        oracle.allgather(wins, rows, c["cols"], c["ld"], oracle.F16)
        return _windows_parity(self.dev, wins, rows, c["rows"])

    def oracle_parity_all(self, threads=None):
        """Every element of every resident window against the oracle's
        reduce_scatter then allgather over the whole windows (their own chunk
        bounds), bit for bit."""
        import oracle
        c = self.cfg
        wins = [h.copy() for h in self.host]                 # the oracle works in place
        oracle.reduce_scatter(wins, c["rows"], c["cols"], c["ld"], oracle.SUM, oracle.F16)
        oracle.allgather(wins, c["rows"], c["cols"], c["ld"], oracle.F16)
        return _windows_parity(self.dev, wins, c["rows"], c["rows"])

    def oracle_rows_per_second(self):
        nb, dt, _ = self.oracle_sample(64)
        return 64.0 / max(dt, 1e-9)


class A2avBench(Workload):
    """all_to_all_v: 16 ranks, bf16 rows of 7168, target_rows 24576. With
    count_div > 1 every send count is divided by it (a sparse exchange on the
    same windows: 64 gives about 1 % of the capacity)."""

    def __init__(self, count_div=1):
        import synth
        self.cfg = synth.DISPATCH_BF16_N16_7168
        self.count_div = count_div
        self.name = ("all_to_all_v_n16_bf16_7168_maxrecv1536" if count_div == 1 else
                     "all_to_all_v_sparse_n16_bf16_7168_maxrecv1536_counts_div%d" % count_div)
        self.storage = "bf16"
        self.kernel = "pairs_claim_kernel<CopyMover>"
        self.dtype_compute = "u16"
        self.sources = MOVE_SOURCES

    def setup_host(self):
        import numpy as np
        import synth
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        self.mr = tr // n
        self.host = [synth.a2av_input(s, n, tr, size) for s in range(n)]
        self.sc = [synth.a2av_send_counts(s, n) // self.count_div for s in range(n)]
        moved = sum(int(np.clip(c_, 0, self.mr).sum()) for c_ in self.sc)
        self.moved_rows = moved

    def bytes_per_launch(self):
        n = self.cfg["nranks"]
        return 2 * 2 * self.cfg["size"] * self.moved_rows + 8 * n * n

    def launches_per_step(self):
        return 1

    def bytes_per_step(self):
        return self.bytes_per_launch()

    def setup_device(self, dev):
        import torch
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        self.dev = [_to_dev(h, dev) for h in self.host]
        self.d_sc = [_to_dev(x, dev) for x in self.sc]
        self.d_tg = [torch.full((tr, size), -1, dtype=torch.int16, device=dev) for _ in range(n)]
        self.d_rc = [torch.zeros(n, dtype=torch.int32, device=dev) for _ in range(n)]

    def launch(self, i, srcs=None, dst=None):
        import tile_level_collective_gb300 as P
        c = self.cfg
        P.ptoc_all_to_all_v(srcs or self.dev, self.d_tg, self.d_sc, self.d_rc, c["target_rows"], c["size"],
                            P.BF16)

    # e2e: inputs and send counts uploaded, targets and recv counts read back;
    # the targets start from the sentinel, so only rows the exchange wrote
    # can match the resident run's
    pipelined_e2e = True

    def setup_e2e(self, dev):
        import torch
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        self.pinned = [_pin(h) for h in self.host] + [_pin(x) for x in self.sc]
        self.e2e_in = [[torch.empty_like(t) for t in self.dev] + [torch.empty_like(t) for t in self.d_sc]
                       for _ in range(2)]
        self.e2e_out = [[torch.full((tr, size), -1, dtype=torch.int16, device=dev) for _ in range(n)] +
                        [torch.zeros(n, dtype=torch.int32, device=dev) for _ in range(n)] for _ in range(2)]
        self.out_pinned = [_pinned_like(self.e2e_out[0]) for _ in range(2)]

    def e2e_upload(self, b):
        _upload(self.e2e_in[b], self.pinned)

    def e2e_compute(self, b):
        import tile_level_collective_gb300 as P
        c = self.cfg
        n = c["nranks"]
        P.ptoc_all_to_all_v(self.e2e_in[b][:n], self.e2e_out[b][:n], self.e2e_in[b][n:], self.e2e_out[b][n:],
                            c["target_rows"], c["size"], P.BF16)

    def e2e_download(self, b):
        _download(self.out_pinned[b], self.e2e_out[b])

    def e2e_verify(self, b):
        _check_same(self.out_pinned[b], self.d_tg + self.d_rc, "target / recv_counts")

    def h2d_bytes(self):
        return sum(_nbytes(h) for h in self.host) + sum(_nbytes(x) for x in self.sc)

    def d2h_bytes(self):
        n = self.cfg["nranks"]
        return sum(_nbytes(h) for h in self.host) + 4 * n * n

    def config(self):
        c = self.cfg
        return {"workload": self.name, "op": "all_to_all_v", "nranks": c["nranks"], "storage_dtype": "bf16",
                "row_elems": c["size"], "target_rows": c["target_rows"], "max_recv": self.mr,
                "send_counts": "uniform int [0, 2047] per (src, dest), seed 1234 + src" +
                               ("" if self.count_div == 1 else ", divided by %d" % self.count_div),
                "moved_rows": self.moved_rows, "bytes_per_step": self.bytes_per_step(),
                "l2": L2_NOTE}

    def oracle_sample(self, rows):
        import numpy as np
        import oracle
        c = self.cfg
        n, size = c["nranks"], c["size"]
        # the same exchange with every count scaled into [0, rows]: a bounded sample
        mr = max(1, min(rows, self.mr))
        tr = mr * n
        ins = [np.ascontiguousarray(h.reshape(n, self.mr, size)[:, :mr].reshape(tr, size)) for h in self.host]
        tg = [np.empty((tr, size), dtype=np.uint16) for _ in range(n)]
        sc = [np.ascontiguousarray(np.clip(x, 0, self.mr) * mr // self.mr).astype(np.int32) for x in self.sc]
        rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
        t0 = time.perf_counter()
        oracle.all_to_all_v(ins, tg, sc, rc, tr, size, 2)
        dt = time.perf_counter() - t0
        moved = sum(int(x.sum()) for x in rc)
        return 4 * size * moved, dt, "the exchange with capacity %d rows per pair (counts scaled)" % mr

    def oracle_parity(self, rows):
        """The whole exchange on the host (a row copy per pair: seconds, and a
        second set of target windows in host memory) against the resident
        targets, sentinel rows included, and recv counts."""
        import numpy as np
        import oracle
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        tg = [np.full((tr, size), c["sentinel"], dtype=np.uint16) for _ in range(n)]
        rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
        sc = [np.ascontiguousarray(x, dtype=np.int32) for x in self.sc]
        oracle.all_to_all_v(self.host, tg, sc, rc, tr, size, 2)
        return _exchange_parity(self.d_tg, tg, "all %d target windows and recv counts" % n,
                                self.d_rc, rc)

    def oracle_rows_per_second(self):
        nb, dt, _ = self.oracle_sample(16)
        return 16.0 / max(dt, 1e-9)


class WindowOpBench(Workload):
    """allreduce (Sum) or broadcast (root 0) in place over 8 fp16 windows
    [8192, 4096] (the reduce_scatter / allgather shapes)."""

    def __init__(self, op):
        import synth
        self.op = op
        self.cfg = synth.WINDOWS_F16_N8_8192X4096
        self.name = "%s_n8_f16_8192x4096" % op
        self.storage = "f16"
        self.kernel = ("reduce_kernel<f16> (all-windows mode)" if op == "allreduce"
                       else "gather_kernel (fixed source window)")
        self.sources = REDUCE_SOURCES if op == "allreduce" else MOVE_SOURCES
        self.dtype_compute = "f32" if op == "allreduce" else "u16"

    def bytes_per_launch(self):
        c = self.cfg
        elems = c["rows"] * c["cols"]
        n = c["nranks"]
        # allreduce: N reads + N writes per element; broadcast: 1 read + N-1 writes
        return (2 * n if self.op == "allreduce" else n) * 2 * elems

    def launches_per_step(self):
        return 1

    def bytes_per_step(self):
        return self.bytes_per_launch()

    def setup_host(self):
        import synth
        self.host = [synth.window(r, self.cfg) for r in range(self.cfg["nranks"])]

    def setup_device(self, dev):
        self.dev = [_to_dev(h, dev) for h in self.host]
        self.saved = [t.clone() for t in self.dev]

    def prepare(self):
        for t, s in zip(self.dev, self.saved):
            t.copy_(s)

    def launch(self, i, srcs=None, dst=None):
        import tile_level_collective_gb300 as P
        c = self.cfg
        wins = srcs or self.dev
        if self.op == "allreduce":
            P.ptoc_allreduce(wins, c["rows"], c["cols"], c["ld"], P.SUM, P.F16)
        else:
            P.ptoc_broadcast(wins, c["rows"], c["cols"], c["ld"], P.F16, root=0)

    # e2e: windows uploaded, updated in place, read back
    pipelined_e2e = True
    e2e_inplace = True

    def setup_e2e(self, dev):
        import torch
        self.pinned = [_pin(h) for h in self.host]
        self.e2e_win = [[torch.empty_like(t) for t in self.dev] for _ in range(2)]
        self.out_pinned = [_pinned_like(self.dev) for _ in range(2)]

    def e2e_upload(self, b):
        _upload(self.e2e_win[b], self.pinned)

    def e2e_compute(self, b):
        self.launch(0, srcs=self.e2e_win[b])

    def e2e_download(self, b):
        _download(self.out_pinned[b], self.e2e_win[b])

    def e2e_verify(self, b):
        _check_same(self.out_pinned[b], self.dev, "window")

    def h2d_bytes(self):
        return sum(_nbytes(h) for h in self.host)

    def d2h_bytes(self):
        return sum(_nbytes(h) for h in self.host)

    def config(self):
        c = self.cfg
        return {"workload": self.name, "op": self.op, "nranks": c["nranks"], "storage_dtype": "f16",
                "shape": [c["rows"], c["cols"]], "ld": c["ld"], "values": "normal(0,1)",
                "step": "one in-place %s (inputs restored before every step, outside the timed events)" % self.op,
                "bytes_per_step": self.bytes_per_step(), "l2": L2_NOTE}

    def oracle_sample(self, rows):
        import numpy as np
        import oracle
        c = self.cfg
        rows = max(1, min(rows, c["rows"]))
        wins = [h[:rows].copy() for h in self.host]          # the oracle works in place
        t0 = time.perf_counter()
        if self.op == "allreduce":
            oracle.allreduce(wins, rows, c["cols"], c["ld"], oracle.SUM, oracle.F16)
        else:
            oracle.broadcast(wins, 0, rows, c["cols"], c["ld"], oracle.F16)
        dt = time.perf_counter() - t0
        n = c["nranks"]
        nb = (2 * n if self.op == "allreduce" else n) * 2 * rows * c["cols"]
        return nb, dt, "%s over rows 0..%d of the 8 windows" % (self.op, rows - 1)

    def oracle_parity(self, rows):
        """Both operations act row by row, so the oracle's pass over the first
        rows gives the full-size values there."""
        import numpy as np
        import oracle
        c = self.cfg
        rows = max(1, min(rows, c["rows"]))
        wins = [h[:rows].copy() for h in self.host]          # the oracle works in place
        if self.op == "allreduce":
            oracle.allreduce(wins, rows, c["cols"], c["ld"], oracle.SUM, oracle.F16)
        else:
            oracle.broadcast(wins, 0, rows, c["cols"], c["ld"], oracle.F16)
        return _windows_parity(self.dev, wins, rows, c["rows"])

    def oracle_parity_all(self, threads=None):
        """Every element of every resident window against the oracle over the
        whole windows, bit for bit. Both operations act row by row, so the
        oracle runs on contiguous row slices of the windows, one host thread
        each."""
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        c = self.cfg
        rows = c["rows"]
        threads = threads or os.cpu_count() or 1
        wins = [h.copy() for h in self.host]                 # the oracle works in place
        bounds = [rows * t // threads for t in range(threads + 1)]

        def part(t):
            a, b = bounds[t], bounds[t + 1]
            if b <= a:
                return
            sl = [w[a:b] for w in wins]
            if self.op == "allreduce":
                oracle.allreduce(sl, b - a, c["cols"], c["ld"], oracle.SUM, oracle.F16)
            else:
                oracle.broadcast(sl, 0, b - a, c["cols"], c["ld"], oracle.F16)

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(part, range(threads)))
        return _windows_parity(self.dev, wins, rows, rows)

    def oracle_rows_per_second(self):
        nb, dt, _ = self.oracle_sample(64)
        return 64.0 / max(dt, 1e-9)


class PairsBench(A2avBench):
    """The symmetric all_to_all (every count = MAX_RECV), or the all_to_all_v
    combine with AtomicType kAdd (the return leg of the dispatch workload:
    bf16 rows added into the senders' outputs), on the MoE dispatch shapes."""

    def __init__(self, op):
        super().__init__()
        self.op = op
        self.name = ("all_to_all_n16_bf16_7168_chunk1536" if op == "all_to_all"
                     else "all_to_all_v_combine_add_n16_bf16_7168_maxrecv1536")
        self.kernel = "pairs_kernel<CopyMover>" if op == "all_to_all" else "pairs_claim_kernel<AddMover<bf16>>"
        # the combine uploads into its outputs (kAdd reads them)
        self.e2e_inplace = op == "combine"
        self.dtype_compute = "u16" if op == "all_to_all" else "f32"

    def setup_host(self):
        import numpy as np
        import synth
        super().setup_host()
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        if self.op == "all_to_all":
            self.moved_rows = n * n * self.mr
        else:
            # dispatch values are normal bf16 (added, so they should be numbers)
            self.host = [synth.values(("normal", 0, 1), synth.DT_BF16, 1234 + s, tr * size).reshape(tr, size)
                         for s in range(n)]
            self.out_host = [synth.values(("normal", 0, 1), synth.DT_BF16, 5678 + s, tr * size).reshape(tr, size)
                             for s in range(n)]

    def bytes_per_launch(self):
        n = self.cfg["nranks"]
        row = 2 * self.cfg["size"]
        if self.op == "all_to_all":
            return 2 * row * self.moved_rows
        # combine with kAdd: read the window row, read and write the output row
        return 3 * row * self.moved_rows + 4 * n * n

    def setup_device(self, dev):
        import torch
        import tile_level_collective_gb300 as P
        super().setup_device(dev)
        c = self.cfg
        if self.op == "combine":
            P.ptoc_all_to_all_v(self.dev, self.d_tg, self.d_sc, self.d_rc, c["target_rows"], c["size"], P.BF16)
            self.d_out = [_to_dev(o, dev) for o in self.out_host]
            self.saved = [t.clone() for t in self.d_out]
            torch.cuda.synchronize()

    def prepare(self):
        if self.op == "combine":
            for t, s in zip(self.d_out, self.saved):
                t.copy_(s)

    def launch(self, i, srcs=None, dst=None):
        import tile_level_collective_gb300 as P
        c = self.cfg
        if self.op == "all_to_all":
            P.ptoc_all_to_all(srcs or self.dev, self.d_tg, c["target_rows"], c["size"], P.BF16)
        else:
            P.ptoc_all_to_all_v_combine(srcs or self.d_tg, self.d_out, self.d_rc, c["target_rows"], c["size"],
                                        P.ATOMIC_ADD, P.BF16)

    # e2e, all_to_all: inputs uploaded, targets (from the sentinel) read back.
    # combine: the dispatched windows, the recv counts and the outputs' prior
    # contents (kAdd adds into them) uploaded, the outputs read back.
    def setup_e2e(self, dev):
        import torch
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        if self.op == "all_to_all":
            self.pinned = [_pin(h) for h in self.host]
            self.e2e_in = [[torch.empty_like(t) for t in self.dev] for _ in range(2)]
            self.e2e_out = [[torch.full((tr, size), -1, dtype=torch.int16, device=dev) for _ in range(n)]
                            for _ in range(2)]
            self.e2e_ref = self.d_tg
        else:
            self.pinned = ([_pin(t.cpu().numpy()) for t in self.d_tg] + [_pin(t.cpu().numpy()) for t in self.d_rc] +
                           [_pin(t.cpu().numpy()) for t in self.saved])
            self.e2e_in = [[torch.empty_like(t) for t in self.d_tg] + [torch.empty_like(t) for t in self.d_rc]
                           for _ in range(2)]
            # the outputs are uploaded too (kAdd reads them), into the set's output buffers
            self.e2e_out = [[torch.empty_like(t) for t in self.d_out] for _ in range(2)]
            self.e2e_ref = self.d_out
        self.out_pinned = [_pinned_like(self.e2e_out[0]) for _ in range(2)]

    def e2e_upload(self, b):
        if self.op == "all_to_all":
            _upload(self.e2e_in[b], self.pinned)
        else:
            n = self.cfg["nranks"]
            _upload(self.e2e_in[b], self.pinned[:2 * n])
            _upload(self.e2e_out[b], self.pinned[2 * n:])

    def e2e_compute(self, b):
        import tile_level_collective_gb300 as P
        c = self.cfg
        n = c["nranks"]
        if self.op == "all_to_all":
            P.ptoc_all_to_all(self.e2e_in[b], self.e2e_out[b], c["target_rows"], c["size"], P.BF16)
        else:
            P.ptoc_all_to_all_v_combine(self.e2e_in[b][:n], self.e2e_out[b], self.e2e_in[b][n:], c["target_rows"],
                                        c["size"], P.ATOMIC_ADD, P.BF16)

    def e2e_download(self, b):
        _download(self.out_pinned[b], self.e2e_out[b])

    def e2e_verify(self, b):
        _check_same(self.out_pinned[b], self.e2e_ref, "output")

    def h2d_bytes(self):
        if self.op == "all_to_all":
            return sum(_nbytes(h) for h in self.host)
        n = self.cfg["nranks"]
        return sum(_nbytes(t) for t in self.d_tg) + 4 * n * n + sum(_nbytes(t) for t in self.saved)

    def d2h_bytes(self):
        return sum(_nbytes(t) for t in (self.d_tg if self.op == "all_to_all" else self.d_out))

    def config(self):
        c = dict(super().config())
        c["workload"] = self.name
        c["op"] = self.op if self.op == "all_to_all" else "all_to_all_v_combine (AtomicType kAdd)"
        if self.op == "all_to_all":
            c.pop("send_counts", None)
            c["chunk_rows"] = self.mr
        c["moved_rows"] = self.moved_rows
        c["bytes_per_step"] = self.bytes_per_step()
        return c

    def oracle_sample(self, rows):
        import numpy as np
        import oracle
        c = self.cfg
        n, size = c["nranks"], c["size"]
        mr = max(1, min(rows, self.mr))
        tr = mr * n
        ins = [np.ascontiguousarray(h.reshape(n, self.mr, size)[:, :mr].reshape(tr, size)) for h in self.host]
        if self.op == "all_to_all":
            tg = [np.empty((tr, size), dtype=np.uint16) for _ in range(n)]
            t0 = time.perf_counter()
            oracle.all_to_all(ins, tg, tr, size, 2)
            dt = time.perf_counter() - t0
            return 4 * size * n * n * mr, dt, "all_to_all with chunks of %d rows" % mr
        # a copy: the kAdd combine adds into its outputs in place
        outs = [h.reshape(n, self.mr, size)[:, :mr].reshape(tr, size).copy() for h in self.out_host]
        rc = [np.clip(np.array(x), 0, self.mr).astype(np.int32) * mr // self.mr for x in self.sc]
        rc = [np.ascontiguousarray(np.array([rc[s][d] for s in range(n)], np.int32)) for d in range(n)]
        t0 = time.perf_counter()
        oracle.all_to_all_v_combine(ins, outs, rc, tr, size, oracle.ATOMIC_ADD, oracle.BF16)
        dt = time.perf_counter() - t0
        moved = sum(int(x.sum()) for x in rc)
        return 6 * size * moved, dt, "the kAdd combine with capacity %d rows per pair (counts scaled)" % mr

    def oracle_parity(self, rows):
        """The whole operation on the host against the resident outputs, bit
        for bit. The combine's windows come from the oracle's own dispatch of
        the same inputs and counts, and it adds into copies of the prior
        outputs (the resident outputs are restored before every step)."""
        import numpy as np
        import oracle
        c = self.cfg
        n, tr, size = c["nranks"], c["target_rows"], c["size"]
        if self.op == "all_to_all":
            tg = [np.full((tr, size), c["sentinel"], dtype=np.uint16) for _ in range(n)]
            oracle.all_to_all(self.host, tg, tr, size, 2)
            return _exchange_parity(self.d_tg, tg, "all %d target windows" % n)
        win = [np.full((tr, size), c["sentinel"], dtype=np.uint16) for _ in range(n)]
        rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
        sc = [np.ascontiguousarray(x, dtype=np.int32) for x in self.sc]
        oracle.all_to_all_v(self.host, win, sc, rc, tr, size, 2)
        outs = [o.copy() for o in self.out_host]
        oracle.all_to_all_v_combine(win, outs, rc, tr, size, oracle.ATOMIC_ADD, oracle.BF16)
        del win
        return _exchange_parity(self.d_out, outs, "all %d output windows" % n)


class BarrierBench(Workload):
    """The credit barrier among N ranks simulated on the GPU: one launch of G
    generations; the metric is the latency of one generation."""
    metric = "credit barrier latency per generation"
    unit = "us"

    def __init__(self, nranks=8, generations=1000):
        self.n, self.g = nranks, generations
        self.name = "credit_barrier_n%d_g%d" % (nranks, generations)
        self.kernel = "credit_barrier_kernel (cooperative, one warp per rank)"
        self.dtype_compute = "i32"
        self.sources = MOVE_SOURCES

    def launches_per_step(self):
        return 1

    def bytes_per_step(self):
        return 0

    def bytes_per_launch(self):
        return 0

    def setup_host(self):
        pass

    def setup_device(self, dev):
        import torch
        self.sig = [torch.zeros(self.n, dtype=torch.int32, device=dev) for _ in range(self.n)]
        self.status = torch.zeros(self.n, dtype=torch.int32, device=dev)

    def launch(self, i, srcs=None, dst=None):
        import tile_level_collective_gb300 as P
        P.ptoc_credit_barrier(self.sig, list(range(self.n)), self.g, 10 ** 9, self.status)

    def config(self):
        return {"workload": self.name, "op": "credit barrier", "nranks": self.n, "generations": self.g,
                "step": "one call of %d generations, all ranks in one cooperative launch" % self.g}


def make_workload(name, rows_div=1):
    """The named workload; rows_div > 1 divides its row counts (a smaller case
    of the same kernel, for profiler captures)."""
    import synth
    wl = None
    if name in ("treduce", "treduce_bf16"):
        wl = TreduceBench(synth.treduce_bf16_n8_4096_valid4000(), "bf16")
    elif name == "treduce_small":
        wl = TreduceBench(synth.treduce_f32_n4_256(), "f32")
    elif name == "treduce_f32":
        wl = TreduceBench(synth.treduce_f32_n8_16384x8192(), "f32")
    elif name == "treduce_i32":
        wl = TreduceBench(synth.treduce_i32_n8_16384x8192(), "i32")
    elif name == "treduce_16384x8192":
        wl = TreducePairBench([TreduceBench(synth.treduce_f32_n8_16384x8192(), "f32"),
                               TreduceBench(synth.treduce_i32_n8_16384x8192(), "i32")])
    elif name == "rs_ag":
        wl = RsAgBench()
    elif name == "a2av":
        wl = A2avBench()
    elif name == "a2av_sparse":
        wl = A2avBench(count_div=64)
    elif name in ("allreduce", "broadcast"):
        wl = WindowOpBench(name)
    elif name in ("all_to_all", "combine"):
        wl = PairsBench(name)
    elif name == "barrier":
        wl = BarrierBench()
    else:
        raise SystemExit("unknown workload %s" % name)
    if rows_div > 1:
        if isinstance(wl, (TreduceBench, TreducePairBench)):
            for part in getattr(wl, "parts", [wl]):
                w = part.w
                w.rows, w.valid_rows = w.rows // rows_div, w.valid_rows // rows_div
                w.name += "_rows_div%d" % rows_div
                part.name = w.name
            if isinstance(wl, TreducePairBench):
                wl.name += "_rows_div%d" % rows_div
        else:
            wl.cfg = dict(wl.cfg)
            key = "rows" if isinstance(wl, (RsAgBench, WindowOpBench)) else "target_rows"
            wl.cfg[key] = wl.cfg[key] // rows_div
            wl.name += "_rows_div%d" % rows_div
    return wl


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def torch_uint8():
    import torch
    return torch.uint8


def _nbytes(a):
    return int(a.nbytes) if hasattr(a, "nbytes") else a.numel() * a.element_size()


def _to_dev(h, dev):
    import numpy as np
    import torch
    h = np.ascontiguousarray(h)
    t = torch.from_numpy(h.view(np.int16) if h.dtype == np.uint16 else h)
    return t.to(dev)


def _upload(dsts, pinned):
    for d, h in zip(dsts, pinned):
        d.view(-1).view(torch_uint8()).copy_(h, non_blocking=True)


def _download(pinned, srcs):
    for o, d in zip(pinned, srcs):
        o.copy_(d.view(-1).view(torch_uint8()), non_blocking=True)


def _pinned_like(ts):
    import torch
    return [torch.empty(_nbytes(t), dtype=torch.uint8).pin_memory() for t in ts]


def _check_same(pinned, refs, what):
    """The downloaded bytes equal the resident run's result tensors."""
    for i, (o, d) in enumerate(zip(pinned, refs)):
        if not bool((o == d.reshape(-1).view(torch_uint8()).cpu()).all()):
            raise RuntimeError("pipelined end-to-end %s %d differs from the resident result" % (what, i))


def _windows_parity(dev_windows, want, rows, total_rows):
    """The resident windows' first `rows` rows against the oracle's windows,
    bit for bit."""
    import numpy as np
    bad = [r for r, (d, w) in enumerate(zip(dev_windows, want))
           if not np.array_equal(np.ascontiguousarray(d[:rows].cpu().numpy()).view(np.uint8), w.view(np.uint8))]
    return {"rows": "0..%d of %d" % (rows - 1, total_rows),
            "result": "bit-exact" if not bad else "MISMATCH in windows " + ", ".join(map(str, bad))}


def _exchange_parity(dev_out, want, what, dev_counts=None, want_counts=None):
    """Whole resident output windows (and counts) against the oracle's, bit
    for bit, one window at a time."""
    import numpy as np
    bad = []
    for d, (t, w) in enumerate(zip(dev_out, want)):
        got = np.ascontiguousarray(t.cpu().numpy()).view(np.uint8)
        if not np.array_equal(got, w.view(np.uint8)):
            bad.append(d)
        elif dev_counts is not None and not np.array_equal(dev_counts[d].cpu().numpy(), want_counts[d]):
            bad.append(d)
    return {"rows": what, "result": "bit-exact" if not bad else "MISMATCH in windows " + ", ".join(map(str, bad))}


def _pin(h):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(h).reshape(-1).view(np.uint8)).pin_memory()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs (copy, burst): of measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s: of fallback"


def kernel_source_hash(files):
    """Hash of the given library source files (kernels, launch code, header)."""
    h = hashlib.sha256()
    for rel in files:
        h.update(rel.encode())
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name, files):
    """DRAM bytes per launch recorded from an ncu capture of the current
    sources of the workload's kernel (profiles/traffic.txt lines: workload
    sha bytes), else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_source_hash(files)
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload_name and parts[1] == sha:
            return int(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        note = []
        if not inside:
            inside = [min(self.rows, key=lambda x: abs(x[0] - (t0 + t1) / 2))[1]]
            note = ["nearest sample (timed region shorter than the sampling period)"]
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons) + note, "samples": len(inside)}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# A replica that dies or never reaches the timing exchange makes the others
# fail with an error after this long instead of waiting for the backend's
# default (ten minutes for NCCL).
PG_TIMEOUT_S = 300


def init_replicas(backend, timeout_s=PG_TIMEOUT_S, **kw):
    import datetime
    import torch.distributed as dist
    dist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s), **kw)


def aggregate(ms_local, bytes_per_step, world, device):
    """Whole-job figures of a replica run: the step time is the max over ranks
    and `value` counts the bytes every rank processed (weak scaling)."""
    ms = max_over_ranks(ms_local, world, device)
    return ms, world * bytes_per_step / (ms / 1e3) / 1e9


def cpu_baseline(wl, budget_s):
    """The oracle as it stands, single-threaded, on a sample of the workload
    (at most the whole step), repeated to about `budget_s` seconds of CPU
    work."""
    rps = wl.oracle_rows_per_second()
    rows = max(1, int(rps * budget_s))
    nb_tot, dt_tot, reps, desc = 0, 0.0, 0, ""
    while dt_tot < budget_s or reps == 0:
        nb, dt, desc = wl.oracle_sample(rows)
        nb_tot, dt_tot, reps = nb_tot + nb, dt_tot + dt, reps + 1
    line = {"value": nb_tot / dt_tot / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%s, %d repetition(s)" % (desc, reps), "seconds": round(dt_tot, 3)}
    if hasattr(wl, "oracle_parity_all"):
        # untimed: every element of the resident run's results against the
        # oracle (row slices on every host core)
        line["parity"] = wl.oracle_parity_all()
    elif hasattr(wl, "oracle_parity"):
        # the same sample, untimed, against the resident run's results
        line["parity"] = wl.oracle_parity(rows)
    if "parity" in line:
        if line["parity"]["result"] != "bit-exact":
            print("bench: results differ from the oracle: %s" % line["parity"], file=sys.stderr)
    if hasattr(wl, "oracle_sample_threaded"):
        # the same oracle over every host core, rows split into contiguous slices
        threads = os.cpu_count() or 1
        n_rows = max(threads, int(rps * threads * budget_s / 4))
        nb_t, dt_t, reps_t = 0, 0.0, 0
        while dt_t < budget_s / 4 or reps_t == 0:
            nb, dt, _ = wl.oracle_sample_threaded(n_rows, threads)
            nb_t, dt_t, reps_t = nb_t + nb, dt_t + dt, reps_t + 1
        line["all_cores"] = {"value": nb_t / dt_t / 1e9, "cores": threads, "seconds": round(dt_t, 3),
                             "sample": "the first %d rows, split into %d row slices on as many threads, "
                             "%d repetition(s)" % (min(n_rows, wl.max_rows()), threads, reps_t)}
    return line


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        init_replicas("nccl")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    wl = make_workload(args.workload, args.rows_div)
    wl.setup_host()
    wl.setup_device(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    nl = wl.launches_per_step()

    for _ in range(args.warmup):
        wl.prepare()
        flush(1)
        for i in range(nl):
            wl.launch(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        time.sleep(0.6)          # let the sampler start before the timed region
    nev = nl if wl.per_launch_timing else 1

    def timed_block():
        """K steps, each bracketed by CUDA events on the launching stream;
        returns the events."""
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nev)] for _ in range(args.steps)]
        for k in range(args.steps):
            wl.prepare()
            flush(k)
            if wl.per_launch_timing:
                for i in range(nl):
                    ev[k][i][0].record(stream)
                    wl.launch(i)
                    ev[k][i][1].record(stream)
            else:
                ev[k][0][0].record(stream)
                for i in range(nl):
                    wl.launch(i)
                ev[k][0][1].record(stream)
        torch.cuda.synchronize()
        return ev

    # The K-step block is timed again, back to back, until the timed region
    # spans --min-timed-seconds, so that the clock sampler sees it several
    # times; every timed step counts.
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    blocks = []
    while not blocks or time.time() - t0 < args.min_timed_seconds:
        blocks.append(timed_block())
    barrier()
    t1 = time.time()
    if sampler:
        sampler.stop()
    timed = [[ev[k][i][0].elapsed_time(ev[k][i][1]) for i in range(nev)] for ev in blocks
             for k in range(args.steps)]
    # a step = its launches on the stream (the flush between steps excluded)
    step_ms = [sum(x) for x in timed]
    ms_local = sum(step_ms) / len(step_ms)
    ms, value = aggregate(ms_local, wl.bytes_per_step(), world, dev)
    block_gbs = sorted(wl.bytes_per_step() * args.steps / (sum(step_ms[b * args.steps:(b + 1) * args.steps])
                                                           / 1e3) / 1e9 for b in range(len(blocks)))

    # roofline of the dominant kernel: launch 0 when launches are timed one by
    # one, else the step's average launch (all of one kernel family)
    if wl.per_launch_timing:
        avg0 = statistics.mean(x[0] for x in timed)
    else:
        avg0 = statistics.mean(step_ms) / nl
    achieved = wl.bytes_per_launch() / (avg0 / 1e3) / 1e9
    peak, peak_src = measured_peak()
    traffic = recorded_traffic(wl.name, wl.sources)

    if isinstance(wl, BarrierBench):
        if rank == 0:
            us = ms * 1e3 / wl.g
            print(json.dumps({"metric": wl.metric, "value": round(us, 4), "unit": wl.unit, "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
                              "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
                              "dtype": "i32", "data": "synthetic", "config": wl.config(),
                              "roofline": None, "e2e": None, "gpu_launches": args.steps * len(blocks),
                              "clocks": sampler.summary(t0, t1) if sampler else None}), flush=True)
        return

    # end to end: pinned host inputs in, results out, every step
    if args.no_e2e:
        e_ms, e_value, e_up = None, None, None
    else:
        e_ms, e_value, e_up = run_e2e(wl, args, dev, stream, world, barrier)
    link = host_link_gbs(dev) + (e_up,) if e_value is not None and rank == 0 else None
    if rank != 0:
        return
    line = build_line(args, wl, world, value, ms, achieved, avg0, peak, peak_src, traffic, e_value, e_ms, nl,
                      sampler.summary(t0, t1) if sampler else None, len(blocks), block_gbs, t1 - t0, link)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_e2e_pipelined(wl, args, dev, world, barrier):
    """Steps of upload -> compute -> download on three streams with two
    buffer sets: step k's upload waits for step k-2's compute to release its
    input set (for in-place ops, for its download), its compute for its upload
    and for step k-2's download to release its output set; the timed region
    spans the first upload to the last download."""
    import torch
    wl.setup_e2e(dev)
    up, comp, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    uploaded, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]
    upload_events = []

    def run(steps, timed=False):
        for k in range(steps):
            b = k & 1
            with torch.cuda.stream(up):
                if used[b]:
                    # the set's inputs are free once computed; in place, its
                    # results must also have been read back
                    up.wait_event(downloaded[b] if wl.e2e_inplace else computed[b])
                if timed:
                    upload_events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                    upload_events[-1][0].record(up)
                wl.e2e_upload(b)
                if timed:
                    upload_events[-1][1].record(up)
                uploaded[b].record(up)
            with torch.cuda.stream(comp):
                comp.wait_event(uploaded[b])
                if used[b]:
                    comp.wait_event(downloaded[b])
                wl.e2e_compute(b)
                computed[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                wl.e2e_download(b)
                downloaded[b].record(down)
            used[b] = True

    run(max(2, min(args.warmup, 3)))
    torch.cuda.synchronize()
    e_steps = max(3, min(args.e2e_steps, args.steps))
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    es.record(up)
    run(e_steps, timed=True)
    down.wait_stream(up)
    down.wait_stream(comp)
    ee.record(down)
    torch.cuda.synchronize()
    wl.e2e_verify((e_steps - 1) & 1)
    up_ms = sum(a.elapsed_time(b) for a, b in upload_events)
    upload_gbs = wl.h2d_bytes() * len(upload_events) / (up_ms / 1e3) / 1e9 if up_ms > 0 else None
    e_ms, e_value = aggregate(es.elapsed_time(ee) / e_steps, wl.bytes_per_step(), world, dev)
    return e_ms, e_value, upload_gbs


def run_e2e(wl, args, dev, stream, world, barrier):
    if not wl.pipelined_e2e:
        raise SystemExit("workload %s has no end-to-end leg" % wl.name)
    return run_e2e_pipelined(wl, args, dev, world, barrier)


def host_link_gbs(dev, nbytes=256 << 20, reps=5):
    """Pinned host <-> device copy rates on this machine (GB/s, best of `reps`
    copies of `nbytes` each way, timed with events on a stream of their own):
    the bound the e2e leg is compared against."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    rates = []
    for up in (True, False):
        best = None
        with torch.cuda.stream(s):
            for _ in range(reps + 1):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                (d.copy_(h, non_blocking=True) if up else h.copy_(d, non_blocking=True))
                b.record(s)
                b.synchronize()
                ms = a.elapsed_time(b)
                best = ms if best is None else min(best, ms)
        rates.append(nbytes / (best / 1e3) / 1e9)
    del h, d
    return rates[0], rates[1]


def line_config(wl, world):
    """The `config` of both arms' lines (identical for the same workload and
    rank count)."""
    return dict(wl.config(), parallelism="replicas" if world > 1 else "single GPU")


def e2e_link_bound(wl, link, world, during=None):
    """The e2e leg's bound on this machine: every byte of a step crosses the
    host link, uploads and downloads each at their measured rate and never
    slowing each other (an optimistic bound: measured together, both ran
    about a fifth slower). `during` is the upload rate the e2e leg itself
    saw (its uploads timed on their stream), which other traffic on the
    host side can hold below the probe's."""
    up, down = link
    t = max(wl.h2d_bytes() / (up * 1e9), wl.d2h_bytes() / (down * 1e9))
    return {"h2d_gbs": round(up, 1), "d2h_gbs": round(down, 1),
            "bound_gbs": round(wl.bytes_per_step() * world / t / 1e9, 2) if t > 0 else None,
            "measured": "pinned 256 MiB copies each way on this GPU, best of 5, after the e2e leg",
            "h2d_gbs_during_e2e": round(during, 1) if during else None}


def build_line(args, wl, world, value, ms, achieved, avg0, peak, peak_src, traffic, e_value, e_ms, nl, clocks,
               nblocks=1, block_gbs=None, timed_s=None, link=None):
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype_compute, "data": "synthetic (seeded SplitMix64, generated on the host)",
        "config": line_config(wl, world),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": wl.kernel,
                     "bytes_per_launch": wl.bytes_per_launch(), "avg_launch_ms": round(avg0, 6),
                     "peak_source": peak_src},
        "e2e": None if e_value is None else {
            "value": round(e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": wl.h2d_bytes(),
            "d2h_bytes_per_step": wl.d2h_bytes(), "ms_per_step": round(e_ms, 6),
            "path": ("every step: pinned host -> device copy of its inputs, the library calls, device -> "
                     "pinned host copy of its results; double-buffered on three streams (upload of step k "
                     "overlaps compute and download of step k-1); the last results checked against the "
                     "resident run"),
            "link": e2e_link_bound(wl, link[:2], world, link[2]) if link else None},
        "gpu_launches": nl * args.steps * nblocks,
        "timing": ("CUDA events around each launch" if wl.per_launch_timing else
                   "CUDA events around each step; its %d launches run back to back (programmatic "
                   "dependent launch lets each overlap the previous one's tail)" % nl)
        + ("; the %d-step block timed %d times back to back (%.2f s of timed region, so that the clock "
           "record samples it), value over all %d timed steps" % (args.steps, nblocks, timed_s or 0.0,
                                                                  args.steps * nblocks)),
        "timed_blocks": nblocks,
        "block_gbs": None if not block_gbs else {"min": round(block_gbs[0], 2),
                                                 "median": round(statistics.median(block_gbs), 2),
                                                 "max": round(block_gbs[-1], 2)},
        "clocks": clocks,
    }
    return line


def run_reference(args):
    """The oracle on the host cores, each step a bounded sample of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = make_workload(args.workload, args.rows_div)
    if isinstance(wl, BarrierBench):
        print(json.dumps({"impl": "reference", "unavailable": "the credit barrier has no CPU timing arm "
                          "(the oracle is a sequential step machine, not a barrier)"}), flush=True)
        return
    wl.setup_host()
    total_steps = args.steps + args.warmup
    per_step = max(0.002, args.reference_seconds / max(1, total_steps))
    rows = max(1, int(wl.oracle_rows_per_second() * per_step))
    for _ in range(args.warmup):
        wl.oracle_sample(rows)
    nb_tot, dt_tot, desc = 0, 0.0, ""
    for _ in range(args.steps):
        nb, dt, desc = wl.oracle_sample(rows)
        nb_tot += nb
        dt_tot += dt
    value = nb_tot / dt_tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt_tot / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype_compute,
        "data": "synthetic (seeded SplitMix64, generated on the host)",
        "config": line_config(wl, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="treduce_16384x8192",
                    choices=["treduce_16384x8192", "treduce", "treduce_bf16", "treduce_small", "treduce_f32",
                             "treduce_i32",
                             "rs_ag", "a2av", "a2av_sparse", "allreduce", "broadcast", "all_to_all", "combine",
                             "barrier"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--min-timed-seconds", type=float, default=0.5,
                    help="repeat the timed K-step block until the timed region spans this long")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiler runs)")
    ap.add_argument("--rows-div", type=int, default=1,
                    help="divide the workload's rows (a smaller case for profiler captures)")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
