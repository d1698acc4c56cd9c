"""Host-side logic of the multi-GPU benchmark, on CPU: world-size-2 gloo ranks
run bench.aggregate (max step time over ranks, whole-job value) and fail with an
error, not a hang, when one rank leaves before the exchange; the argument
parser keeps its documented defaults (one GPU, at least three warm-up steps,
the 16384 x 8192 TREDUCE case), and the reference arm's JSON line has the keys
of the benchmark line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [2.0, 5.0][rank]          # rank 1 is the slow one
    ms, value = bench.aggregate(ms_local, 1_000_000_000, world, torch.device("cpu"))
    results[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    for rank in range(world):
        ms, value = got[rank]
        assert ms == 5.0                              # the max over ranks
        assert abs(value - 2 * 1e9 / 5e-3 / 1e9) < 1e-6  # both ranks' bytes / max time


def _rank_leaves_early(rank, world, port, mode, results):
    import time
    import torch
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    bench.init_replicas("gloo", timeout_s=3, rank=rank, world_size=world)
    if rank == 1:
        if mode == "stalls":             # alive, but never reaches the exchange
            time.sleep(8)
        return                           # leaves before the timing exchange
    t0 = time.time()
    try:
        bench.aggregate(2.0, 1_000_000_000, world, torch.device("cpu"))
        results[rank] = ("no error", time.time() - t0)
    except Exception as e:               # the backend reports the missing peer
        results[rank] = (type(e).__name__, time.time() - t0)


@pytest.mark.parametrize("mode", ["exits", "stalls"])
def test_a_replica_that_leaves_makes_the_others_fail_not_hang(mode):
    """A rank that exits, or stalls, before the max-over-ranks exchange: the
    remaining rank's exchange raises (a closed connection at once, or the
    process group's 3 s timeout) instead of waiting."""
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_leaves_early, args=(world, port, mode, results), nprocs=world, join=True)
        got = dict(results)
    what, seconds = got[0]
    assert what != "no error"
    assert seconds < 10


def test_parity_leg_compares_the_resident_results():
    """The CPU-baseline leg's parity check on host stand-ins for the resident
    results: a correct result passes, one changed element fails, and a sample
    that stops before the changed row passes."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    wl = bench.make_workload("treduce_small", 1)
    wl.setup_host()
    w = wl.w
    wl.dst_init = np.zeros((w.rows, w.ld), dtype=wl.host[0].dtype)
    good = wl.dst_init.copy()
    assert oracle.treduce(wl.host, good, w.valid_rows, w.valid_cols, w.ld, oracle.SUM, oracle.F32) == 0
    wl.dsts = [torch.from_numpy(good.copy())]
    assert wl.oracle_parity(64)["result"] == "bit-exact"
    bad = good.copy()
    bad[3, 5] = np.nextafter(bad[3, 5], np.float32(10))
    wl.dsts = [torch.from_numpy(bad)]
    assert wl.oracle_parity(64)["result"] == "MISMATCH in sum"
    assert wl.oracle_parity(3)["result"] == "bit-exact"


@pytest.mark.parametrize("name", ["rs_ag", "allreduce", "broadcast"])
def test_window_samples_leave_the_inputs_alone(name):
    """The oracle works in place on windows: the CPU-baseline sample and the
    parity check must run it on copies, so that repeated samples, and the
    parity check after them, see the workload's own inputs (small windows
    stand in for the 8 x 8192 x 4096 ones)."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    wl = bench.make_workload(name, 1)
    wl.cfg = dict(wl.cfg, nranks=4, rows=12, cols=40, ld=40)
    wl.setup_host()
    before = [h.copy() for h in wl.host]
    for _ in range(3):
        wl.oracle_sample(12)
    assert all(np.array_equal(a, b) for a, b in zip(before, wl.host))
    want = [h.copy() for h in wl.host]
    c = wl.cfg
    if name == "rs_ag":
        oracle.reduce_scatter(want, 12, 40, 40, oracle.SUM, oracle.F16)
        oracle.allgather(want, 12, 40, 40, oracle.F16)
    elif name == "allreduce":
        oracle.allreduce(want, 12, 40, 40, oracle.SUM, oracle.F16)
    else:
        oracle.broadcast(want, 0, 12, 40, 40, oracle.F16)
    wl.dev = [torch.from_numpy(w.view(np.int16).copy()) for w in want]      # stand-ins for the resident run
    assert wl.oracle_parity(12)["result"] == "bit-exact"
    assert wl.oracle_parity(5)["result"] == "bit-exact"
    # the full-size leg: every row of every window, row slices on threads
    assert wl.oracle_parity_all(threads=5)["result"] == "bit-exact"
    assert all(np.array_equal(a, b) for a, b in zip(before, wl.host))
    wl.dev[2][11, 39] ^= 1
    assert wl.oracle_parity_all(threads=3)["result"] == "MISMATCH in windows 2"


@pytest.mark.parametrize("name", ["a2av", "a2av_sparse", "all_to_all", "combine"])
def test_exchange_parity_leg(name):
    """The exchanges' parity check on host stand-ins for the resident outputs
    (small windows stand in for the 16 x 24576 x 7168 ones): the oracle's own
    result passes, one changed element fails."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    wl = bench.make_workload(name, 1)
    wl.cfg = dict(wl.cfg, nranks=3, size=8, target_rows=12)
    wl.setup_host()
    c = wl.cfg
    n, tr, size = 3, 12, 8
    sc = [np.ascontiguousarray(x, dtype=np.int32) for x in wl.sc]
    tg = [np.full((tr, size), c["sentinel"], dtype=np.uint16) for _ in range(n)]
    rc = [np.zeros(n, dtype=np.int32) for _ in range(n)]
    if name == "all_to_all":
        oracle.all_to_all(wl.host, tg, tr, size, 2)
    else:
        oracle.all_to_all_v(wl.host, tg, sc, rc, tr, size, 2)
    wl.d_tg = [torch.from_numpy(t.view(np.int16).copy()) for t in tg]
    wl.d_rc = [torch.from_numpy(r.copy()) for r in rc]
    if name == "combine":
        outs = [o.copy() for o in wl.out_host]
        oracle.all_to_all_v_combine(tg, outs, rc, tr, size, oracle.ATOMIC_ADD, oracle.BF16)
        wl.d_out = [torch.from_numpy(o.view(np.int16).copy()) for o in outs]
    assert wl.oracle_parity(0)["result"] == "bit-exact"
    changed = wl.d_out if name == "combine" else wl.d_tg
    changed[1][tr - 1, size - 1] ^= 1
    assert wl.oracle_parity(0)["result"] == "MISMATCH in windows 1"


def test_windows_parity_helper():
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    want = [np.arange(40, dtype=np.uint16).reshape(5, 8) + r for r in range(3)]
    dev = [torch.from_numpy(np.vstack([w.view(np.int16), np.zeros((2, 8), np.int16)])) for w in want]
    assert bench._windows_parity(dev, want, 5, 7)["result"] == "bit-exact"
    dev[2][4, 7] += 1
    assert bench._windows_parity(dev, want, 5, 7)["result"] == "MISMATCH in windows 2"


def test_defaults_and_reference_line():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "ours" and a.workload == "treduce_16384x8192"
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--reference-seconds", "1",
                          "--workload", "treduce_small"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    # the same config dict as the GPU arm's line for this workload at N = 1
    assert line["config"] == bench.line_config(bench.make_workload("treduce_small"), 1)


def test_default_workload_is_the_largest_treduce_case():
    """The default step is the 8-rank [16384, 8192] TREDUCE: f32 Sum and the
    int32 Max variant, one launch each, (N + 1) * 4 bytes per valid element."""
    sys.path.insert(0, ROOT)
    import bench
    wl = bench.make_workload(bench.parse([]).workload)
    assert wl.launches_per_step() == 2
    assert [(p.storage, p.w.ops) for p in wl.parts] == [("f32", ["sum"]), ("i32", ["max"])]
    for p in wl.parts:
        w = p.w
        assert (w.nranks, w.rows, w.cols, w.ld, w.valid_rows, w.valid_cols) == (8, 16384, 8192, 8192, 16384, 8192)
    assert wl.bytes_per_launch() == 9 * 4 * 16384 * 8192
    assert wl.bytes_per_step() == 2 * wl.bytes_per_launch()
    cfg = bench.line_config(wl, 1)
    assert cfg["workload"] == "treduce_n8_16384x8192_f32sum_i32max" and cfg["parallelism"] == "single GPU"


def test_full_parity_leg_of_the_default_workload():
    """The default workload's parity check compares every element of both
    results with the oracle (row slices on threads): host stand-ins for the
    resident results pass when they are the oracle's, and one changed
    element in either part fails (rows divided by 512 stand in for the full
    case)."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    wl = bench.make_workload("treduce_16384x8192", rows_div=512)
    wl.setup_host()
    for p in wl.parts:
        w = p.w
        p.dst_init = np.zeros((w.rows, w.ld), dtype=p.host[0].dtype)
        want = p.dst_init.copy()
        op = {"sum": oracle.SUM, "max": oracle.MAX}[w.ops[0]]
        code = {"f32": oracle.F32, "i32": oracle.I32}[p.storage]
        assert oracle.treduce(p.host, want, w.valid_rows, w.valid_cols, w.ld, op, code) == 0
        p.dsts = [torch.from_numpy(want)]
    got = wl.oracle_parity_all(threads=5)
    assert got["result"] == "bit-exact" and got["rows"].startswith("all 32 of 32")
    d = wl.parts[1].dsts[0]
    d[31, 8191] += 1
    assert wl.oracle_parity_all(threads=3)["result"] == "i32 MISMATCH in max"


def test_threaded_oracle_sample_matches_one_call():
    """The all-cores CPU baseline splits rows over threads; its result equals
    one oracle call over the same rows, byte for byte."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    wl = bench.make_workload("treduce_small")
    wl.setup_host()
    w = wl.w
    rows = 37
    ref = np.empty((rows, w.ld), dtype=wl.host[0].dtype)
    nb, dt, got = wl.oracle_sample_threaded(rows, 5)
    for op in w.ops:
        oracle.treduce(wl.host, ref, rows, w.valid_cols, w.ld, {"sum": oracle.SUM, "max": oracle.MAX,
                                                                 "min": oracle.MIN}[op], oracle.F32)
    assert got.shape == ref.shape
    assert np.array_equal(got[:, :w.valid_cols].view(np.uint32), ref[:, :w.valid_cols].view(np.uint32))
    assert nb == (w.nranks + 1) * 4 * rows * w.valid_cols * len(w.ops)


def test_traffic_source_lists_exist():
    """Every kernel source a traffic record is keyed to exists, and the lists
    cover every device-code file of the library."""
    import glob
    sys.path.insert(0, ROOT)
    import bench
    listed = set(bench.REDUCE_SOURCES) | set(bench.MOVE_SOURCES)
    for rel in listed:
        assert os.path.exists(os.path.join(ROOT, rel)), rel
    csrc = os.path.join(ROOT, "tile_level_collective_gb300", "csrc")
    device = {os.path.relpath(f, ROOT) for f in glob.glob(os.path.join(csrc, "*"))
              if f.endswith((".cuh", ".h")) or os.path.basename(f).startswith(("reduce_", "movement"))}
    assert device <= listed, device - listed


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm's rank 0 alone times the oracle and
    prints the line; the other ranks exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "2", "--warmup", "1", "--reference-seconds", "1",
                          "--workload", "treduce_small"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == ""


def test_e2e_link_bound():
    """The e2e leg's bound: the slower direction of the host link sets the
    step time, the step's bytes over that time is the bound, whole job."""
    import bench

    class W:
        def h2d_bytes(self):
            return 8 * 10 ** 9

        def d2h_bytes(self):
            return 1 * 10 ** 9

        def bytes_per_step(self):
            return 9 * 10 ** 9

    b = bench.e2e_link_bound(W(), (200.0, 100.0), 1)
    assert b["h2d_gbs"] == 200.0 and b["d2h_gbs"] == 100.0
    assert b["bound_gbs"] == pytest.approx(9e9 / 0.04 / 1e9)        # upload: 40 ms against 10 ms down
    assert b["h2d_gbs_during_e2e"] is None
    b = bench.e2e_link_bound(W(), (200.0, 10.0), 2, during=150.04)
    assert b["bound_gbs"] == pytest.approx(2 * 9e9 / 0.1 / 1e9)      # download: 100 ms
    assert b["h2d_gbs_during_e2e"] == 150.0
