"""Multi-rank host logic of bench.py on CPU: two gloo ranks (replicas) meet at
the barrier and agree on the max-over-ranks time, as the timed region does."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        ms = d.max(10.0 * rank + 1.0)   # each rank's own "elapsed time"
        d.barrier()
        q.put((d.rank, d.world, ms))
    finally:
        d.close()


def test_two_gloo_ranks_take_the_max():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert got == [(0, 2, 11.0), (1, 2, 11.0)]
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(None, 3.5) == 3.5
    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", "1"))
    if d.world == 1:
        d.barrier()
        assert d.max(2.0) == 2.0


def test_persistent_launch_count():
    """bench.py's roofline divides by the persistent kernel's launches only:
    a group with m >= 2 items adds a preparing launch to the full count, and
    an item with k == 0 a small launch of its own."""
    import ctypes

    sys.path.insert(0, ROOT)
    import bench
    import packed_bit_gemv_tern_b300 as tern
    from packed_bit_gemv_tern_b300 import build
    build.build()
    tern.load()
    w = tern.CMatrix(4096, 4096, 0x1000, 0x2000, None)
    w0 = tern.CMatrix(8, 0, 0x1000, 0x2000, None)
    for m, n, k_zero, total, main in ((1, 100, 0, 1, 1), (7, 8, 0, 2, 1), (7, 200, 0, 4, 2), (2, 1, 0, 2, 1),
                                      (1, 3, 2, 3, 1), (7, 3, 2, 4, 1)):
        arr = (tern.CBatchItem * n)()
        for i in range(n):
            arr[i].w, arr[i].x, arr[i].y, arr[i].m = ctypes.addressof(w), 0x3000, 0x4000, m
        for i in range(1, 1 + k_zero):  # items with k == 0 beside the real ones
            arr[i].w = ctypes.addressof(w0)
        assert tern.tern_gemm_batched_launches(arr) == total
        assert bench.persistent_launches(arr) == main
        assert [it.m for it in arr] == [m] * n  # the caller's array is untouched


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference (the oracle on the host cores) prints the
    contract's JSON line with the oracle described as its own baseline."""
    import json
    import subprocess

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--workload", "c0"], capture_output=True, text=True, timeout=300,
                         env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_step_spread_helpers():
    """The per-call spread: nearest-rank percentiles, and a failure inside the
    spread pass (here: no GPU) is reported in the line, never raised."""
    sys.path.insert(0, ROOT)
    import bench
    st = bench.spread_stats([float(v) for v in range(101, 0, -1)])  # 1..101 in any order
    assert (st["steps"], st["us_per_call_p10"], st["us_per_call_median"], st["us_per_call_p90"]) == (101, 11.0, 51.0, 91.0)
    assert bench.spread_stats([2.5])["us_per_call_median"] == 2.5

    class NoGraph:
        def replay(self):
            raise RuntimeError("no graph")

    out = bench.step_spread(NoGraph(), None, 3, 1)
    assert set(out) == {"error"}
