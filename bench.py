#!/usr/bin/env python3
"""Benchmark of the ternary packed-weight GEMV on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c1] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Metric: packed-weight GB/s at M=1 (and
microseconds per call), as a fraction of the measured HBM peak.

Workloads (seeded synthetic inputs, shapes of the Neutrino-1 8B linears):
  c0  M=1 GEMV 1024x4096            c1  M=1 GEMV 4096x4096 (default)
  c2  M=1 down 4096x12288 + fused gate/up 2x12288x4096 (SiLU(g)*u)
  c3  M=7 gate/up (fused) + down    c4  36-layer sweep, 252 linears per step

One step is one pass over the workload's calls.  c0-c3 rotate over distinct
device buffers holding more than three times the 126 MB L2 of packed weights,
so every call streams from HBM; the calls of one step are captured once in a
CUDA graph and replayed.  ``--impl reference`` times the fp64 CPU oracle on
the host cores instead (a deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed-weight GB/s and µs/call at M=1 (fraction of B300 HBM peak)"
FALLBACK_HBM_GBS = 6400.0
NOMINAL_HBM_GBS = 8000.0
ROTATE_MB_DEFAULT = 400  # c0-c3: MiB of distinct packed weights per step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--workload", default="c1", choices=["c0", "c1", "c2", "c3", "c4", "head"],
                    help="head: the int8 output head alone (151,936 x 4,096, m = 1, fused argmax)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--rotate-mb", type=int, default=ROTATE_MB_DEFAULT,
                    help="c0-c3: MiB of distinct packed weights one step streams (keep above the 126 MB L2)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the single-call, ordered-sweep and output-head measurements")
    ap.add_argument("--api", default="batched", choices=["batched", "single"],
                    help="batched: one persistent tern_gemm_batched launch per step; single: one launch per call")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: each rank runs its own independent batch)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        return reduce_max(self.pg, v)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def reduce_max(dist, v: float) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return v
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# ncu traffic summary (per launch), valid only while the kernel source is unchanged
# ---------------------------------------------------------------------------
def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "packed_bit_gemv_tern_b300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_digest") != kernel_source_digest():
        return None, None
    return e.get("dram_bytes_per_launch"), e.get("kernel")


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------
def step_spread(graph, stream, n: int, ncalls: int) -> dict:
    """Spread of the per-call time: a second pass of n steps after the timed
    region, each step between its own CUDA events (so consecutive steps do not
    overlap here, unlike in the timed region); p10, median and p90 of the step
    time divided by the calls per step.  Never fails the bench line."""
    try:
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                a.record(stream)
                graph.replay()
                b.record(stream)
        stream.synchronize()
        out = spread_stats([1e3 * a.elapsed_time(b) / ncalls for a, b in evs])
        out["how"] = "each step between its own CUDA events, after the timed region"
        return out
    except Exception as e:  # the spread is informative only
        return {"error": f"{type(e).__name__}: {e}"}


def spread_stats(us_per_call) -> dict:
    """p10, median and p90 (nearest rank) of per-call times in µs."""
    per = sorted(us_per_call)

    def pct(q):
        return round(per[min(len(per) - 1, int(q * (len(per) - 1) + 0.5))], 4)

    return {"steps": len(per), "us_per_call_p10": pct(0.1), "us_per_call_median": pct(0.5),
            "us_per_call_p90": pct(0.9)}


def _graph_ms(fn, stream, reps: int, warm: int = 3) -> float:
    """Mean ms of one replay of a CUDA graph of fn(), after an eager pass and
    warm-up replays, between CUDA events on the launching stream."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def extras(args, dev, stream, wl, peak):
    """More measurements on rank 0, each never failing the bench line:
    single_call (c1 as back-to-back tern_gemv launches in one graph, one
    launch per call), ordered_sweep (the 36-layer decode sweep as 4 launch
    groups per layer in dependency order, 144 tern_gemm_batched calls per
    token), base3 (the 1.6-bit base-3 format on c1's rows) and lm_head (the
    151,936 x 4,096 int8 output head with the fused argmax, m = 1)."""
    import torch

    import packed_bit_gemv_tern_b300 as tern
    from packed_bit_gemv_tern_b300 import synth, workloads
    out = {}
    try:
        wl1 = wl if args.workload == "c1" else workloads.build("c1", device=dev, rotate_bytes=400 * workloads.MiB)
        ms = _graph_ms(lambda: workloads.run_calls(wl1.calls, stream), stream, reps=100)
        n = len(wl1.calls)
        ach = wl1.algorithmic_bytes / (ms * 1e-3) / 1e9
        out["single_call"] = {"workload": f"c1 as {n} back-to-back tern_gemv launches per graph replay",
                              "us_per_call": round(1e3 * ms / n, 3), "gbs": round(ach, 2), "frac": round(ach / peak, 4)}
    except Exception as e:
        out["single_call"] = {"error": f"{type(e).__name__}: {e}"}
    try:
        groups, packed, keep = workloads.layer_sweep(dev)
        ms = _graph_ms(lambda: [tern.tern_gemm_batched(g, stream) for g in groups], stream, reps=20)
        gbs = packed / (ms * 1e-3) / 1e9
        out["ordered_sweep"] = {"workload": f"{synth.LAYERS} layers x (q|k|v, o, gate/up SwiGLU, down) in order, "
                                            "4 layers of distinct weights reused cyclically (184 MB)",
                                "groups_per_token": len(groups), "us_per_token": round(1e3 * ms, 2),
                                "gbs_packed": round(gbs, 2), "frac": round(gbs / peak, 4)}
        del keep
    except Exception as e:
        out["ordered_sweep"] = {"error": f"{type(e).__name__}: {e}"}
    try:
        # base-3 format: one tern5_gemv over 409,600 x 4,160 (c1's 100 x 4096
        # rows, K padded to a multiple of 80), 341 MB of codes drawn uniformly
        # over the valid bytes
        rng = np.random.default_rng(555)
        rows5, k5 = 409600, 4160
        c5 = torch.from_numpy(rng.integers(0, 243, (rows5, k5 // 5), dtype=np.uint8)).to(dev)
        s5 = torch.from_numpy(synth.scales(rng, rows5)).to(dev)
        w5 = tern.Tern5Matrix(c5, s5, k5)
        x5 = torch.from_numpy(synth.activations(rng, 1, k5).view(np.int16)).to(dev).view(torch.bfloat16)
        y5 = torch.empty((1, rows5), dtype=torch.float32, device=dev)
        ms = _graph_ms(lambda: tern.tern5_gemm(w5, x5, 1, y5, stream=stream), stream, reps=20)
        gb = w5.packed_bytes / (ms * 1e-3) / 1e9
        out["base3"] = {"workload": "base-3 codes (5 weights a byte), 409,600 x 4,160 at m = 1, one tern5_gemm",
                        "us_per_call": round(1e3 * ms, 2), "gbs_codes": round(gb, 2), "frac": round(gb / peak, 4),
                        "gweights_per_s": round(rows5 * k5 / (ms * 1e-3) / 1e9, 1),
                        "two_bit_equivalent_gbs": round(rows5 * k5 / 4 / (ms * 1e-3) / 1e9, 2)}
        del c5, w5
    except Exception as e:
        out["base3"] = {"error": f"{type(e).__name__}: {e}"}
    head = None
    try:
        rng = np.random.default_rng(777)
        rows, k = 151936, 4096
        w = rng.integers(-128, 128, (rows, k), dtype=np.int8)
        sc = rng.uniform(0.5e-3, 2e-3, rows).astype(np.float32)
        dw = tern.I8Matrix.from_host(w, sc, device=dev)
        del w
        xb = synth.activations(rng, 1, k)
        x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        logits = torch.empty((1, rows), dtype=torch.float32, device=dev)
        am = torch.empty((1,), dtype=torch.int32, device=dev)
        ms = _graph_ms(lambda: tern.tern_lmhead_argmax(dw, x, 1, logits, am, stream=stream), stream, reps=50)
        alg = rows * k + 8 * rows + 2 * k  # int8 weights, scales, logits, x
        ach = alg / (ms * 1e-3) / 1e9
        consistent = int(am.item()) == int(torch.argmax(logits[0]).item())
        head = {"workload": "int8 output head 151,936 x 4,096 (622 MB) + per-row scale, m = 1, fused argmax",
                "us_per_call": round(1e3 * ms, 2), "gbs": round(ach, 2), "frac": round(ach / peak, 4),
                "launches_per_call": 3, "argmax_matches_logits": consistent}
    except Exception as e:
        head = {"error": f"{type(e).__name__}: {e}"}
    return out, head


def persistent_launches(batch) -> int:
    """Launches of the persistent batched kernel for a batch: the launch count
    of the same items with m = 1, less the small launch of each item with
    rows > 0 and k == 0.  The launch groups do not depend on m; a group that
    holds items with m >= 2 adds one short activation-preparing launch, which
    the full count includes."""
    import ctypes

    import packed_bit_gemv_tern_b300 as tern
    arr = (tern.CBatchItem * len(batch))()
    ctypes.memmove(arr, batch, ctypes.sizeof(arr))
    k_zero = 0
    for it in arr:
        it.m = 1
        w = tern.CMatrix.from_address(it.w)
        k_zero += 1 if w.rows > 0 and w.k == 0 else 0
    return tern.tern_gemm_batched_launches(arr) - k_zero


def oracle_sample_rate(wl, budget_s: float, threads: int):
    """Time the fp64 oracle over a bounded sample of the workload's calls.

    Returns (packed GB/s, packed bytes processed, seconds, description).
    The sample walks the calls in order, each call over a slice of its rows,
    until ``budget_s`` of wall time has been spent.
    """
    import oracle
    done_bytes, t0, ncalls, nrows = 0, time.perf_counter(), 0, 0
    packed = getattr(wl, "_oracle_packed", None)
    if packed is None:
        packed = {}
        for h in wl.host:
            for lin in (h["lin"], h.get("up")):
                if lin is not None and id(lin) not in packed:
                    packed[id(lin)] = oracle.pack(lin.t)
        wl._oracle_packed = packed
    t0 = time.perf_counter()
    while True:
        for c, h in zip(wl.calls, wl.host):
            lin = h["lin"]
            rows = min(lin.rows, max(threads * 16, 256))
            if "up" in h:
                _oracle_swiglu_rows(oracle, packed, lin, h, rows, threads)
                done_bytes += 2 * rows * lin.k // 4
            else:
                _oracle_gemm_rows(oracle, packed[id(lin)], lin, h["x_bits"], rows, threads)
                done_bytes += rows * lin.k // 4
            ncalls += 1
            nrows += rows
            if time.perf_counter() - t0 >= budget_s:
                dt = time.perf_counter() - t0
                desc = (f"{ncalls} calls of workload {wl.name}, first {nrows // max(ncalls, 1)} rows of each "
                        f"(all K columns), {done_bytes / 1e6:.1f} MB of packed weights")
                return done_bytes / dt / 1e9, done_bytes, dt, desc


def _oracle_gemm_rows(oracle, codes, lin, x_bits, rows, threads):
    oracle.gemm(codes[:rows], lin.scale[:rows], lin.k, x_bits, threads=threads)


def _oracle_swiglu_rows(oracle, packed, lin, h, r, threads):
    oracle.swiglu(packed[id(lin)][:r], lin.scale[:r], packed[id(h["up"])][:r], h["up"].scale[:r], lin.k,
                  h["x_bits"], threads=threads)


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args, dist: Dist):
    """Reference arm: the fp64 CPU oracle as it stands, on the host cores."""
    if dist.rank != 0:
        return 0
    from packed_bit_gemv_tern_b300 import synth, workloads  # noqa: F401
    wl = _host_only_workload(args.workload)
    threads = os.cpu_count() or 1
    per_step_budget = max(0.002, min(1.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_rate(wl, per_step_budget, threads)
    tot_bytes, tot_s = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        _, b, dt, desc = oracle_sample_rate(wl, per_step_budget, threads)
        tot_bytes += b
        tot_s += dt
    gbs = tot_bytes / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / max(1, args.steps), 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {wl.desc}"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step ~{per_step_budget:.3f} s: {desc}"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class _HostWL:
    def __init__(self, name, desc):
        self.name, self.desc, self.calls, self.host = name, desc, [], []


def _host_only_workload(name):
    """Host copies of one unit of a workload (no GPU), for the oracle arm."""
    from packed_bit_gemv_tern_b300 import synth
    spec = synth.WORKLOADS[name]
    rng = np.random.default_rng(spec["seed"])
    wl = _HostWL(name, spec["desc"])
    if name in ("c0", "c1"):
        rows = 1024 if name == "c0" else 4096
        lin = synth.linear(rng, rows, 4096)
        wl.calls.append(None)
        wl.host.append(dict(lin=lin, x_bits=synth.activations(rng, 1, 4096)))
    elif name in ("c2", "c3"):
        m = 1 if name == "c2" else 7
        pz = 0.71 if name == "c2" else synth.P_ZERO
        gate = synth.linear(rng, 12288, 4096, p_zero=pz)
        up = synth.linear(rng, 12288, 4096, p_zero=pz)
        down = synth.linear(rng, 4096, 12288, p_zero=pz)
        wl.calls += [None, None]
        wl.host.append(dict(lin=gate, up=up, x_bits=synth.activations(rng, m, 4096)))
        wl.host.append(dict(lin=down, x_bits=synth.activations(rng, m, 12288)))
    else:
        for lname, rows, k in synth.LAYER_LINEARS:
            lin = synth.linear(rng, rows, k, p_zero=synth.sweep_zero_fraction(0, lname))
            wl.calls.append(None)
            wl.host.append(dict(lin=lin, x_bits=synth.activations(rng, 1, k)))
    return wl


def run_head(args, dist: Dist):
    """--workload head: the int8 output head with the fused argmax as the
    timed step (one tern_lmhead_argmax call; 622 MB of weights, more than the
    L2), the same timing protocol as the ternary workloads."""
    import torch

    import packed_bit_gemv_tern_b300 as tern
    from packed_bit_gemv_tern_b300 import synth
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    tern.load()
    stream = torch.cuda.Stream(device=dev)
    rng = np.random.default_rng(777 + 1000 * dist.rank)
    rows, k = 151936, 4096
    w = rng.integers(-128, 128, (rows, k), dtype=np.int8)
    sc = rng.uniform(0.5e-3, 2e-3, rows).astype(np.float32)
    dw = tern.I8Matrix.from_host(w, sc, device=dev)
    del w
    x = torch.from_numpy(synth.activations(rng, 1, k).view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.empty((1, rows), dtype=torch.float32, device=dev)
    am = torch.empty((1,), dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        tern.tern_lmhead_argmax(dw, x, 1, logits, am, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        tern.tern_lmhead_argmax(dw, x, 1, logits, am, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    dist.barrier()
    clk = clocks.stop()
    ms = dist.max(ev0.elapsed_time(ev1))
    if tern.tern_last_device_error(stream) != tern.TERN_OK:
        raise SystemExit("device error during the timed region")
    step_ms = ms / args.steps
    alg = rows * k + 8 * rows + 2 * k
    ach = alg / (step_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    line = {
        "metric": "int8 output-head GB/s and µs/call at M=1 (fraction of B300 HBM peak)",
        "value": round(dist.world * rows * k / (step_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x, int8 w, fp32 acc", "data": "synthetic (seeded)",
        "config": {"workload": "head: int8 output head 151,936 x 4,096 + per-row scale, m = 1, fused argmax",
                   "us_per_call": round(1e3 * step_ms, 3), "graph": "one CUDA graph per call, replayed",
                   "l2": "622 MB of weights per call, more than the L2",
                   "argmax_matches_logits": int(am.item()) == int(torch.argmax(logits[0]).item())},
        "roofline": {"bound": "hbm", "achieved": round(ach, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(ach / peak, 4), "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_launch": alg, "duration": "CUDA-event time per call (3 launches, the head kernel dominant)"},
        "clocks": clk, "gpu_launches": 3 * args.steps, "e2e": None, "cpu_baseline": None,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_ours(args, dist: Dist):
    import torch

    import packed_bit_gemv_tern_b300 as tern
    from packed_bit_gemv_tern_b300 import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    tern.load()
    wl = workloads.build(args.workload, device=dev, seed_offset=dist.rank, rotate_bytes=args.rotate_mb * workloads.MiB)
    ncalls = len(wl.calls)
    stream = torch.cuda.Stream(device=dev)

    batch = workloads.batch_of(wl.calls) if args.api == "batched" else None
    launches_per_step = tern.tern_gemm_batched_launches(batch) if batch is not None else ncalls
    # the dominant kernel's launches: the persistent kernel's (batched), or every call's
    main_launches = persistent_launches(batch) if batch is not None else ncalls
    prep_launches = launches_per_step - main_launches

    def step_fn():
        if batch is not None:
            workloads.run_batched(batch, stream)
        else:
            workloads.run_calls(wl.calls, stream)

    # one eager pass (sets kernel attributes), then capture the step in a graph
    with torch.cuda.stream(stream):
        step_fn()
    stream.synchronize()
    if tern.tern_last_device_error(stream) != tern.TERN_OK:
        raise SystemExit("device error after the first pass")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_fn()
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[dist.local]))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max = dist.max(ms)
    if tern.tern_last_device_error(stream) != tern.TERN_OK:
        raise SystemExit("device error during the timed region")
    spread = step_spread(graph, stream, min(args.steps, 200), ncalls)

    packed = wl.packed_bytes
    alg = wl.algorithmic_bytes
    step_ms = ms_max / args.steps
    value = dist.world * packed * args.steps / (ms_max * 1e-3) / 1e9
    us_per_call = 1e3 * step_ms / ncalls
    # the step's time over the dominant kernel's launches: with a preparing
    # launch in the step, its (mostly overlapped) time is charged to them
    per_launch_s = ms * 1e-3 / (args.steps * main_launches)
    achieved = (alg / main_launches) / per_launch_s / 1e9
    peak, peak_kind = peaks()
    # The recorded DRAM traffic is per launch of the batched kernel at the
    # default step size; another launch shape has no recorded figure.
    traffic, traffic_kernel = None, None
    if batch is not None and args.rotate_mb == ROTATE_MB_DEFAULT:
        traffic, traffic_kernel = ncu_traffic(args.workload)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, stream, dist, batch)

    more, head = ({}, None)
    if dist.rank == 0 and not args.no_extras:
        more, head = extras(args, dev, stream, wl, peak)

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        # median of three samples on every host core, and one on a single core
        threads = os.cpu_count() or 1
        runs = [oracle_sample_rate(wl, max(1.0, 4.0 / threads), threads) for _ in range(3)]
        gbs = statistics.median(r[0] for r in runs)
        one = oracle_sample_rate(wl, 3.0, 1)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": runs[0][3], "runs": [round(r[0], 4) for r in runs], "stat": "median of 3",
               "value_1core": round(one[0], 4), "sample_1core": one[3]}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x, 2-bit ternary w, fp32 acc",
        "data": "synthetic (seeded; code mix of the model page)",
        "config": {"workload": f"{args.workload}: {wl.desc}", "calls_per_step": ncalls,
                   "distinct_draws": wl.distinct, "packed_bytes_per_step": packed,
                   "algorithmic_bytes_per_step": alg, "us_per_call": round(us_per_call, 4),
                   "l2": "inputs larger than L2: each step streams %.0f MB of distinct buffers" % (packed / 1e6),
                   "graph": "one CUDA graph per step, replayed", "parallelism": f"replicas x{dist.world}",
                   "gpu": torch.cuda.get_device_name(dev), "spread": spread,
                   "single_call": more.get("single_call"), "ordered_sweep": more.get("ordered_sweep"),
                   "base3": more.get("base3"),
                   "api": (f"tern_gemm_batched: {main_launches} persistent launch(es) per step"
                           + (f" and {prep_launches} activation-preparing launch(es)" if prep_launches else "")
                           if args.api == "batched" else "one tern_* launch per call")},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "traffic_kernel": traffic_kernel,
                     "bytes_per_launch": alg // main_launches,
                     "duration": ("CUDA-event step time / persistent launches per step"
                                  + (" (includes the activation-preparing launch)" if prep_launches else ""))},
        "clocks": clk,
        "lm_head": head,
        "gpu_launches": args.steps * launches_per_step,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_e2e(args, wl, stream, dist: Dist, batch=None):
    """Same metric through the public API with host buffers: every step copies
    all of its activations from pinned host memory, runs the calls (one
    batched launch, or one launch per call), and copies every output back;
    weights are the resident model.  With the batched API two device buffer
    sets alternate, and the copies run on a second stream, so step i+1's
    upload and step i-1's download overlap step i's kernel (a serving
    pipeline); every step's own copies are inside the timed region."""
    import torch

    from packed_bit_gemv_tern_b300 import workloads

    hx = wl.x_flat.cpu().pin_memory()
    h2d = hx.numel() * hx.element_size()
    d2h = wl.y_flat.numel() * wl.y_flat.element_size()

    if batch is None:  # one launch per call: serial copy, run, copy
        hy = torch.empty(wl.y_flat.shape, dtype=torch.float32).pin_memory()

        def step():
            wl.x_flat.copy_(hx, non_blocking=True)
            workloads.run_calls(wl.calls, stream)
            hy.copy_(wl.y_flat, non_blocking=True)
            stream.synchronize()

        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
            dist.barrier()
            t0 = time.perf_counter()
            for _ in range(args.e2e_steps):
                step()
            dt = time.perf_counter() - t0
        n_steps = args.e2e_steps
        how = "per step: one pinned H2D copy of all x, the tern ABI calls, one D2H copy of all y; serial; host-timed"
    else:
        x1, y1, batch1, _items1 = workloads.io_copy(wl)
        xs, ys, batches = (wl.x_flat, x1), (wl.y_flat, y1), (batch, batch1)
        hys = [torch.empty(wl.y_flat.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
        dev = wl.x_flat.device
        ups, downs = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        for bt in batches:  # first calls (per-device set-up, tensor maps) outside capture
            workloads.run_batched(bt, stream)
        stream.synchronize()

        # A serving loop's pipeline of `seg` steps, captured once as a CUDA
        # graph: step i uploads into buffer set i % 2 on `ups` (after that
        # set's previous download), runs the batched call on `stream`, and
        # downloads on `downs`, so step i's kernel overlaps step i+1's upload
        # and step i-1's download.  Replaying the graph replays every step's
        # copies; only the host's per-call work is paid once.
        seg = min(args.e2e_steps, 10)
        reps = -(-args.e2e_steps // seg)
        n_steps = reps * seg
        ev = [[torch.cuda.Event() for _ in range(seg)] for _ in range(3)]
        up, done, freed = ev
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            start = torch.cuda.Event()
            start.record(stream)
            ups.wait_event(start)
            downs.wait_event(start)
            for i in range(seg):
                b = i & 1
                if i >= 2:
                    ups.wait_event(freed[i - 2])
                with torch.cuda.stream(ups):
                    xs[b].copy_(hx, non_blocking=True)
                up[i].record(ups)
                stream.wait_event(up[i])
                workloads.run_batched(batches[b], stream)
                done[i].record(stream)
                downs.wait_event(done[i])
                with torch.cuda.stream(downs):
                    hys[b].copy_(ys[b], non_blocking=True)
                freed[i].record(downs)
            stream.wait_event(freed[seg - 1])

        with torch.cuda.stream(stream):
            for _ in range(2):
                gr.replay()
            stream.synchronize()
            dist.barrier()
            t0 = time.perf_counter()
            for _ in range(reps):
                gr.replay()
            stream.synchronize()
            dt = time.perf_counter() - t0
        # the copied-back outputs are the device path's, bit for bit
        workloads.run_batched(batch, stream)
        stream.synchronize()
        ref = wl.y_flat.cpu()
        for h in hys:
            if not torch.equal(h, ref):
                raise RuntimeError("e2e outputs differ from the device path's")
        how = (f"per step: one pinned H2D copy of all x, the tern_gemm_batched call, one D2H copy of all y; two "
               f"device buffer sets, uploads and downloads on their own streams overlapping the neighbouring "
               f"steps' kernels; {seg}-step segments of that pipeline captured once in a CUDA graph and replayed "
               f"{reps} times; host-timed from the first replay to the last download; copied-back outputs "
               f"checked bitwise against the device path")
    dt = dist.max(dt)
    return {"value": round(dist.world * wl.packed_bytes * n_steps / dt / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_steps, "how": how}


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            if args.workload == "head":
                print(json.dumps({"impl": "reference", "unavailable": "no oracle arm for the head workload"}))
                return 0
            return run_reference(args, dist)
        if args.workload == "head":
            return run_head(args, dist)
        return run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
