"""Benchmark of the streaming-attention hot path on one GB300 (or N replicas).

One step = one pass of the whole path:
  1. kv_stream_insert     on the scale-up workload (36 layer caches,
                          prefix 512 + 6 views x 8 frames x 256 tokens),
  2. stream_attn_prefill  of its 1536 new-frame queries x 32 heads per layer,
  3. stream_attn_verify   of a 9-token block on the Alpamayo-shaped cache
                          (prefix 256 + 4 x 4 x 180, 16 tail tokens), batch 64,
                          with the greedy accept-length reduction.
After the step loop, kv_stream_insert alone is timed on rotating input sets
that do not fit L2, and the one-kernel stream_attn_prefill_insert (steps 1
and 2 fused) is timed beside it.

The reported value is the prefill attention's algorithmic TFLOP/s over the
whole step (unmasked query-key pairs only, 4*d FLOP each); the verify
kernel's HBM GB/s and the insert's GB/s are reported beside it.  Inputs stay
resident in HBM; the caches (about 2.8 GB) are far larger than L2, so
consecutive steps cannot hit in L2.

The end-to-end figure runs the same step from pinned host buffers: every
step's inputs are copied up and its outputs copied down inside the timed
region.  Step i+1's upload and step i's download run on two copy streams
while step i's kernels run; the fully serial form is reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from streaming_kv_cache_gb300 import synth  # noqa: E402

METRIC = "stream-prefill attn TFLOP/s (% bf16 peak); verify-step HBM GB/s (% peak)"
PREFILL_W = synth.WORKLOADS["scaleup_36L"]
VERIFY_W = synth.WORKLOADS["alpamayo_verify"]          # batch 64
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# algorithmic work

def prefill_pairs(w) -> int:
    """Visible (query, key) pairs per query head and cache: new-frame token
    (v, t) sees every key with logical index <= P + v*F*T + (F-1)*T + t."""
    tot = 0
    for v in range(w.V):
        base = w.P + v * w.F * w.T + (w.F - 1) * w.T + 1
        tot += w.T * base + w.T * (w.T - 1) // 2
    return tot


def prefill_flop(w) -> float:
    return 4.0 * w.d * w.Hq * w.C * prefill_pairs(w)


def window_flop(w) -> float:
    """Every window token a query: token i sees keys 0..i."""
    n = w.n_window
    return 4.0 * w.d * w.Hq * w.C * n * (n + 1) / 2


def tail_flop(w, n: int, tail_len: int = 0) -> float:
    """n tail tokens after tail_len tail rows: token j sees the window, the
    tail_len rows and tokens 0..j."""
    return 4.0 * w.d * w.Hq * w.C * (n * (w.n_window + tail_len) + n * (n + 1) / 2)


def verify_bytes(w) -> float:
    """Per launch: K and V of every visible key once per (cache, kv head),
    the block's Q in and O out, the block K/V read and written to the tail."""
    keys = w.P + w.V * w.F * w.T + w.tail_len + w.blk
    kv = 2.0 * keys * w.d * 2 * w.Hkv
    q_o = 2.0 * w.blk * w.Hq * w.d * 2
    blk_kv = 2.0 * 2 * w.blk * w.Hkv * w.d * 2
    return w.C * (kv + q_o + blk_kv)


def insert_bytes(w) -> float:
    return 2.0 * 2 * w.C * w.V * w.T * w.Hkv * w.d * 2   # K and V, read + write


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def traffic_for(kernel_file: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel_file)
    if not ent:
        return None
    return ent["bytes_per_launch"] if ent.get("source_sha") == source_sha(kernel_file) else None


def source_sha(kernel_file: str) -> str:
    """Hash of a kernel's source file and every header of the library (the
    kernels include them): a change to any of them voids recorded counters."""
    csrc = os.path.join(ROOT, "streaming_kv_cache_gb300", "csrc")
    h = hashlib.sha256(open(os.path.join(csrc, kernel_file), "rb").read())
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    """nvidia-smi every 50 ms around the timed region; summary() keeps the
    samples whose timestamps fall between mark_start() and mark_stop()
    (the board's power reading is a trailing average, so it is not kept)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_stop(self):
        self.t1 = datetime.datetime.now()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                if self.t0 is not None and self.t1 is not None and not (self.t0 <= ts <= self.t1):
                    continue
                sm.append(float(f[2]))
                mx = max(mx, float(f[3]))
            except ValueError:
                continue
            for n, val in zip(names, f[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CPU oracle as a bounded-sample baseline

def oracle_sample(seconds: float = 12.0):
    """Time the fp64 oracle on a bounded sample of the prefill workload: one
    layer cache, a spread of new-frame query rows (all 32 heads, full
    recompute over the 12,800-key window).  Returns (TFLOP/s, cores, text)."""
    from oracle import skv_oracle as O
    w = PREFILL_W.with_(C=1)
    pk, pv = synth.prefix_kv(w, "cpu")
    win = O.StreamWindow(w.P, w.V, w.F, w.T, w.Hkv, w.d, pk[0], pv[0])
    for i in range(w.F + 1):
        k, v = synth.frame_kv(w, i, "cpu")
        win.insert(k[0], v[0])
    q = synth.frame_q(w, w.F, "cpu")[0]

    def flop(rows):
        return sum(4.0 * w.d * w.Hq * (win.new_frame_index(int(j) // w.T, int(j) % w.T) + 1)
                   for j in rows)

    n, spent, done_flop, calls, n_rows = 8, 0.0, 0.0, 0, 0
    rng = np.random.default_rng(0)
    while spent < seconds and calls < 64:
        rows = np.sort(rng.choice(w.n_new, size=min(n, w.n_new), replace=False))
        t0 = time.perf_counter()
        O.stream_prefill(win, q, w.theta, w.sm_scale, rows=rows)
        dt = time.perf_counter() - t0
        spent += dt
        done_flop += flop(rows)
        calls += 1
        n_rows += len(rows)
        n = min(w.n_new, n * 2) if dt < seconds / 8 else n
    affinity = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    cores = blas_threads() or affinity
    text = ("fp64 NumPy oracle, %d prefill calls on one layer cache of the scale-up workload "
            "(%d query rows x %d heads in total, full recompute over the %d-key window), "
            "%.1f s, %d BLAS threads on %d host cores"
            % (calls, n_rows, w.Hq, w.n_window, spent, cores, affinity))
    return done_flop / spent / 1e12, cores, text, spent


def blas_threads():
    """Threads of the BLAS NumPy calls into, where threadpoolctl can tell
    (None otherwise)."""
    try:
        from threadpoolctl import threadpool_info
    except ImportError:
        return None
    n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
    return max(n) if n and max(n) > 0 else None


# ---------------------------------------------------------------------------

def max_over_ranks(dist, values, device):
    """The largest of each timing over all ranks (each rank's own values
    when there is no process group): the job is as slow as its slowest
    replica."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world: int, work_per_step: float, steps: int, ms: float, scale: float = 1e12) -> float:
    """Whole-job throughput: every rank does work_per_step per step (weak
    scaling), so the job does world * work_per_step * steps in ms (the
    max over ranks)."""
    return world * work_per_step * steps / (ms * 1e-3) / scale


def check_pipelined(torch, pipelined, step, dev_in, dev_out, h_in, h_out, heads):
    """Untimed self-check of the overlapped end-to-end loop.  Four steps whose
    host inputs alternate A B B A (the queries differ, so both double-buffer
    slots change content between uses) run first one at a time on the
    compute stream, then, from the same ring heads, through the overlapped
    loop; every step's host outputs must be bit-identical.  (The prefill
    streams keys in physical ring order, so its summation order follows the
    ring heads; restoring them makes the two runs the same computation.)  A
    copy that overtook the kernels using its buffer shows up as a mismatch.
    Raises on a mismatch; returns a one-line description."""
    q_b = list(h_in)
    for j in (2, 3):                       # the prefill queries and the verify block queries
        q_b[j] = (h_in[j].float() * -0.5).to(h_in[j].dtype).pin_memory()
    variants = [h_in, q_b]
    order = [0, 1, 1, 0]
    saved = [t.clone() for t in heads]
    want = []
    for v in order:
        for d, h in zip(dev_in, variants[v]):
            d.copy_(h)
        step(False)
        torch.cuda.synchronize()
        want.append([d.to("cpu", copy=True) for d in dev_out])
    for t, c in zip(heads, saved):
        t.copy_(c)
    got = [[torch.empty_like(t).pin_memory() for t in h_out] for _ in order]
    pipelined(len(order), host_in=lambda i: variants[order[i]], host_out=lambda i: got[i])
    torch.cuda.synchronize()
    for i in range(len(order)):
        for name, a, b in zip(("prefill out", "verify out", "accept_len", "next_token"), got[i], want[i]):
            if not torch.equal(a, b):
                raise RuntimeError("overlapped end-to-end step %d: %s differs from the same step "
                                   "run alone" % (i, name))
    if torch.equal(want[0][0], want[1][0]):
        raise RuntimeError("end-to-end self-check: the two input variants gave the same output")
    for d, h in zip(dev_in, h_in):         # leave the timed inputs as they were
        d.copy_(h)
    return ("4 overlapped steps, inputs A B B A, from the same ring heads: host outputs "
            "bit-identical to the same steps run one at a time")


def step_config() -> dict:
    """The workload of one bench step, as both arms report it."""
    return {"workload": "scaleup_36L step (insert + prefill, 36 layer caches, P=512, "
                        "6 views x 8 frames x 256 tokens, 1536 queries, Hq=32/Hkv=8/d=128) "
                        "+ alpamayo_verify (B=64, 9-token block, 16 tail tokens)",
            "l2": "inputs larger than L2 (caches 2.8 GB), no flush",
            "prefill_gflop_per_step": prefill_flop(PREFILL_W) / 1e9,
            "verify_mb_per_step": verify_bytes(VERIFY_W) / 1e6,
            "insert_mb_per_step": insert_bytes(PREFILL_W) / 1e6}


def emit(obj):
    print(json.dumps(obj), flush=True)


def run_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(seconds=min(per_step, 3.0))
    vals, secs, cores, text = [], 0.0, 1, ""
    for _ in range(args.steps):
        v, cores, text, sp = oracle_sample(seconds=per_step)
        vals.append(v)
        secs += sp
    value = statistics.median(vals)
    emit({"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
          "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": step_config(),
          "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                           "sample": text},
          "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


def small_batch_verify(skv, torch, dev, randn, reps: int = 3, calls: int = 20) -> dict:
    """The verify call alone at batch 1 and 8 (the pages' deployment is batch
    one): a cache per batch set up as the bench's, each call captured 20 times
    into a CUDA graph and replayed; the median device time per call and the
    algorithmic bytes per second.  The 13 MB of a batch-one cache stay in L2
    between the replayed calls, so these are latency figures."""
    res = {}
    for B in (1, 8):
        w = VERIFY_W.with_(C=B)
        cache = skv.StreamCache(w.C, w.P, w.V, w.F, w.T, w.Hkv, w.d, w.theta, tail_cap=w.tail_cap)
        skv.kv_write_rows(cache, 0, randn((w.C, w.P, w.Hkv, w.d)), randn((w.C, w.P, w.Hkv, w.d)))
        for _ in range(w.F):
            skv.kv_stream_insert(cache, randn((w.C, w.V, w.T, w.Hkv, w.d)), randn((w.C, w.V, w.T, w.Hkv, w.d)))
        skv.kv_write_rows(cache, cache.n_visual, randn((w.C, w.tail_len, w.Hkv, w.d)),
                          randn((w.C, w.tail_len, w.Hkv, w.d)))
        qb = randn((w.C, w.blk, w.Hq, w.d), w.q_scale)
        kb = randn((w.C, w.blk, w.Hkv, w.d))
        vb = randn((w.C, w.blk, w.Hkv, w.d))
        tail = torch.full((w.C,), w.tail_len, dtype=torch.int32, device=dev)
        ws = skv.verify_workspace(cache, w.Hq, w.blk)
        out = torch.empty_like(qb)
        for _ in range(3):
            skv.stream_attn_verify(cache, tail, qb, kb, vb, w.sm_scale, ws=ws, out=out)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph):
                for _ in range(calls):
                    skv.stream_attn_verify(cache, tail, qb, kb, vb, w.sm_scale, ws=ws, out=out)
        torch.cuda.current_stream().wait_stream(side)
        graph.replay()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b) / calls)
        if cache.device_status():
            raise RuntimeError("device status %d" % cache.device_status())
        med = statistics.median(ms)
        res["B%d" % B] = {"us": med * 1e3, "gbs": verify_bytes(w) / (med * 1e-3) / 1e9}
        del cache, graph
    return res


def run_only(args):
    """One kernel alone on a reduced case (for ncu captures): scale-up
    geometry with --layers caches for prefill/insert/window/tail, the verify
    workload with batch --layers for verify."""
    import torch
    from streaming_kv_cache_gb300 import build as B
    B.build()
    from streaming_kv_cache_gb300 import skv
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)

    def randn(shape, scale=1.0):
        return (torch.randn(shape, generator=gen, device=dev) * scale).to(torch.bfloat16)

    w = (VERIFY_W if args.only == "verify" else PREFILL_W).with_(C=args.layers)
    if args.only == "tail":
        w = w.with_(tail_cap=max(w.tail_cap, args.tail_n))
    if args.only == "verify" and args.blk:
        w = w.with_(blk=args.blk)
    if args.only == "verify" and args.tail_cap:
        w = w.with_(tail_cap=args.tail_cap)
    mrope = None
    if args.mrope:
        # multi-section rotary: frames in rows of --mrope tokens, 5/16 of the
        # frequencies each on height and width, dealt in turn with temporal
        n_hw = (w.d // 2) * 5 // 16
        sec = [(i % 3 if i // 3 < n_hw else 0) for i in range(w.d // 2)]
        mrope = (args.mrope, sec)
    cache = skv.StreamCache(w.C, w.P, w.V, w.F, w.T, w.Hkv, w.d, w.theta, tail_cap=w.tail_cap, mrope=mrope)
    skv.kv_write_rows(cache, 0, randn((w.C, w.P, w.Hkv, w.d)), randn((w.C, w.P, w.Hkv, w.d)))
    k_new = randn((w.C, w.V, w.T, w.Hkv, w.d))
    for _ in range(w.F):
        skv.kv_stream_insert(cache, k_new, k_new)
    if args.only == "prefill":
        q = randn((w.C, w.n_new, w.Hq, w.d), w.q_scale)
        out = torch.empty_like(q)
        fn = lambda: skv.stream_attn_prefill(cache, q, w.sm_scale, out=out)
        work = prefill_flop(w) / 1e12
        unit = "TFLOP/s"
    elif args.only == "window":
        q = randn((w.C, w.n_window, w.Hq, w.d), w.q_scale)
        out = torch.empty_like(q)
        fn = lambda: skv.stream_attn_window(cache, q, w.sm_scale, out=out)
        work = window_flop(w) / 1e12
        unit = "TFLOP/s"
    elif args.only == "tail":
        n = args.tail_n
        q = randn((w.C, n, w.Hq, w.d), w.q_scale)
        kt = randn((w.C, n, w.Hkv, w.d))
        tail = torch.zeros((w.C,), dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        fn = lambda: skv.stream_attn_prefill_tail(cache, tail, q, kt, kt, w.sm_scale, out=out)
        work = tail_flop(w, n) / 1e12
        unit = "TFLOP/s"
    elif args.only == "prefill_insert":
        q = randn((w.C, w.n_new, w.Hq, w.d), w.q_scale)
        out = torch.empty_like(q)
        fn = lambda: skv.stream_attn_prefill_insert(cache, k_new, k_new, q, w.sm_scale, out=out)
        work = prefill_flop(w) / 1e12
        unit = "TFLOP/s"
    elif args.only == "insert":
        fn = lambda: skv.kv_stream_insert(cache, k_new, k_new)
        work = insert_bytes(w) / 1e9
        unit = "GB/s"
    else:
        skv.kv_write_rows(cache, cache.n_visual, randn((w.C, w.tail_len, w.Hkv, w.d)),
                          randn((w.C, w.tail_len, w.Hkv, w.d)))
        qb = randn((w.C, w.blk, w.Hq, w.d), w.q_scale)
        kb = randn((w.C, w.blk, w.Hkv, w.d))
        tail = torch.full((w.C,), w.tail_len, dtype=torch.int32, device=dev)
        ws = skv.verify_workspace(cache, w.Hq, w.blk)
        out = torch.empty_like(qb)
        fn = lambda: skv.stream_attn_verify(cache, tail, qb, kb, kb, w.sm_scale, ws=ws, out=out)
        work = verify_bytes(w) / 1e9
        unit = "GB/s"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    # the calls are captured once into a CUDA graph and replayed, so the mean
    # is device time, free of Python and launch overhead
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                fn()
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    ms = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b) / args.steps)
    status = cache.device_status()
    med = statistics.median(ms)
    emit({"only": args.only, "layers_or_batch": w.C, "mrope_grid_w": args.mrope, "ms_median": med, "ms": ms,
          "throughput": work / (med * 1e-3), "unit": unit, "device_status": status})
    if status:
        sys.exit(3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["prefill", "prefill_insert", "verify", "insert", "window", "tail"],
                    default=None,
                    help="profiling aid: time one kernel alone on a reduced case and print its ms")
    ap.add_argument("--layers", type=int, default=4,
                    help="layer caches (prefill/insert) or batch (verify) of the --only case")
    ap.add_argument("--tail-n", type=int, default=128,
                    help="tail tokens of the --only tail case (after an empty tail)")
    ap.add_argument("--mrope", type=int, default=0,
                    help="multi-section rotary on the --only case, frames in rows of this many tokens")
    ap.add_argument("--tail-cap", type=int, default=0,
                    help="tail capacity of the --only verify case (default: the workload's 128)")
    ap.add_argument("--blk", type=int, default=None,
                    help="verify block size of the --only verify case (default: the workload's 9)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.only:
        run_only(args)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from streaming_kv_cache_gb300 import build as B
    if rank == 0:
        B.build()
    if dist:
        dist.barrier()
    from streaming_kv_cache_gb300 import skv

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)

    def randn(shape, scale=1.0):
        return (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * scale).to(torch.bfloat16)

    # scale-up streaming workload: prefix + full window, then one step per iteration
    pw = PREFILL_W
    pc = skv.StreamCache(pw.C, pw.P, pw.V, pw.F, pw.T, pw.Hkv, pw.d, pw.theta, tail_cap=pw.tail_cap)
    skv.kv_write_rows(pc, 0, randn((pw.C, pw.P, pw.Hkv, pw.d)), randn((pw.C, pw.P, pw.Hkv, pw.d)))
    k_new = randn((pw.C, pw.V, pw.T, pw.Hkv, pw.d))
    v_new = randn((pw.C, pw.V, pw.T, pw.Hkv, pw.d))
    for _ in range(pw.F):
        skv.kv_stream_insert(pc, k_new, v_new)
    q_new = randn((pw.C, pw.n_new, pw.Hq, pw.d), pw.q_scale)
    p_out = torch.empty_like(q_new)

    # verify workload: Alpamayo-shaped cache x 64, 16 tail tokens, 9-token block
    vw = VERIFY_W
    vc = skv.StreamCache(vw.C, vw.P, vw.V, vw.F, vw.T, vw.Hkv, vw.d, vw.theta, tail_cap=vw.tail_cap)
    skv.kv_write_rows(vc, 0, randn((vw.C, vw.P, vw.Hkv, vw.d)), randn((vw.C, vw.P, vw.Hkv, vw.d)))
    vk = randn((vw.C, vw.V, vw.T, vw.Hkv, vw.d))
    for _ in range(vw.F):
        skv.kv_stream_insert(vc, vk, vk)
    skv.kv_write_rows(vc, vc.n_visual, randn((vw.C, vw.tail_len, vw.Hkv, vw.d)),
                      randn((vw.C, vw.tail_len, vw.Hkv, vw.d)))
    q_blk = randn((vw.C, vw.blk, vw.Hq, vw.d), vw.q_scale)
    k_blk = randn((vw.C, vw.blk, vw.Hkv, vw.d))
    v_blk = randn((vw.C, vw.blk, vw.Hkv, vw.d))
    tgt, drf, _ = synth.planted_ids(vw.C, vw.blk, "bench")
    tgt_d, drf_d = torch.from_numpy(tgt).to(dev), torch.from_numpy(drf).to(dev)
    tail0 = torch.full((vw.C,), vw.tail_len, dtype=torch.int32, device=dev)
    ws = skv.verify_workspace(vc, vw.Hq, vw.blk)
    v_out = torch.empty_like(q_blk)
    acc = torch.empty((vw.C,), dtype=torch.int32, device=dev)
    nxt = torch.empty((vw.C,), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    launches_per_step = 1 + 1 + 2      # insert; prefill; verify: tail write (+ accept) and attention
    ev = {n: [] for n in ("insert", "prefill", "verify")}

    # a step's device inputs and outputs (a second set serves the pipelined
    # end-to-end loop below)
    dev_in = [k_new, v_new, q_new, q_blk, k_blk, v_blk, tgt_d, drf_d]
    dev_out = [p_out, v_out, acc, nxt]

    def step(record, ins=dev_in, outs=dev_out):
        kn, vn, qn, qb, kb, vb, tg, dr = ins
        po, vo, ac, nx = outs
        if record:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record()
        skv.kv_stream_insert(pc, kn, vn)
        if record:
            e[1].record()
        skv.stream_attn_prefill(pc, qn, pw.sm_scale, out=po)
        if record:
            e[2].record()
        skv.stream_attn_verify(vc, tail0, qb, kb, vb, vw.sm_scale, target_ids=tg,
                               draft_ids=dr, ws=ws, out=vo, accept_len=ac, next_token=nx)
        if record:
            e[3].record()
            ev["insert"].append((e[0], e[1]))
            ev["prefill"].append((e[1], e[2]))
            ev["verify"].append((e[2], e[3]))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clk.mark_start()
        start.record()
        for _ in range(args.steps):
            step(True)
        stop.record()
        torch.cuda.synchronize()
        clk.mark_stop()
    if dist:
        dist.barrier()
    t_ms = start.elapsed_time(stop)
    status = pc.device_status() | vc.device_status()
    if status:
        raise RuntimeError("device status %d during the bench: %s" % (status, skv.status_string(status)))

    def avg(name):
        return statistics.mean(a.elapsed_time(b) for a, b in ev[name])

    k_ms = {n: avg(n) for n in ev}

    # --- the stand-alone frame insert: three input sets of 453 MB in turn,
    # so that no call finds its inputs in L2 (the ring heads advance as in a
    # step; the step's own inputs are the first set)
    ins_in = [(k_new, v_new)] + [(randn(k_new.shape), randn(v_new.shape)) for _ in range(2)]
    for i in range(3):
        skv.kv_stream_insert(pc, *ins_in[i % 3])
    torch.cuda.synchronize()
    ins_ev = []
    for i in range(12):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        skv.kv_stream_insert(pc, *ins_in[i % 3])
        b.record()
        ins_ev.append((a, b))
    torch.cuda.synchronize()
    ins_ms = statistics.mean(a.elapsed_time(b) for a, b in ins_ev)
    # the insert and the prefill as one kernel (stream_attn_prefill_insert)
    fz_ev = []
    for i in range(8):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        skv.stream_attn_prefill_insert(pc, *ins_in[i % 3], q_new, pw.sm_scale, out=p_out)
        b.record()
        if i >= 2:
            fz_ev.append((a, b))
    torch.cuda.synchronize()
    fz_ms = statistics.mean(a.elapsed_time(b) for a, b in fz_ev)
    del ins_in
    if pc.device_status():
        raise RuntimeError("device status %d in the insert timing" % pc.device_status())

    # --- end to end through host buffers (pinned), same step, same metric
    h_k = k_new.cpu().pin_memory(); h_v = v_new.cpu().pin_memory(); h_q = q_new.cpu().pin_memory()
    h_qb = q_blk.cpu().pin_memory(); h_kb = k_blk.cpu().pin_memory(); h_vb = v_blk.cpu().pin_memory()
    h_t = torch.from_numpy(tgt).pin_memory(); h_d = torch.from_numpy(drf).pin_memory()
    h_out = torch.empty(p_out.shape, dtype=p_out.dtype).pin_memory()
    h_vout = torch.empty(v_out.shape, dtype=v_out.dtype).pin_memory()
    h_acc = torch.empty(acc.shape, dtype=acc.dtype).pin_memory()
    h_nxt = torch.empty(nxt.shape, dtype=nxt.dtype).pin_memory()
    ins = [h_k, h_v, h_q, h_qb, h_kb, h_vb, h_t, h_d]
    outs = [h_out, h_vout, h_acc, h_nxt]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)

    def e2e_step():
        for d, h in zip(dev_in, ins):
            d.copy_(h, non_blocking=True)
        step(False)
        for h, d in zip(outs, dev_out):
            h.copy_(d, non_blocking=True)

    # serial form: copy in, compute, copy out, one after another on one stream
    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s2, t2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record()
    for _ in range(args.steps):
        e2e_step()
    t2.record()
    torch.cuda.synchronize()
    serial_ms = s2.elapsed_time(t2)

    # pipelined form: step i+1's inputs go up on one copy stream and step i's
    # outputs come down on another while step i's kernels run; device inputs
    # and outputs are double-buffered so that no copy touches a buffer a
    # kernel in flight still reads or writes.  Every step's copies stay inside
    # the timed region.
    dev_in2 = [dev_in, [torch.empty_like(t) for t in dev_in]]
    dev_out2 = [dev_out, [torch.empty_like(t) for t in dev_out]]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ks = torch.cuda.current_stream()

    def e2e_pipelined(n_steps, host_in=lambda i: ins, host_out=lambda i: outs):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]      # the step that read set s is done
        read = [torch.cuda.Event() for _ in range(2)]      # outputs of set s are on the host
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(ks)
        up.wait_event(a)
        down.wait_event(a)

        def upload(k, i):
            with torch.cuda.stream(up):
                for d, h in zip(dev_in2[k], host_in(i)):
                    d.copy_(h, non_blocking=True)
                in_ready[k].record(up)

        upload(0, 0)
        for i in range(n_steps):
            k = i & 1
            if i + 1 < n_steps:
                if i >= 1:
                    up.wait_event(used[k ^ 1])             # step i-1 read set k^1
                upload(k ^ 1, i + 1)
            ks.wait_event(in_ready[k])
            if i >= 2:
                ks.wait_event(read[k])                      # step i-2's outputs are down
            step(False, dev_in2[k], dev_out2[k])
            used[k].record(ks)
            down.wait_event(used[k])
            with torch.cuda.stream(down):
                for h, d in zip(host_out(i), dev_out2[k]):
                    h.copy_(d, non_blocking=True)
                read[k].record(down)
        ks.wait_event(read[(n_steps - 1) & 1])              # the copy-out stream is in order
        b.record(ks)
        return a, b

    e2e_pipelined(args.warmup)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s3, t3 = e2e_pipelined(args.steps)
    torch.cuda.synchronize()
    e2e_ms = s3.elapsed_time(t3)
    status = pc.device_status() | vc.device_status()
    if status:
        raise RuntimeError("device status %d in the end-to-end loops: %s" % (status, skv.status_string(status)))
    e2e_check = check_pipelined(torch, e2e_pipelined, step, dev_in, dev_out, ins, outs, [pc.head, vc.head])

    # the verify call alone at batch 1 and 8 (reported beside the step, untimed by it)
    try:
        small = small_batch_verify(skv, torch, dev, randn)
    except Exception as exc:  # a failure here must not cost the step's line
        small = {"error": str(exc)[:200]}

    t_ms, e2e_ms, serial_ms = max_over_ranks(dist, [t_ms, e2e_ms, serial_ms], dev)

    flop = prefill_flop(pw)
    ms_per_step = t_ms / args.steps
    value = job_throughput(world, flop, args.steps, t_ms)
    e2e_value = job_throughput(world, flop, args.steps, e2e_ms)
    pk, src = peaks()
    pre_tf = flop / (k_ms["prefill"] * 1e-3) / 1e12
    ver_gbs = verify_bytes(vw) / (k_ms["verify"] * 1e-3) / 1e9
    ins_gbs = insert_bytes(pw) / (ins_ms * 1e-3) / 1e9
    tag = "of measured" if src == "measured" else "of fallback"

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, text, _ = oracle_sample()
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": text}

    if rank == 0:
        emit({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": step_config(),
            "kernels_ms": k_ms,
            "roofline": {"bound": "tensor", "kernel": "stream_attn_prefill", "achieved": pre_tf,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": pre_tf / pk["bf16_tflops"], "peak_source": tag + " (burst)",
                         "frac_of_sustained": pre_tf / pk["bf16_tflops_sustained"],
                         "traffic": traffic_for("prefill_tc.cu")},
            "verify_roofline": {"bound": "hbm", "kernel": "stream_attn_verify", "achieved": ver_gbs,
                                "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": ver_gbs / pk["hbm_gbs"], "peak_source": tag,
                                "traffic": traffic_for("verify_tc.cu")},
            "insert_roofline": {"bound": "hbm", "kernel": "kv_stream_insert (stand-alone)", "achieved": ins_gbs,
                                "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": ins_gbs / pk["hbm_gbs"], "peak_source": tag,
                                "ms": ins_ms, "inputs": "3 rotating input sets of 453 MB each, "
                                                        "larger than L2"},
            "verify_small_batch": dict(small, note="one verify call (tail write + attention) at batch 1 "
                                                   "and 8, 9-token block, graph replay of 20 calls, median "
                                                   "of 3; the cache stays in L2 between calls",
                                       hbm_frac={k: v["gbs"] / pk["hbm_gbs"] for k, v in small.items()
                                                 if isinstance(v, dict)}),
            "fused_prefill_insert": {"ms": fz_ms, "tflops": flop / (fz_ms * 1e-3) / 1e12,
                                     "vs_insert_plus_prefill_ms": k_ms["insert"] + k_ms["prefill"],
                                     "note": "insert and prefill as one kernel, same results bit for bit; "
                                             "not used in the step because it is slower"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
                    "copies": "pinned host buffers; step i+1's inputs up and step i's outputs "
                              "down on two copy streams while step i's kernels run "
                              "(double-buffered device inputs and outputs)",
                    "check": e2e_check,
                    "serial": {"value": job_throughput(world, flop, args.steps, serial_ms),
                               "ms_per_step": serial_ms / args.steps,
                               "copies": "in, kernels, out one after another on one stream"}},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        })
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
