#!/usr/bin/env python
"""Benchmark of the LRKV decode on the factored cache (GB300).

The headline step is one lrkv_decode call over the long-context workload:
4 sequences x 65,536 visible rows, 32 heads, d_h = 128, rank 48, bf16 cache
with fp32 accumulation, 5% of the shared key rows scaled by 8.  A step
absorbs q_h B_h^K, scans the factored history with one online softmax per
head, combines the split pieces and lifts the private sum through (B_h^V)^T.
The metric is the cache bytes an ideal kernel must read per second (the
shared rows counted once per sequence, never per head) and its fraction of
the measured HBM bandwidth; decode tokens/s = batch / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs one independent replica per GPU under torchrun (weak scaling, no
data-path collective).  `--impl reference` times the fp64 CPU oracle on the
host cores instead (rank 0 only).  Prints one JSON line.

Timing: W eager warm-up steps, then the K steps are captured as a CUDA graph,
replayed until the GPU has run warm work for a while, and the K-step region is
timed several times (CUDA events on the launching stream); `ms_per_step` is
the median region over K, with the min and max beside it.  `roofline` is the
scan kernel's own: algorithmic bytes per launch over the median duration of
one isolated launch (events right around the kernel, launches replayed from a
graph).  Besides the headline, the line carries: `decode_legs` (the same
measurement on the other decode workloads), `e2e` (host copies in and out
every step, one public-API call per step), `decode_step` (the new token's
rows from its layer input, then the decode, as dependent steps),
`decode_normed` (post-projection RMSNorm key scales), `decode_paged` (the
rows in 256-row pages through a block table), `decode_rope` (full RoPE of the
keys, exact: keys rebuilt tile by tile and rotated), `compare` (dense MHA, GQA
and absorbed MLA at the headline's batch, length and heads) and `prefill` (append GEMM,
causal prefill and the normalised-key prefill of 2 x 4096 tokens, against the
bf16 tensor peak).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LRKV decode cache GB/s (% of HBM peak) & tokens/s; prefill TFLOP/s (% peak)"
PROFILES = os.path.join(ROOT, "profiles")
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0
WARM_MS = 200.0        # warm work replayed before a timed region
TIMED_MS = 1000.0      # the timed repeats of the headline span at least this long


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="headline decode only (no e2e, no other legs)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the length x concurrency sweep")
    ap.add_argument("--max-len", type=int, default=None,
                    help="rows per sequence of the headline workload (a smaller copy of its recipe)")
    return ap.parse_args()


# ---------------------------------------------------------------- accounting

def decode_bytes(w, seq_lens):
    """Algorithmic bytes of one decode call: every visible cache row once
    (2 (d_h + H r) elements per token), the bases, q, and the fp32 outputs."""
    s = w.elem_bytes
    tokens = int(sum(int(x) for x in seq_lens))
    cache = tokens * 2 * (w.head_dim + w.heads * w.rank) * s
    bases = 2 * w.heads * w.head_dim * w.rank * s
    q = w.batch * w.heads * w.head_dim * s
    out = w.batch * w.heads * (w.head_dim + 1) * 4
    split = cache + q  # what the split-KV kernel itself must move
    return cache + bases + q + out, split, cache


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16 burst (cuBLAS)"
    except Exception:
        return 1900.0, "fallback bf16 burst"


def _profile_traffic(workload, src_sha):
    """DRAM bytes per scan launch from the committed ncu summary of this
    workload, if it was taken on the current kernel sources."""
    try:
        with open(os.path.join(PROFILES, f"decode_stream_{workload}.json")) as f:
            d = json.load(f)
        if d.get("source_sha256") == src_sha:
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def _src_sha():
    """sha256 of the decode kernel sources with comments and blank lines
    removed (a comment edit leaves the profiled code, and its hash, as is)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "compressed_cache_decode_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("decode") or name == "ptx.cuh":
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
            h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()


def _spread(xs):
    """median, min and max of a list of per-step times (ms)."""
    return {"median": statistics.median(xs), "min": min(xs), "max": max(xs), "n": len(xs)}


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"lrkv_clocks_{os.getpid()}_{index}.csv")

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            return None
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "samples_under_load": len(loaded)}


# ------------------------------------------------------------- CPU baseline
#
# The oracle (fp64, explicit K_h/V_h reconstruction) runs on bounded samples
# of (sequence, head) pairs.  Each spawned worker (one BLAS thread) receives
# the rows of its own few pairs once, before any timing; a round then asks
# every worker for one pair at once.  Throughput is reported in the metric's
# unit: the workload's algorithmic bytes per decode step times the fraction
# of its (sequence, head) pairs the oracle finished, per second.

def _pair_worker(conn):
    import torch
    from oracle import lrkv_oracle as O
    data = conn.recv()
    conn.send("ready")
    k = 0
    while True:
        msg = conn.recv()
        if msg is None:
            break
        q, k_s, v_s, z_k, z_v, b_k, b_v, L = data[k % len(data)]
        k += 1
        O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, torch.tensor([L], dtype=torch.int32))
        conn.send(1)


def _pair_slices(case, b, h):
    """The inputs of one (sequence, head) pair as a one-sequence, one-head
    decode: q [1,1,d_h], k_s/v_s [1,L,d_h], z [1,L,1,r], bases [1,d_h,r]."""
    L = int(case["seq_lens"][b])
    sl = lambda t: t.contiguous().clone()  # noqa: E731
    return (sl(case["q"][b:b + 1, h:h + 1]), sl(case["k_s"][b:b + 1, :L]), sl(case["v_s"][b:b + 1, :L]),
            sl(case["z_k"][b:b + 1, :L, h:h + 1]), sl(case["z_v"][b:b + 1, :L, h:h + 1]),
            sl(case["b_k"][h:h + 1]), sl(case["b_v"][h:h + 1]), L)


def _sample_pairs(w, n, seed=0):
    import random
    rng = random.Random(seed)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.heads)]
    rng.shuffle(pairs)
    return [pairs[i % len(pairs)] for i in range(n)]


class PairWorkers:
    """`cores` spawned processes, each holding `per` (sequence, head) pairs of
    the case; round() runs one pair on every worker at once."""

    def __init__(self, w, case, cores, per=2, seed=0):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        self.procs, self.conns = [], []
        try:
            for _ in range(cores):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_pair_worker, args=(b,), daemon=True)
                p.start()
                self.procs.append(p)
                self.conns.append(a)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        order = _sample_pairs(w, cores * per, seed)
        for i, c in enumerate(self.conns):
            c.send([_pair_slices(case, *order[i * per + j]) for j in range(per)])
        for c in self.conns:
            assert c.recv() == "ready"
        self.cores = cores

    def round(self):
        for c in self.conns:
            c.send(1)
        return sum(c.recv() for c in self.conns)

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=30)


def cpu_baseline(w, case, seconds, cores):
    """The oracle timed on a bounded sample: rounds of `cores` (sequence,
    head) pairs, one per core, until `seconds` of wall time have passed."""
    workers = PairWorkers(w, case, cores, seed=1)
    total_bytes, _, _ = decode_bytes(w, case["seq_lens"])
    workers.round()  # untimed: imports and first-touch in every worker
    n, t0 = 0, time.perf_counter()
    while True:
        n += workers.round()
        el = time.perf_counter() - t0
        if el >= seconds or n >= 4096:
            break
    workers.close()
    frac = n / (w.batch * w.heads)
    return {"value": total_bytes * frac / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} (sequence, head) pairs of {w.name} ({frac:.3g} of a decode step; each pair "
                      f"an fp64 explicit K_h/V_h reconstruction over its full history), {el:.1f} s wall; "
                      f"GB/s = the step's algorithmic bytes x that fraction / wall time"}


def reference_arm(a, w):
    """--impl reference: the fp64 oracle on the host cores.  A step is a
    bounded sample of the workload: one (sequence, head) pair per core."""
    from compressed_cache_decode_gb300 import inputs
    case = inputs.make_decode_inputs(w, seed=0)
    cores = min(os.cpu_count() or 1, 16)
    workers = PairWorkers(w, case, cores, seed=2)
    total_bytes, _, _ = decode_bytes(w, case["seq_lens"])
    del case
    for _ in range(a.warmup):
        workers.round()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        workers.round()
    el = time.perf_counter() - t0
    workers.close()
    frac = cores / (w.batch * w.heads)
    value = total_bytes * frac * a.steps / el / 1e9 if a.steps > 0 else 0.0
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": el / max(a.steps, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "pairs_per_step": cores, "batch": w.batch, "heads": w.heads,
                       "head_dim": w.head_dim, "rank": w.rank, "seq_len": w.max_len},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{cores} (sequence, head) pairs of {w.name} per step ({frac:.3g} of "
                                       f"a decode step); GB/s = the step's algorithmic bytes x that fraction "
                                       f"/ wall time"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------ GPU timing

def max_over_ranks(value, world, device):
    """The job's time for a per-rank time: the slowest rank's (all-reduce MAX
    over the default process group; the value itself when world == 1)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank, world, ms_per_step):
    """Whole-job throughput: all ranks' bytes per step over the slowest rank's
    step time (every rank decodes its own batch: replicas)."""
    return bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


class StepTimer:
    """K calls of `fn(i, stream)` captured as one CUDA graph (eager launches
    when capture is off or fails), replayed warm, then timed."""

    def __init__(self, fn, K, W, stream, use_graph=True):
        import torch
        self.fn, self.K, self.stream = fn, K, stream
        with torch.cuda.stream(stream):
            for i in range(W):
                fn(i, stream)
        torch.cuda.synchronize()
        self.graph = None
        if use_graph:
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    for i in range(K):
                        fn(i, torch.cuda.current_stream())
                torch.cuda.synchronize()
                self.graph = g
            except Exception as e:  # fall back to eager launches
                print(f"graph capture failed ({e}); timing eager launches", file=sys.stderr)
                torch.cuda.synchronize()

    def _region(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            for i in range(self.K):
                self.fn(i, self.stream)

    def warm(self, ms=WARM_MS):
        import torch
        t0 = time.perf_counter()
        n = 0
        while n < 2 or (time.perf_counter() - t0) * 1e3 < ms:
            with torch.cuda.stream(self.stream):
                self._region()
            torch.cuda.synchronize()
            n += 1

    def time(self, repeats=None, min_ms=0.0):
        """Per-step ms of each timed K-step region."""
        import torch
        out = []
        t0 = time.perf_counter()
        while True:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(self.stream):
                e0.record(self.stream)
                self._region()
                e1.record(self.stream)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) / self.K)
            if repeats is not None and len(out) >= repeats and (time.perf_counter() - t0) * 1e3 >= min_ms:
                break
            if len(out) >= 2000:
                break
        return out


LAUNCH_REPLAYS = 10  # replays whose launches are read by scan_launch_ms


def scan_launch_ms(profiled, n, stream, use_graph=True):
    """Mean duration of one isolated scan launch: `profiled(i, ev0, ev1, s)`
    enqueues a decode with CUDA events right around its scan kernel; the n
    calls are replayed from a graph (so the interval holds the kernel, not the
    host's launch latency), warm, then LAUNCH_REPLAYS more replays are read
    one by one (n x LAUNCH_REPLAYS launches).  The mean, not the median: event
    intervals on these GPUs come in steps of ~2 us, so a median of a ~25 us
    launch jumps by a whole step while the mean of a few hundred samples
    does not.  Returns (mean, median, min, max, kind)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            profiled(i, evs[i][0], evs[i][1], stream)
    torch.cuda.synchronize()
    kind = "eager"
    g = None
    if use_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for i in range(n):
                    profiled(i, evs[i][0], evs[i][1], torch.cuda.current_stream())
            torch.cuda.synchronize()
            kind = "graph"
        except Exception as e:
            print(f"profiled graph capture failed ({e}); eager timing", file=sys.stderr)
            g = None
            torch.cuda.synchronize()
    def replay():
        with torch.cuda.stream(stream):
            if g is not None:
                g.replay()
            else:
                for i in range(n):
                    profiled(i, evs[i][0], evs[i][1], stream)
        torch.cuda.synchronize()

    t0 = time.perf_counter()
    while True:
        replay()
        if (time.perf_counter() - t0) * 1e3 >= 50.0:
            break
    ms = []
    for _ in range(LAUNCH_REPLAYS):
        replay()
        ms += [e0.elapsed_time(e1) for e0, e1 in evs]
    return statistics.fmean(ms), statistics.median(ms), min(ms), max(ms), kind


class DecodeSetup:
    """One decode workload on the device: inputs, rotating cache replicas
    when the cache is small enough to stay in L2, outputs and workspace."""

    def __init__(self, w, dev, seed, max_len=None):
        import torch
        from compressed_cache_decode_gb300 import inputs, lrkv
        if max_len is not None and max_len != w.max_len:
            import dataclasses
            w = dataclasses.replace(w, name=f"{w.name}@L{max_len}", max_len=max_len)
        self.w = w
        self.case = inputs.make_decode_inputs(w, seed=seed)
        d = {k: v.to(dev) for k, v in self.case.items()}
        self.dims = lrkv.make_dims(w.batch, w.heads, w.head_dim, w.rank, w.max_len, w.torch_dtype)
        self.ws = lrkv.decode_workspace(self.dims, dev)
        n_out = w.batch * w.heads * w.head_dim
        self.out_lse = torch.empty(n_out + w.batch * w.heads, dtype=torch.float32, device=dev)
        self.out = self.out_lse[:n_out].view(w.batch, w.heads, w.head_dim)
        self.lse = self.out_lse[n_out:].view(w.batch, w.heads)
        self.total_bytes, self.split_bytes, self.cache_alg = decode_bytes(w, self.case["seq_lens"])
        self.cache_bytes = sum(d[k].numel() * d[k].element_size() for k in ("k_s", "v_s", "z_k", "z_v"))
        if self.cache_alg >= 4 * L2_BYTES:
            self.n_rep = 1
            self.l2 = f"inputs larger than L2 ({self.cache_alg / 1e6:.0f} MB read per step > {L2_BYTES / 1e6:.0f} MB)"
        elif self.cache_alg >= 4096:
            self.n_rep = min(16, max(2, math.ceil(4 * L2_BYTES / self.cache_alg)))
            self.l2 = (f"{self.n_rep} rotating cache replicas ({self.n_rep * self.cache_alg / 1e6:.0f} MB read "
                       f"per cycle > L2 {L2_BYTES / 1e6:.0f} MB)")
        else:
            self.n_rep = 1
            self.l2 = "L2-resident (launch-latency bound: microseconds only)"
        self.reps = [d] + [{k: (v.clone() if k in ("k_s", "v_s", "z_k", "z_v") else v) for k, v in d.items()}
                           for _ in range(self.n_rep - 1)]

    def step(self, i, s):
        from compressed_cache_decode_gb300 import lrkv
        x = self.reps[i % self.n_rep]
        st = lrkv.lrkv_decode(self.dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"], x["b_k"], x["b_v"],
                              x["seq_lens"], self.out, self.lse, self.ws, self.ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode")

    def profiled(self, i, e0, e1, s):
        from compressed_cache_decode_gb300 import lrkv
        x = self.reps[i % self.n_rep]
        st = lrkv.lrkv_decode_profiled(self.dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"], x["b_k"],
                                       x["b_v"], x["seq_lens"], self.out, self.lse, self.ws, self.ws.numel(), e0,
                                       e1, s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode_profiled")


def call_latency_us(step, n_rep, stream, n=200, use_graph=True):
    """Per-call latency: each call's own CUDA-event interval (one decode per
    graph replay, cycled over the cache replicas so that every call reads a
    cold cache), after warm replays.  Percentiles in microseconds."""
    import torch
    graphs = []
    if use_graph:
        try:
            for i in range(n_rep):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    step(i, torch.cuda.current_stream())
                graphs.append(g)
            torch.cuda.synchronize()
        except Exception as e:
            print(f"latency graph capture failed ({e}); eager calls", file=sys.stderr)
            graphs = []
            torch.cuda.synchronize()

    def one(i):
        if graphs:
            graphs[i % len(graphs)].replay()
        else:
            step(i, stream)

    with torch.cuda.stream(stream):
        for i in range(max(20, 2 * n_rep)):
            one(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            evs[i][0].record(stream)
            one(i)
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    t = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)

    def pct(p):
        return t[min(len(t) - 1, int(round(p / 100.0 * (len(t) - 1))))]

    return {"p50": pct(50), "p90": pct(90), "p99": pct(99), "min": t[0], "max": t[-1], "n": n,
            "timing": "CUDA events around each call (graph replay of one call, " +
                      ("graph" if graphs else "eager") + "), calls back to back"}


# The length x concurrency grid of the sweep (the headline's head shape): the
# points the pages' evaluation design asks for on both sides of the
# bandwidth/compute and latency/throughput transitions, up to 2^20 cached rows.
SWEEP_BATCH = (1, 4, 16, 64)
SWEEP_LEN = (1024, 4096, 16384, 65536)
SWEEP_MAX_ROWS = 1 << 20


class SweepSetup:
    """A decode point of the sweep on device-generated inputs (the headline's
    recipe: cache entries and q ~ N(0,1), B ~ N(0,1/r)); rotating cache
    replicas while the cache is small enough to stay in L2."""

    def __init__(self, w, B, L, dev, seed):
        import dataclasses
        import torch
        from compressed_cache_decode_gb300 import lrkv
        self.w = dataclasses.replace(w, name=f"{w.name}@B{B}xL{L}", batch=B, max_len=L, ragged=None,
                                     outlier_frac=0.0)
        H, dh, r = w.heads, w.head_dim, w.rank
        g = torch.Generator(device=dev).manual_seed(1000 + seed)
        bf = torch.bfloat16

        def nrm(*shape, std=1.0):
            return (torch.randn(*shape, generator=g, device=dev) * std).to(bf)

        self.seq_lens = torch.full((B,), L, dtype=torch.int32, device=dev)
        self.q, self.b_k, self.b_v = nrm(B, H, dh), nrm(H, dh, r, std=r ** -0.5), nrm(H, dh, r, std=r ** -0.5)
        self.total_bytes, self.split_bytes, cache_alg = decode_bytes(self.w, self.seq_lens.cpu())
        self.n_rep = 1 if cache_alg >= 4 * L2_BYTES else min(16, max(2, math.ceil(4 * L2_BYTES / cache_alg)))
        self.caches = [(nrm(B, L, dh), nrm(B, L, dh), nrm(B, L, H, r), nrm(B, L, H, r)) for _ in range(self.n_rep)]
        self.dims = lrkv.make_dims(B, H, dh, r, L, bf)
        self.ws = lrkv.decode_workspace(self.dims, dev)
        self.out = torch.empty((B, H, dh), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, H), dtype=torch.float32, device=dev)

    def step(self, i, s):
        from compressed_cache_decode_gb300 import lrkv
        k_s, v_s, z_k, z_v = self.caches[i % self.n_rep]
        st = lrkv.lrkv_decode(self.dims, self.q, k_s, v_s, z_k, z_v, self.b_k, self.b_v, self.seq_lens, self.out,
                              self.lse, self.ws, self.ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode")


def sweep_leg(w, K, W, stream, use_graph, peak, world, dev, seed):
    """Length x concurrency sweep of the decode (the headline's head shape):
    per point the step rate, its HBM fraction, tokens/s and the per-call
    latency quantiles."""
    import torch
    points = []
    for B in SWEEP_BATCH:
        for L in SWEEP_LEN:
            if B * L > SWEEP_MAX_ROWS:
                continue
            sp = SweepSetup(w, B, L, dev, seed)
            t = StepTimer(sp.step, K, W, stream, use_graph)
            t.warm(ms=50)
            ms = max_over_ranks(_spread(t.time(repeats=5))["median"], world, dev)
            del t
            lat = call_latency_us(sp.step, sp.n_rep, stream, n=100, use_graph=use_graph)
            points.append({"batch": B, "seq_len": L, "ms_per_step": ms,
                           "gbs": job_gbs(sp.total_bytes, world, ms),
                           "hbm_frac": sp.total_bytes / (ms * 1e-3) / 1e9 / peak,
                           "tokens_per_s": B * world / (ms * 1e-3), "bytes_per_step": sp.total_bytes,
                           "cache_replicas": sp.n_rep,
                           "latency_us": {k: v for k, v in lat.items() if k != "timing"}})
            del sp
            torch.cuda.empty_cache()
    return {"heads": w.heads, "head_dim": w.head_dim, "rank": w.rank, "data": "synthetic, generated on the device",
            "timing": f"median of 5 timed regions of {K} steps per point; latency: CUDA events around each of "
                      "100 back-to-back calls (graph replays)", "points": points}


def scan_kernel_name(w):
    return "lrkv_decode_stream_kernel" if w.dtype == "bf16" else "lrkv_decode_split_kernel"


def decode_leg(setup, K, W, stream, use_graph, peak, world, dev, repeats=7, min_ms=0.0):
    """Step rate (median of timed K-step regions) and the isolated scan
    launch of one decode workload."""
    w = setup.w
    timer = StepTimer(setup.step, K, W, stream, use_graph)
    timer.warm()
    ms = timer.time(repeats=repeats, min_ms=min_ms)
    sp = _spread(ms)
    ms_step = max_over_ranks(sp["median"], world, dev)
    iso, iso_med, iso_min, iso_max, kind = scan_launch_ms(setup.profiled, min(K, 20), stream, use_graph)
    achieved = setup.split_bytes / (iso * 1e-3) / 1e9
    lat = call_latency_us(setup.step, setup.n_rep, stream, n=200, use_graph=use_graph)
    return {
        "latency_us": lat,
        "workload": w.name, "ms_per_step": ms_step, "ms_per_step_spread": sp,
        "gbs": job_gbs(setup.total_bytes, world, ms_step), "hbm_frac": setup.total_bytes / (ms_step * 1e-3) / 1e9 / peak,
        "tokens_per_s": w.batch * world / (ms_step * 1e-3), "bytes_per_step": setup.total_bytes,
        "seq_len_sum": int(setup.case["seq_lens"].long().sum()), "l2": setup.l2,
        "graph": timer.graph is not None,
        "roofline": {"bound": "hbm", "kernel": scan_kernel_name(w), "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "algorithmic_bytes_per_launch": setup.split_bytes,
                     "launch_ms": iso, "launch_ms_median": iso_med, "launch_ms_min": iso_min,
                     "launch_ms_max": iso_max,
                     "launch_timing": f"CUDA events right around each isolated scan launch on the launching "
                                      f"stream ({kind} launches), mean of {min(K, 20) * LAUNCH_REPLAYS}"},
    }, timer


# ------------------------------------------------------------ prefill leg

def prefill_flops(w):
    """Algorithmic FLOPs of the prefill workload: causal (query, key) pairs
    only, 2 (d_h + r) per pair for the scores and 2 (d_h + r) for the values,
    plus q B^K and the (B^V)^T lift; and the append GEMM 2 M N K."""
    T, B, H, dh, r, d = w.q_len, w.batch, w.heads, w.head_dim, w.rank, w.d_model
    pairs = B * H * T * (T + 1) // 2
    attn = pairs * 4 * (dh + r) + 2 * (2 * B * T * H * dh * r)
    append = 2 * (B * T) * (2 * dh + 2 * H * r) * d
    return attn, append


def prefill_leg(dev, iters=10):
    """Times append (x -> factored cache) and causal prefill on the prefill
    workload with CUDA events, L2 flushed (256 MB write) before each timed
    launch.  Returns TFLOP/s against the measured bf16 peak."""
    import torch
    from compressed_cache_decode_gb300 import inputs, lrkv
    w = inputs.WORKLOADS[inputs.PREFILL_WORKLOAD]
    c = inputs.make_prefill_inputs(w, seed=0)
    d = {k: v.to(dev) for k, v in c.items()}
    B, T, H, dh, r = w.batch, w.q_len, w.heads, w.head_dim, w.rank
    k_s = torch.empty((B, T, dh), dtype=torch.bfloat16, device=dev)
    v_s = torch.empty_like(k_s)
    z_k = torch.empty((B, T, H, r), dtype=torch.bfloat16, device=dev)
    z_v = torch.empty_like(z_k)
    dims = lrkv.make_dims(B, H, dh, r, T, torch.bfloat16)
    nws = lrkv.lrkv_prefill_workspace_size(dims, T)
    ws = torch.zeros(max(nws, 16), dtype=torch.uint8, device=dev)
    out = torch.empty((B, T, H, dh), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def app():
        st = lrkv.lrkv_append(dims, w.d_model, T, d["x"], d["w_sk"], d["w_sv"], d["u_k"], d["u_v"],
                              d["start_pos"], k_s, v_s, z_k, z_v, ws, ws.numel())
        assert st == lrkv.LRKV_OK

    def pre():
        st = lrkv.lrkv_prefill(dims, T, d["q"], k_s, v_s, z_k, z_v, d["b_k"], d["b_v"], d["seq_lens"],
                               out, lse, ws, ws.numel())
        assert st == lrkv.LRKV_OK

    # post-projection RMSNorm of the keys: the scales of every appended row
    # (computed once after the append; the timed call multiplies them in)
    kscale = torch.empty((B, H, T), dtype=torch.float32, device=dev)

    def pre_normed():
        st = lrkv.lrkv_prefill_normed(dims, T, d["q"], k_s, v_s, z_k, z_v, d["b_k"], d["b_v"], kscale,
                                      d["seq_lens"], out, lse, ws, ws.numel())
        assert st == lrkv.LRKV_OK

    def kscales():
        lrkv.key_scales(k_s, z_k, d["b_k"], d["start_pos"], T, kscale, eps=1e-6)

    res, kinds = {}, {}
    for name, fn in (("append", app), ("prefill", pre), ("key_scales", kscales), ("prefill_normed", pre_normed)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        # each call captured once and replayed, so that the interval holds the
        # kernel and not the host's argument marshalling and tensor-map set-up
        run = fn
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                fn()
            torch.cuda.synchronize()
            run = g.replay
            kinds[name] = "graph"
        except Exception as e:
            print(f"prefill leg: graph capture of {name} failed ({e}); eager calls", file=sys.stderr)
            torch.cuda.synchronize()
            kinds[name] = "eager"
        ts = []
        for _ in range(iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        res[name] = _spread(ts)
    attn, append = prefill_flops(w)
    peak = _bf16_peak()
    hbm, _ = _peaks()
    # key scales read k_s and z_k of every row and B^K, write one fp32 per (head, row)
    ks_bytes = B * T * (dh + H * r) * 2 + H * dh * r * 2 + B * H * T * 4
    ms = {k: v["median"] for k, v in res.items()}
    return {"workload": w.name,
            "attention": {"ms": ms["prefill"], "tflops": attn / (ms["prefill"] * 1e-3) / 1e12,
                          "algorithmic_flop": attn, "spread": res["prefill"]},
            "append": {"ms": ms["append"], "tflops": append / (ms["append"] * 1e-3) / 1e12,
                       "algorithmic_flop": append, "spread": res["append"]},
            "attention_normed": {"ms": ms["prefill_normed"],
                                 "tflops": attn / (ms["prefill_normed"] * 1e-3) / 1e12},
            "key_scales": {"ms": ms["key_scales"], "algorithmic_bytes": ks_bytes,
                           "gbs": ks_bytes / (ms["key_scales"] * 1e-3) / 1e9,
                           "hbm_frac": ks_bytes / (ms["key_scales"] * 1e-3) / 1e9 / hbm},
            "peak_tflops": peak[0], "peak_kind": peak[1],
            "attention_frac": attn / (ms["prefill"] * 1e-3) / 1e12 / peak[0],
            "append_frac": append / (ms["append"] * 1e-3) / 1e12 / peak[0],
            "timing": f"CUDA events around each launch (replayed from a CUDA graph: "
                      f"{', '.join(f'{k} {v}' for k, v in kinds.items())}), L2 flushed before it, median of {iters}"}


# -------------------------------------------------------------------- legs

def _token_weights(w, dev, seed=1234):
    """Projection weights of a layer of width d_model = heads x head_dim (the
    new token's rows come from them), x of the new token, seeded."""
    import torch
    d_model = w.heads * w.head_dim
    g = torch.Generator().manual_seed(seed)
    xs = torch.randn(w.batch, d_model, generator=g).to(torch.bfloat16).to(dev)
    wr = [(torch.randn(n, d_model, generator=g) / d_model ** 0.5).to(torch.bfloat16).to(dev)
          for n in (w.head_dim, w.head_dim, w.heads * w.rank, w.heads * w.rank)]
    return d_model, xs, wr


def decode_step_leg(setup, K, W, stream, use_graph, world, dev, base_ms):
    """The new token's rows from its layer input, then the decode, as a chain
    of dependent steps (one lrkv_decode_step per step)."""
    from compressed_cache_decode_gb300 import lrkv
    w = setup.w
    d_model, xs, wr = _token_weights(w, dev)

    def fstep(i, s):
        x = setup.reps[i % setup.n_rep]
        st = lrkv.lrkv_decode_step(setup.dims, d_model, xs, *wr, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"],
                                   x["b_k"], x["b_v"], x["seq_lens"], setup.out, setup.lse, setup.ws,
                                   setup.ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode_step")

    t = StepTimer(fstep, K, W, stream, use_graph)
    t.warm()
    sp = _spread(t.time(repeats=7))
    f_ms = max_over_ranks(sp["median"], world, dev)
    w_bytes = sum(x.numel() * 2 for x in wr)
    rows_bytes = w.batch * 2 * (w.head_dim + w.heads * w.rank) * 2
    alg = setup.total_bytes + w_bytes + xs.numel() * 2 + rows_bytes
    return {"workload": w.name, "d_model": d_model, "ms_per_step": f_ms, "ms_per_step_spread": sp,
            "decode_ms_per_step": base_ms, "projection_ms_per_step": f_ms - base_ms,
            "algorithmic_bytes": alg, "gbs": job_gbs(alg, world, f_ms)}


def decode_normed_leg(setup, K, W, stream, use_graph, world, dev, base_ms):
    """Decode with post-projection RMSNorm of the keys: the cached reciprocal
    key scales (one fp32 per head and token) multiply the summed scores."""
    import torch
    from compressed_cache_decode_gb300 import lrkv
    w = setup.w
    kscales = []
    for x in setup.reps:
        t = torch.empty((w.batch, w.heads, w.max_len), dtype=torch.float32, device=dev)
        lrkv.key_scales(x["k_s"], x["z_k"], x["b_k"], torch.zeros(w.batch, dtype=torch.int32, device=dev),
                        w.max_len, t, eps=1e-6)
        kscales.append(t)
    torch.cuda.synchronize()

    def nstep(i, s):
        x = setup.reps[i % setup.n_rep]
        st = lrkv.lrkv_decode_normed(setup.dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"], x["b_k"], x["b_v"],
                                     kscales[i % setup.n_rep], x["seq_lens"], setup.out, setup.lse, setup.ws,
                                     setup.ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode_normed")

    t = StepTimer(nstep, K, W, stream, use_graph)
    t.warm()
    sp = _spread(t.time(repeats=7))
    n_ms = max_over_ranks(sp["median"], world, dev)
    scale_bytes = int(setup.case["seq_lens"].long().sum()) * w.heads * 4
    del kscales
    return {"workload": w.name, "ms_per_step": n_ms, "ms_per_step_spread": sp, "decode_ms_per_step": base_ms,
            "algorithmic_bytes": setup.total_bytes + scale_bytes,
            "gbs": job_gbs(setup.total_bytes + scale_bytes, world, n_ms), "key_scale_bytes": scale_bytes}


def decode_paged_leg(setup, K, W, stream, use_graph, world, dev, base_ms, page=256):
    """Decode over a paged cache: the same rows in `page`-row pages of a
    pool, in a seeded random page order, through a block table."""
    from compressed_cache_decode_gb300 import inputs, lrkv
    w = setup.w
    pc = inputs.paged_from_contiguous(setup.case, page_size=page, seed=7)
    pd = {k: v.to(dev) for k, v in pc.items()}
    del pc
    preps = [pd] + [{k: (v.clone() if k in ("k_s", "v_s", "z_k", "z_v") else v) for k, v in pd.items()}
                    for _ in range(setup.n_rep - 1)]
    n_pages = pd["k_s"].shape[0]

    def pstep(i, s):
        x = preps[i % setup.n_rep]
        st = lrkv.lrkv_decode_paged(setup.dims, page, n_pages, x["block_table"], x["q"], x["k_s"], x["v_s"],
                                    x["z_k"], x["z_v"], x["b_k"], x["b_v"], x["seq_lens"], setup.out, setup.lse,
                                    setup.ws, setup.ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode_paged")

    t = StepTimer(pstep, K, W, stream, use_graph)
    t.warm()
    sp = _spread(t.time(repeats=7))
    p_ms = max_over_ranks(sp["median"], world, dev)
    return {"workload": w.name, "page_size": page, "pages": n_pages, "ms_per_step": p_ms, "ms_per_step_spread": sp,
            "decode_ms_per_step": base_ms, "gbs": job_gbs(setup.total_bytes, world, p_ms)}


def decode_rope_leg(setup, K, W, stream, use_graph, world, dev, base_ms):
    """Decode with full RoPE of the keys on the same cache (the query taken as
    already rotated): the keys are rebuilt tile by tile (d_h r multiply-adds
    per row and head on the tensor cores), turned by the library's table and
    dotted with the query.  Reported against the plain decode of the cache."""
    import torch
    from compressed_cache_decode_gb300 import lrkv
    w = setup.w
    table = lrkv.rope_table(w.max_len, w.head_dim, device=dev)
    ws = torch.empty(lrkv.lrkv_decode_rope_workspace_size(setup.dims), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def rstep(i, s):
        x = setup.reps[i % setup.n_rep]
        st = lrkv.lrkv_decode_rope(setup.dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"], x["b_k"], x["b_v"],
                                   table, w.max_len, x["seq_lens"], setup.out, setup.lse, ws, ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode_rope")

    t = StepTimer(rstep, K, W, stream, use_graph)
    t.warm()
    sp = _spread(t.time(repeats=7))
    r_ms = max_over_ranks(sp["median"], world, dev)
    tokens = int(setup.case["seq_lens"].long().sum())
    table_bytes = w.max_len * w.head_dim * 4
    rebuild_flop = 2 * tokens * w.heads * w.head_dim * w.rank
    return {"workload": w.name, "ms_per_step": r_ms, "ms_per_step_spread": sp, "decode_ms_per_step": base_ms,
            "algorithmic_bytes": setup.total_bytes + table_bytes,
            "gbs": job_gbs(setup.total_bytes + table_bytes, world, r_ms),
            "hbm_frac": (setup.total_bytes + table_bytes) / (r_ms * 1e-3) / 1e9 / _peaks()[0],
            "rebuild_flop": rebuild_flop, "rebuild_tflops": rebuild_flop / (r_ms * 1e-3) / 1e12 * world}


def compare_leg(w, K, W, stream, use_graph, world, dev, lrkv_ms, peak):
    """The comparison decodes at the headline's batch, length, heads and
    dtype (review §5: a fair serving comparison runs absorbed MLA and
    optimized GQA beside the factored kernel): dense MHA and GQA (8 KV heads)
    over materialised K/V, and absorbed MLA with a 512-wide latent; inputs
    drawn on the device (timing only; parity is in the tests)."""
    import torch
    from compressed_cache_decode_gb300 import lrkv
    B, L, H, dh = w.batch, w.max_len, w.heads, w.head_dim
    gen = torch.Generator(device=dev).manual_seed(11)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    out = torch.empty((B, H, dh), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    res = {}

    def timed(fn, alg_bytes):
        t = StepTimer(fn, K, W, stream, use_graph)
        t.warm()
        sp = _spread(t.time(repeats=7))
        ms = max_over_ranks(sp["median"], world, dev)
        return {"ms_per_step": ms, "ms_per_step_spread": sp, "algorithmic_bytes": alg_bytes,
                "gbs": job_gbs(alg_bytes, world, ms), "hbm_frac": alg_bytes / (ms * 1e-3) / 1e9 / peak,
                "vs_lrkv_time": ms / lrkv_ms}

    q = torch.randn((B, H, dh), generator=gen, device=dev).to(torch.bfloat16)
    for name, hkv in (("mha", H), ("gqa8", 8)):
        k = torch.randn((B, L, hkv, dh), generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn((B, L, hkv, dh), generator=gen, device=dev).to(torch.bfloat16)
        _, _, ws = lrkv.dense_decode(q, k, v, lens, out=out, lse=lse)
        dims = lrkv.lrkv_dense_dims(B, H, hkv, dh, L, 0.0)

        def dstep(i, s, k=k, v=v, ws=ws, dims=dims):
            st = lrkv.load().lrkv_dense_decode(lrkv.ctypes.byref(dims), lrkv._ptr(q), lrkv._ptr(k), lrkv._ptr(v),
                                               lrkv._ptr(lens), lrkv._ptr(out), lrkv._ptr(lse), lrkv._ptr(ws),
                                               ws.numel(), lrkv._stream_handle(s))
            if st != lrkv.LRKV_OK:
                raise lrkv.LRKVError(st, "lrkv_dense_decode")

        alg = B * L * 2 * hkv * dh * 2 + q.numel() * 2 + B * H * (dh + 1) * 4
        res[name] = dict(timed(dstep, alg), kv_heads=hkv, cache_elems_per_token=2 * hkv * dh)
        del k, v, ws
        torch.cuda.empty_cache()
    dc = 512
    c = torch.randn((B, L, dc), generator=gen, device=dev).to(torch.bfloat16)
    w_uk = (torch.randn((H, dh, dc), generator=gen, device=dev) / dc ** 0.5).to(torch.bfloat16)
    w_uv = (torch.randn((H, dh, dc), generator=gen, device=dev) / dc ** 0.5).to(torch.bfloat16)
    _, _, ws = lrkv.mla_decode(q, c, w_uk, w_uv, lens, out=out, lse=lse)
    mdims = lrkv.lrkv_mla_dims(B, H, dh, dc, L, 0.0)

    def mstep(i, s):
        st = lrkv.load().lrkv_mla_decode(lrkv.ctypes.byref(mdims), lrkv._ptr(q), lrkv._ptr(c), lrkv._ptr(w_uk),
                                         lrkv._ptr(w_uv), lrkv._ptr(lens), lrkv._ptr(out), lrkv._ptr(lse),
                                         lrkv._ptr(ws), ws.numel(), lrkv._stream_handle(s))
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_mla_decode")

    alg = B * L * dc * 2 + 2 * H * dh * dc * 2 + q.numel() * 2 + B * H * (dh + 1) * 4
    res["mla512"] = dict(timed(mstep, alg), latent_dim=dc, cache_elems_per_token=dc,
                         score_value_flop=4 * B * L * H * dc)
    del c, w_uk, w_uv, ws
    torch.cuda.empty_cache()
    res["lrkv"] = {"ms_per_step": lrkv_ms, "cache_elems_per_token": 2 * (dh + H * w.rank)}
    res["shape"] = {"batch": B, "seq_len": L, "heads": H, "head_dim": dh, "dtype": "bf16", "position": "none"}
    return res


def e2e_leg(setup, K, stream, use_graph, world, dev):
    """End to end through the public API: every step copies the new token's
    layer input x, its query q and the lengths from pinned host memory (one
    packed copy), makes ONE library call (lrkv_decode_step: the token's cache
    rows from x, then the decode over the cache that now holds them) and
    reads out and lse back (one copy); the host waits for each step's result
    before the next.  Timed two ways: eager (the C-ABI call made from Python
    every step) and with each step's copies and call replayed from a graph.
    The GB/s counts the decode's algorithmic bytes only (the projection's
    weight reads are extra work, not credited)."""
    import torch
    from compressed_cache_decode_gb300 import lrkv
    w = setup.w
    d_model, xs, wr = _token_weights(w, dev, seed=4321)
    host_parts = [("x", xs.cpu()), ("q", setup.case["q"].contiguous()),
                  ("seq_lens", setup.case["seq_lens"].contiguous())]
    offs, n_in = [], 0
    for _, v in host_parts:
        offs.append(n_in)
        n_in += (v.numel() * v.element_size() + 255) // 256 * 256
    host_in = torch.zeros(n_in, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(n_in, dtype=torch.uint8, device=dev)
    views = {}
    for (k, v), o in zip(host_parts, offs):
        nb = v.numel() * v.element_size()
        host_in[o:o + nb].copy_(v.reshape(-1).view(torch.uint8))
        views[k] = dev_in[o:o + nb].view(v.dtype).view(v.shape)
    host_out = torch.empty_like(setup.out_lse, device="cpu").pin_memory()
    h2d = sum(v.numel() * v.element_size() for _, v in host_parts)
    d2h = host_out.numel() * 4

    def body(i, s):
        x = setup.reps[i % setup.n_rep]
        dev_in.copy_(host_in, non_blocking=True)
        st = lrkv.lrkv_decode_step(setup.dims, d_model, views["x"], *wr, views["q"], x["k_s"], x["v_s"], x["z_k"],
                                   x["z_v"], x["b_k"], x["b_v"], views["seq_lens"], setup.out, setup.lse, setup.ws,
                                   setup.ws.numel(), s)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode_step")
        host_out.copy_(setup.out_lse, non_blocking=True)

    graphs = None
    if use_graph:
        try:
            graphs = []
            for r in range(setup.n_rep):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    body(r, torch.cuda.current_stream())
                graphs.append(g)
            torch.cuda.synchronize()
        except Exception as e:
            print(f"end-to-end graph capture failed ({e})", file=sys.stderr)
            graphs = None
            torch.cuda.synchronize()

    def run(n, graphed):
        with torch.cuda.stream(stream):
            for i in range(n):
                if graphed:
                    graphs[i % setup.n_rep].replay()
                else:
                    body(i, stream)
                stream.synchronize()

    K_e2e = max(K, 10)
    res = {}
    for kind in (["eager", "graph"] if graphs is not None else ["eager"]):
        g = kind == "graph"
        t0 = time.perf_counter()
        while (time.perf_counter() - t0) < 0.1:
            run(3, g)
        reps = []
        for _ in range(5):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(K_e2e, g)
            e1.record(stream)
            torch.cuda.synchronize()
            reps.append(e0.elapsed_time(e1) / K_e2e)
        res[kind] = _spread(reps)
    e_ms = max_over_ranks(res["eager"]["median"], world, dev)
    out = {"value": job_gbs(setup.total_bytes, world, e_ms), "unit": "GB/s", "ms_per_step": e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "call": "lrkv_decode_step",
           "workload": w.name, "timing": "eager: host copy in, one C-ABI call, copy out, host waits, every step",
           "eager": res["eager"]}
    if "graph" in res:
        g_ms = max_over_ranks(res["graph"]["median"], world, dev)
        out["graph"] = dict(res["graph"], gbs=job_gbs(setup.total_bytes, world, g_ms))
    return out


# -------------------------------------------------------------------- main

def main():
    a = _args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from compressed_cache_decode_gb300 import inputs
    w = inputs.WORKLOADS[a.workload or inputs.DECODE_BENCH_WORKLOAD]
    if w.kind != "decode":
        raise SystemExit("bench.py times the decode workloads")

    if a.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(a, w)), flush=True)
        return

    import torch
    import torch.distributed as dist
    from compressed_cache_decode_gb300 import build as _build
    from compressed_cache_decode_gb300 import lrkv

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    lrkv.load()
    peak, peak_kind = _peaks()
    use_graph = not a.no_graph
    K, W = a.steps, a.warmup
    stream = torch.cuda.Stream(device=dev)

    # ---- headline: timed repeats of the K-step region, clocks sampled ----
    head = DecodeSetup(w, dev, seed=rank, max_len=a.max_len)
    w = head.w
    timer = StepTimer(head.step, K, W, stream, use_graph)
    timer.warm()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms_list = timer.time(repeats=7, min_ms=TIMED_MS)
    if world > 1:
        dist.barrier()
    spread = _spread(ms_list)
    ms_step = max_over_ranks(spread["median"], world, dev)
    iso, iso_med, iso_min, iso_max, iso_kind = scan_launch_ms(head.profiled, min(K, 20), stream, use_graph)
    del timer
    latency = call_latency_us(head.step, head.n_rep, stream, n=200, use_graph=use_graph)

    e2e = e2e_leg(head, K, stream, use_graph, world, dev) if not a.no_legs else None
    normed_leg = decode_normed_leg(head, K, W, stream, use_graph, world, dev, ms_step) if not a.no_legs else None
    paged_leg = decode_paged_leg(head, K, W, stream, use_graph, world, dev, ms_step) if not a.no_legs else None
    rope_leg = decode_rope_leg(head, K, W, stream, use_graph, world, dev, ms_step) if not a.no_legs else None
    cmp_leg = None
    if not a.no_legs:
        del head.reps[1:]
        torch.cuda.empty_cache()
        cmp_leg = compare_leg(w, K, W, stream, use_graph, world, dev, ms_step, peak)

    # ---- the other decode workloads, and the decode step on the 4K one ----
    legs, step_leg = {}, None
    if not a.no_legs:
        for name in inputs.DECODE_LEG_WORKLOADS:
            s = DecodeSetup(inputs.WORKLOADS[name], dev, seed=rank)
            leg, _ = decode_leg(s, K, W, stream, use_graph, peak, world, dev)
            legs[name] = leg
            if name == "decode_bf16_b8_h16_d64_r28_L4096":
                step_leg = decode_step_leg(s, K, W, stream, use_graph, world, dev, leg["ms_per_step"])
            del s
            torch.cuda.empty_cache()

    sweep = None
    if not a.no_legs and not a.no_sweep:
        sweep = sweep_leg(w, K, W, stream, use_graph, peak, world, dev, seed=rank)

    prefill = None
    if not a.no_prefill:
        prefill = prefill_leg(dev)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(w, head.case, a.cpu_seconds, min(os.cpu_count() or 1, 16))

    if rank == 0:
        gbs = job_gbs(head.total_bytes, world, ms_step)
        achieved = head.split_bytes / (iso * 1e-3) / 1e9
        traffic = _profile_traffic(w.name, _src_sha())
        res = {
            "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_step, "ms_per_step_spread": spread, "latency_us": latency,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
            "tokens_per_s": w.batch * world / (ms_step * 1e-3),
            "hbm_frac": gbs / world / peak,
            "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": w.head_dim,
                       "rank": w.rank, "seq_len": w.max_len, "seq_len_sum": int(head.case["seq_lens"].long().sum()),
                       "cache_fraction_of_mha": 1 / w.heads + w.rank / w.head_dim,
                       "bytes_per_step": head.total_bytes, "l2": head.l2,
                       "graph": use_graph, "parallelism": f"replicas x{world}",
                       "timing": f"median of {spread['n']} timed regions of {K} steps (graph replays, after "
                                 f">= {WARM_MS:.0f} ms of warm replays)"},
            "roofline": {"bound": "hbm", "kernel": "lrkv_decode_stream_kernel", "achieved": achieved,
                         "peak": peak, "peak_kind": f"{peak_kind} HBM copy", "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": head.split_bytes, "launch_ms": iso,
                         "launch_ms_median": iso_med, "launch_ms_min": iso_min, "launch_ms_max": iso_max,
                         "launch_timing": f"CUDA events right around each isolated scan launch on the launching "
                                          f"stream ({iso_kind} launches), mean of {min(K, 20) * LAUNCH_REPLAYS}",
                         "step_rate_gbs": head.split_bytes / (ms_step * 1e-3) / 1e9,
                         "step_rate_frac": head.split_bytes / (ms_step * 1e-3) / 1e9 / peak},
            "cpu_baseline": cpu,
            "e2e": e2e,
            # a bf16 step on the streaming path is two launches (scan, merge)
            "gpu_launches": 2 * K,
            "clocks": clk.summary(),
            "decode_legs": legs or None,
            "decode_step": step_leg,
            "decode_normed": normed_leg,
            "decode_paged": paged_leg,
            "decode_rope": rope_leg,
            "compare": cmp_leg,
            "sweep": sweep,
            "prefill": prefill,
        }
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
