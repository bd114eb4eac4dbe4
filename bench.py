#!/usr/bin/env python
"""Benchmark of one LRKV decode step on the factored cache (GB300).

A step is one lrkv_decode call over a batch of 8 sequences x 16 heads,
d_h = 64, rank 28, 4096 visible rows each (bf16 cache, fp32 accumulation):
absorb q_h B_h^K, scan the factored history with one online softmax per head,
combine the split pieces and lift the private sum through (B_h^V)^T.  The
metric is the cache bytes an ideal kernel must read per second (the shared
rows counted once per sequence, never per head) and its fraction of the
measured HBM bandwidth; decode tokens/s = batch / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs one independent replica per GPU under torchrun (weak scaling, no
data-path collective).  `--impl reference` times the fp64 CPU oracle on the
host cores instead (rank 0 only).  Prints one JSON line.

Besides the headline step, the line carries: `roofline` (the scan kernel's
average launch duration over the timed region, with the isolated per-launch
figure beside it), `e2e` (host copies in and out every step), and the legs of
the rest of the path on the same cache: `decode_step` (the new token's rows
from its layer input, then the decode, as dependent steps), `decode_normed`
(post-projection RMSNorm key scales), `decode_paged` (the rows in 256-row pages
through a block table) and `prefill` (append GEMM, causal prefill and the
normalised-key prefill of 2 x 4096 tokens, against the bf16 tensor peak).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LRKV decode cache GB/s (% of HBM peak) & tokens/s; prefill TFLOP/s (% peak)"
PROFILE_JSON = os.path.join(ROOT, "profiles", "decode_stream_b8_h16_d64_r28_L4096.json")
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
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


def _profile_traffic(split_kernel_src_sha):
    """DRAM bytes per split launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    try:
        with open(PROFILE_JSON) as f:
            d = json.load(f)
        if d.get("source_sha256") == split_kernel_src_sha:
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


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"lrkv_clocks_{os.getpid()}.csv")

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
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU baseline

_POOL_DATA = None


def _pool_init(data):
    global _POOL_DATA
    _POOL_DATA = data


def _oracle_task(task):
    """One piece of the CPU baseline: the fp64 oracle on one sequence's heads."""
    from oracle import lrkv_oracle as O
    b, heads = task
    d = _POOL_DATA
    sl = slice(b, b + 1)
    O.decode_reference(d["q"][sl], d["k_s"][sl], d["v_s"][sl], d["z_k"][sl], d["z_v"][sl],
                       d["b_k"], d["b_v"], d["seq_lens"][sl], pairs=[(0, h) for h in heads])
    return len(heads)


class OraclePool:
    """Spawned worker processes, one BLAS thread each, holding the inputs."""

    def __init__(self, case, cores):
        import multiprocessing as mp
        self.cores = cores
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(cores, initializer=_pool_init, initargs=(case,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.pool.map(_oracle_task, [(0, [0])] * cores)  # import oracle in every worker

    def run(self, tasks):
        return sum(self.pool.map(_oracle_task, tasks, chunksize=1))

    def close(self):
        self.pool.close()
        self.pool.join()


def _tasks(w, split):
    heads = list(range(w.heads))
    per = max(1, math.ceil(w.heads / split))
    return [(b, heads[i:i + per]) for b in range(w.batch) for i in range(0, w.heads, per)]


def cpu_baseline(w, case, seconds, cores):
    """Oracle timed on a bounded sample: whole decode steps (all sequences and
    heads) repeated until `seconds` of wall time have passed."""
    pool = OraclePool(case, cores)
    tasks = _tasks(w, max(1, (2 * cores) // w.batch))
    total_bytes, _, _ = decode_bytes(w, case["seq_lens"])
    n, t0 = 0, time.perf_counter()
    while True:
        pool.run(tasks)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 400:
            break
    pool.close()
    return {"value": total_bytes * n / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} full decode step(s) of {w.name} (all {w.batch}x{w.heads} sequence-head "
                      f"pairs, fp64 explicit K_h/V_h reconstruction), {el:.1f} s wall"}


def reference_arm(a, w):
    """--impl reference: the fp64 oracle on the host cores, one bounded sample
    (one sequence, all heads) per step."""
    from compressed_cache_decode_gb300 import inputs
    case = inputs.make_decode_inputs(w, seed=0)
    cores = min(os.cpu_count() or 1, 16)
    pool = OraclePool(case, cores)
    per_b = _tasks(w, cores)
    B = w.batch
    _, _, cache_all = decode_bytes(w, case["seq_lens"])
    seq_bytes = cache_all / B + 2 * w.heads * w.head_dim * w.rank * w.elem_bytes \
        + w.heads * w.head_dim * (w.elem_bytes + 4)
    for i in range(a.warmup):
        b = i % B
        pool.run([t for t in per_b if t[0] == b])
    t0 = time.perf_counter()
    for i in range(a.steps):
        b = i % B
        pool.run([t for t in per_b if t[0] == b])
    el = time.perf_counter() - t0
    pool.close()
    value = seq_bytes * a.steps / el / 1e9
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": el / a.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "batch_per_step": 1, "heads": w.heads,
                       "head_dim": w.head_dim, "rank": w.rank, "seq_len": w.max_len},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"one sequence (all {w.heads} heads) of {w.name} per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


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
    ws = torch.zeros(16, dtype=torch.uint8, device=dev)
    out = torch.empty((B, T, H, dh), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def app():
        st = lrkv.lrkv_append(dims, w.d_model, T, d["x"], d["w_sk"], d["w_sv"], d["u_k"], d["u_v"],
                              d["start_pos"], k_s, v_s, z_k, z_v, ws, 16)
        assert st == lrkv.LRKV_OK

    def pre():
        st = lrkv.lrkv_prefill(dims, T, d["q"], k_s, v_s, z_k, z_v, d["b_k"], d["b_v"], d["seq_lens"],
                               out, lse, ws, 16)
        assert st == lrkv.LRKV_OK

    # post-projection RMSNorm of the keys: the scales of every appended row
    # (computed once after the append; the timed call multiplies them in)
    kscale = torch.empty((B, H, T), dtype=torch.float32, device=dev)

    def pre_normed():
        st = lrkv.lrkv_prefill_normed(dims, T, d["q"], k_s, v_s, z_k, z_v, d["b_k"], d["b_v"], kscale,
                                      d["seq_lens"], out, lse, ws, 16)
        assert st == lrkv.LRKV_OK

    res = {}
    for name, fn in (("append", app), ("prefill", pre), ("prefill_normed", pre_normed)):
        if name == "prefill_normed":
            lrkv.key_scales(k_s, z_k, d["b_k"], d["start_pos"], T, kscale, eps=1e-6)
        for _ in range(3):
            fn()
        ts = []
        for _ in range(iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        res[name] = statistics.median(ts)
    attn, append = prefill_flops(w)
    peak = _bf16_peak()
    return {"workload": w.name,
            "attention": {"ms": res["prefill"], "tflops": attn / (res["prefill"] * 1e-3) / 1e12,
                          "algorithmic_flop": attn},
            "append": {"ms": res["append"], "tflops": append / (res["append"] * 1e-3) / 1e12,
                       "algorithmic_flop": append},
            "attention_normed": {"ms": res["prefill_normed"],
                                 "tflops": attn / (res["prefill_normed"] * 1e-3) / 1e12},
            "peak_tflops": peak[0], "peak_kind": peak[1],
            "attention_frac": attn / (res["prefill"] * 1e-3) / 1e12 / peak[0],
            "append_frac": append / (res["append"] * 1e-3) / 1e12 / peak[0]}


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16 burst (cuBLAS)"
    except Exception:
        return 1900.0, "fallback bf16 burst"


# -------------------------------------------------------------------- GPU arm

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

    case = inputs.make_decode_inputs(w, seed=rank)
    d = {k: v.to(dev) for k, v in case.items()}
    dims = lrkv.make_dims(w.batch, w.heads, w.head_dim, w.rank, w.max_len, w.torch_dtype)
    ws = lrkv.decode_workspace(dims, dev)
    # out and lse in one buffer, so that a step's results come back in one copy
    n_out = w.batch * w.heads * w.head_dim
    out_lse = torch.empty(n_out + w.batch * w.heads, dtype=torch.float32, device=dev)
    out = out_lse[:n_out].view(w.batch, w.heads, w.head_dim)
    lse = out_lse[n_out:].view(w.batch, w.heads)

    # rotate cache replicas so that consecutive steps never hit in L2
    cache_bytes = sum(d[k].numel() * d[k].element_size() for k in ("k_s", "v_s", "z_k", "z_v"))
    n_rep = max(2, math.ceil(4 * L2_BYTES / cache_bytes)) if cache_bytes < 4 * L2_BYTES else 1
    reps = [d] + [{k: (v.clone() if k in ("k_s", "v_s", "z_k", "z_v") else v) for k, v in d.items()}
                  for _ in range(n_rep - 1)]
    total_bytes, split_bytes, _ = decode_bytes(w, case["seq_lens"])
    stream = torch.cuda.Stream(device=dev)

    def step(i, s=None):
        x = reps[i % n_rep]
        st = lrkv.lrkv_decode(dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"], x["b_k"],
                              x["b_v"], x["seq_lens"], out, lse, ws, ws.numel(), s or stream)
        if st != lrkv.LRKV_OK:
            raise lrkv.LRKVError(st, "lrkv_decode")

    K, W = a.steps, a.warmup
    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()

    graph = None
    if not a.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                for i in range(K):
                    step(i, torch.cuda.current_stream())
            torch.cuda.synchronize()
            graph.replay()  # warm the graph once (untimed)
            torch.cuda.synchronize()
        except Exception as e:  # fall back to eager launches
            print(f"graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                for i in range(K):
                    step(i)
            ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_max = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    ms_step = ms_max / K

    # dominant kernel (split-KV scan) timed alone with events around it; the
    # profiled calls are replayed from a CUDA graph (as the step is), so that
    # the interval holds the kernel rather than the host's launch latency
    n_prof = min(K, 50)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_prof)]

    def prof_calls(s):
        for i in range(n_prof):
            x = reps[i % n_rep]
            st = lrkv.lrkv_decode_profiled(dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"],
                                           x["b_k"], x["b_v"], x["seq_lens"], out, lse, ws,
                                           ws.numel(), evs[i][0], evs[i][1], s)
            if st != lrkv.LRKV_OK:
                raise lrkv.LRKVError(st, "lrkv_decode_profiled")

    split_timing = "eager"
    with torch.cuda.stream(stream):
        prof_calls(stream)  # warm, and the eager fallback
    torch.cuda.synchronize()
    if graph is not None:
        try:
            pg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pg, stream=stream, capture_error_mode="thread_local"):
                prof_calls(torch.cuda.current_stream())
            torch.cuda.synchronize()
            pg.replay()
            torch.cuda.synchronize()
            pg.replay()
            torch.cuda.synchronize()
            split_timing = "graph"
        except Exception as e:
            print(f"profiled graph capture failed ({e}); using the eager timing", file=sys.stderr)
            torch.cuda.synchronize()
    split_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)

    # end to end through the public API: each step copies the new token's
    # query, the lengths and the token's cache rows from pinned host memory
    # (packed in one buffer: one host->device copy, then device-side placement
    # into the resident cache), decodes, and reads out and lse back (one copy).
    host_parts = [("q", case["q"].contiguous()), ("seq_lens", case["seq_lens"].contiguous())] + \
        [(k, case[k][:, -1:].contiguous()) for k in ("k_s", "v_s", "z_k", "z_v")]
    offs, n_in = [], 0
    for k, v in host_parts:
        offs.append(n_in)
        n_in += (v.numel() * v.element_size() + 255) // 256 * 256
    host_in = torch.zeros(n_in, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(n_in, dtype=torch.uint8, device=dev)
    in_views = []
    for (k, v), o in zip(host_parts, offs):
        nb = v.numel() * v.element_size()
        host_in[o:o + nb].copy_(v.reshape(-1).view(torch.uint8))
        in_views.append((k, dev_in[o:o + nb].view(v.dtype).view(v.shape)))
    host_out_lse = torch.empty_like(out_lse, device="cpu").pin_memory()
    h2d = sum(v.numel() * v.element_size() for _, v in host_parts)
    d2h = host_out_lse.numel() * 4
    K_e2e = min(K, 100)

    def e2e_body(i, s=None):
        x = reps[i % n_rep]
        dev_in.copy_(host_in, non_blocking=True)
        for k, v in in_views:
            if k in ("q", "seq_lens"):
                x[k].copy_(v)
            else:
                x[k][:, -1:].copy_(v)
        step(i, s)
        host_out_lse.copy_(out_lse, non_blocking=True)

    # one CUDA graph per cache replica holds a step's copies and the decode
    # call (as a serving loop replays its step); the host still waits for each
    # step's outputs before the next step starts
    e2e_graphs = None
    if not a.no_graph:
        try:
            e2e_graphs = []
            for r in range(n_rep):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    e2e_body(r, torch.cuda.current_stream())
                e2e_graphs.append(g)
            torch.cuda.synchronize()
        except Exception as e:
            print(f"end-to-end graph capture failed ({e}); eager steps", file=sys.stderr)
            e2e_graphs = None
            torch.cuda.synchronize()

    def e2e_step(i):
        if e2e_graphs is not None:
            e2e_graphs[i % n_rep].replay()
        else:
            e2e_body(i)
        stream.synchronize()

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K_e2e):
            e2e_step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K_e2e, world, dev)

    # decode step: the new token's rows from its layer input (d_model =
    # heads x head_dim), then the decode, as one call per step, from a graph
    step_leg = None
    if not a.no_graph:
        d_model = w.heads * w.head_dim
        g = torch.Generator().manual_seed(1234)
        xs = torch.randn(w.batch, d_model, generator=g).to(torch.bfloat16).to(dev)
        ws_rows = [(torch.randn(n, d_model, generator=g) / d_model ** 0.5).to(torch.bfloat16).to(dev)
                   for n in (w.head_dim, w.head_dim, w.heads * w.rank, w.heads * w.rank)]

        def fstep(i, s=None):
            x = reps[i % n_rep]
            st = lrkv.lrkv_decode_step(dims, d_model, xs, *ws_rows, x["q"], x["k_s"], x["v_s"], x["z_k"],
                                       x["z_v"], x["b_k"], x["b_v"], x["seq_lens"], out, lse, ws, ws.numel(),
                                       s or stream)
            if st != lrkv.LRKV_OK:
                raise lrkv.LRKVError(st, "lrkv_decode_step")

        with torch.cuda.stream(stream):
            for i in range(W):
                fstep(i)
        torch.cuda.synchronize()
        fg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fg, stream=stream, capture_error_mode="thread_local"):
            for i in range(K):
                fstep(i, torch.cuda.current_stream())
        torch.cuda.synchronize()
        fg.replay()
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            f0.record(stream)
            fg.replay()
            f1.record(stream)
        torch.cuda.synchronize()
        f_ms = max_over_ranks(f0.elapsed_time(f1) / K, world, dev)
        w_bytes = sum(t.numel() * 2 for t in ws_rows)
        rows_bytes = w.batch * 2 * (w.head_dim + w.heads * w.rank) * 2
        step_leg = {"d_model": d_model, "ms_per_step": f_ms, "decode_ms_per_step": ms_step,
                    "projection_ms_per_step": f_ms - ms_step,
                    "algorithmic_bytes": total_bytes + w_bytes + xs.numel() * 2 + rows_bytes,
                    "gbs": job_gbs(total_bytes + w_bytes + xs.numel() * 2 + rows_bytes, world, f_ms)}

    # decode with post-projection RMSNorm of the keys: the cached reciprocal
    # key scales (one fp32 per head and token) multiply the summed scores
    normed_leg = None
    if not a.no_graph:
        kscales = []
        for x in reps:
            t = torch.empty((w.batch, w.heads, w.max_len), dtype=torch.float32, device=dev)
            lrkv.key_scales(x["k_s"], x["z_k"], x["b_k"], torch.zeros(w.batch, dtype=torch.int32, device=dev),
                            w.max_len, t, eps=1e-6)
            kscales.append(t)
        torch.cuda.synchronize()

        def nstep(i, s=None):
            x = reps[i % n_rep]
            st = lrkv.lrkv_decode_normed(dims, x["q"], x["k_s"], x["v_s"], x["z_k"], x["z_v"], x["b_k"], x["b_v"],
                                         kscales[i % n_rep], x["seq_lens"], out, lse, ws, ws.numel(), s or stream)
            if st != lrkv.LRKV_OK:
                raise lrkv.LRKVError(st, "lrkv_decode_normed")

        with torch.cuda.stream(stream):
            for i in range(W):
                nstep(i)
        torch.cuda.synchronize()
        ng = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ng, stream=stream, capture_error_mode="thread_local"):
            for i in range(K):
                nstep(i, torch.cuda.current_stream())
        torch.cuda.synchronize()
        ng.replay()
        torch.cuda.synchronize()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            n0.record(stream)
            ng.replay()
            n1.record(stream)
        torch.cuda.synchronize()
        n_ms = max_over_ranks(n0.elapsed_time(n1) / K, world, dev)
        scale_bytes = int(case["seq_lens"].long().sum()) * w.heads * 4
        normed_leg = {"ms_per_step": n_ms, "decode_ms_per_step": ms_step,
                      "algorithmic_bytes": total_bytes + scale_bytes,
                      "gbs": job_gbs(total_bytes + scale_bytes, world, n_ms),
                      "key_scale_bytes": scale_bytes}

    # decode over a paged cache: the same rows in 256-row pages of a pool, in a
    # seeded random page order, through a block table
    paged_leg = None
    if not a.no_graph:
        page = 256
        pc = inputs.paged_from_contiguous(case, page_size=page, seed=7)
        pd = {k: v.to(dev) for k, v in pc.items()}
        preps = [pd] + [{k: (v.clone() if k in ("k_s", "v_s", "z_k", "z_v") else v) for k, v in pd.items()}
                        for _ in range(n_rep - 1)]
        n_pages = pd["k_s"].shape[0]

        def pstep(i, s=None):
            x = preps[i % n_rep]
            st = lrkv.lrkv_decode_paged(dims, page, n_pages, x["block_table"], x["q"], x["k_s"], x["v_s"],
                                        x["z_k"], x["z_v"], x["b_k"], x["b_v"], x["seq_lens"], out, lse, ws,
                                        ws.numel(), s or stream)
            if st != lrkv.LRKV_OK:
                raise lrkv.LRKVError(st, "lrkv_decode_paged")

        with torch.cuda.stream(stream):
            for i in range(W):
                pstep(i)
        torch.cuda.synchronize()
        pg_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pg_graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(K):
                pstep(i, torch.cuda.current_stream())
        torch.cuda.synchronize()
        pg_graph.replay()
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            p0.record(stream)
            pg_graph.replay()
            p1.record(stream)
        torch.cuda.synchronize()
        p_ms = max_over_ranks(p0.elapsed_time(p1) / K, world, dev)
        paged_leg = {"page_size": page, "pages": n_pages, "ms_per_step": p_ms, "decode_ms_per_step": ms_step,
                     "gbs": job_gbs(total_bytes, world, p_ms)}
        del preps, pd

    prefill = None
    if not a.no_prefill:
        prefill = prefill_leg(dev)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(w, case, a.cpu_seconds, min(os.cpu_count() or 1, 16))

    if rank == 0:
        peak, peak_kind = _peaks()
        gbs = job_gbs(total_bytes, world, ms_step)
        # the scan's average launch duration over the timed region: one scan
        # launch per step, back to back (each launched ahead, programmatic
        # dependent launch), the combine beside it on SMs the scan leaves free
        achieved = split_bytes / (ms_step * 1e-3) / 1e9
        isolated = split_bytes / (split_ms * 1e-3) / 1e9
        traffic = _profile_traffic(_src_sha())
        res = {
            "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
            "tokens_per_s": w.batch * world / (ms_step * 1e-3),
            "hbm_frac": gbs / world / peak,
            "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": w.head_dim,
                       "rank": w.rank, "seq_len": w.max_len,
                       "cache_fraction_of_mha": 1 / w.heads + w.rank / w.head_dim,
                       "bytes_per_step": total_bytes,
                       "l2": f"{n_rep} rotating cache replicas ({n_rep * cache_bytes / 1e6:.0f} MB > L2 "
                             f"{L2_BYTES / 1e6:.0f} MB)",
                       "graph": graph is not None, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "lrkv_decode_stream_kernel", "achieved": achieved,
                         "peak": peak, "peak_kind": f"{peak_kind} HBM copy", "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": split_bytes, "launch_ms": ms_step,
                         "launch_timing": "CUDA events around the timed region of K back-to-back steps "
                                          "(one scan launch per step) on the launching stream",
                         "isolated_launch_ms": split_ms, "isolated_achieved": isolated,
                         "isolated_frac": isolated / peak,
                         "isolated_timing": f"CUDA events around each launch alone, {split_timing} launches "
                                            "(includes the launch and drain the chained steps overlap)"},
            "cpu_baseline": cpu,
            "e2e": {"value": job_gbs(total_bytes, world, e2e_ms), "unit": "GB/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "graph": e2e_graphs is not None},
            # a bf16 step on the streaming path is two launches (scan, merge)
            "gpu_launches": 2 * K,
            "clocks": clk.summary(),
            "decode_step": step_leg,
            "decode_normed": normed_leg,
            "decode_paged": paged_leg,
            "prefill": prefill,
        }
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
