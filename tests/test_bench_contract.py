"""The bench's JSON contract on CPU: the reference arm (the fp64 oracle on the
host cores) prints one JSON line with the keys every arm carries, on the
headline workload; the algorithmic byte count of a decode is the cache rows
once plus q (67,125,248 B for 8 sequences x 4096 rows, 16 heads, d_h 64, rank
28, bf16; 1,744,863,232 B for 4 x 65,536 rows, 32 heads, d_h 128, rank 48)."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_decode_bytes_of_the_bench_workload():
    import bench
    from compressed_cache_decode_gb300 import inputs
    w = inputs.WORKLOADS["decode_bf16_b8_h16_d64_r28_L4096"]
    lens = torch.full((w.batch,), w.max_len, dtype=torch.int32)
    total, split, cache = bench.decode_bytes(w, lens)
    assert cache == 8 * 4096 * 2 * (64 + 16 * 28) * 2 == 67_108_864
    assert split == 67_125_248
    assert total == split + 2 * 16 * 64 * 28 * 2 + 8 * 16 * 65 * 4
    w4 = inputs.WORKLOADS["decode_bf16_b4_h32_d128_r48_L65536_outliers"]
    total4, split4, cache4 = bench.decode_bytes(w4, torch.full((4,), 65536, dtype=torch.int32))
    assert cache4 == 4 * 65536 * 2 * (128 + 32 * 48) * 2 == 1_744_830_464
    assert split4 == cache4 + 4 * 32 * 128 * 2 == 1_744_863_232


def test_reference_arm_prints_the_contract_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
    d = json.loads(line)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "decode_bf16_b4_h32_d128_r48_L65536_outliers"
    assert d["config"]["pairs_per_step"] == d["cpu_baseline"]["cores"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
