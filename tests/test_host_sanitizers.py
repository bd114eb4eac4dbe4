"""The C ABI's host side under AddressSanitizer and UndefinedBehaviorSanitizer.

Builds the library's sources with the host compiler's sanitizers (device code
as PTX only: nothing is launched) and links them with `host_checks.cpp`,
which exercises status strings, cache accounting, the launch planning behind
every workspace-size query over a grid of shapes (LRKV_SM_COUNT stands in
for a device; the default plans and the planner's tuning branches) and the
argument checks of every compute entry point.  Any
sanitizer report or failed expectation fails the test.  Runs on the CPU machine.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "compressed_cache_decode_gb300", "csrc")
SAN = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",
       "-Xcompiler", "-fno-sanitize-recover=undefined", "-Xcompiler", "-fno-omit-frame-pointer"]
COMMON = ["-O1", "-g", "-std=c++17", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
PTX_ONLY = ["-gencode", "arch=compute_103a,code=compute_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_host_side_under_asan_and_ubsan(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    srcs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))

    def compile_one(src):
        obj = str(tmp_path / (os.path.basename(src) + ".o"))
        cmd = [nvcc, *PTX_ONLY, *COMMON, "-Xcompiler", "-fPIC", *SAN, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        assert res.returncode == 0, f"nvcc failed on {src}:\n{res.stderr[-2000:]}"
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    drv_obj = str(tmp_path / "host_checks.o")
    res = subprocess.run([nvcc, *COMMON, *SAN, "-c", os.path.join(HERE, "host_checks.cpp"), "-o", drv_obj],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    exe = str(tmp_path / "host_checks")
    res = subprocess.run([nvcc, *PTX_ONLY, *SAN, "-o", exe, drv_obj, *objs], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    base = dict(os.environ, LRKV_SM_COUNT="152",
                ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0:abort_on_error=0",
                UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    # the default plans, then the planner's tuning branches (the narrow merge,
    # B^K in registers, an L2 window) and another SM count
    for extra in ({}, {"LRKV_DECODE_WIDE_MERGE": "0", "LRKV_DECODE_BK_REGS": "1", "LRKV_DECODE_PREFETCH_TILES": "4"},
                  {"LRKV_SM_COUNT": "148"}):
        run = subprocess.run([exe], capture_output=True, text=True, env=dict(base, **extra), timeout=300)
        report = run.stdout + run.stderr
        assert run.returncode == 0, f"{extra}: " + report[-4000:]
        assert "runtime error" not in report and "AddressSanitizer" not in report, f"{extra}: " + report[-4000:]
        assert "host checks ok" in run.stdout, extra
