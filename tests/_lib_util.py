"""Helpers shared by the tests: build-on-demand of the CUDA library and the
parity assertions (tolerances of the decode/prefill contract)."""
import os
import re
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADER = os.path.join(ROOT, "include", "lrkv.h")


def ensure_built():
    from compressed_cache_decode_gb300 import build
    return build.build()


def header_symbols():
    """Function names declared in include/lrkv.h."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lrkv_[a-z0-9_]+)\s*\(", text)))


def gpu_available():
    return torch.cuda.is_available()


# Tolerances: fp32 storage -> max|err| <= 1e-5 * max|o_ref|; bf16 storage with
# fp32 accumulation -> max|err| <= 1e-2 * max|o_ref| + 1e-3 and per-row
# |lse - lse_ref| <= 2e-3 (natural log).
def assert_decode_close(out, lse, out_ref, lse_ref, dtype, mask=None, what=""):
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    if mask is not None:
        out, out_ref = out[mask], out_ref[mask]
        lse, lse_ref = lse[mask], lse_ref[mask]
    finite = np.isfinite(lse_ref)
    scale = np.max(np.abs(out_ref)) if out_ref.size else 0.0
    err = np.max(np.abs(out - out_ref)) if out_ref.size else 0.0
    if dtype == "f32":
        tol = 1e-5 * scale
        lse_tol = 1e-5
    else:
        tol = 1e-2 * scale + 1e-3
        lse_tol = 2e-3
    assert err <= tol, f"{what}: max|o - o_ref| = {err:.3e} > {tol:.3e}"
    # empty histories: out exactly 0 and lse = -inf
    assert np.all(np.isneginf(lse[~finite])), f"{what}: lse of empty history must be -inf"
    if np.any(finite):
        lerr = np.max(np.abs(lse[finite] - lse_ref[finite]))
        assert lerr <= lse_tol, f"{what}: max|lse - lse_ref| = {lerr:.3e} > {lse_tol:.1e}"
    return err, tol
