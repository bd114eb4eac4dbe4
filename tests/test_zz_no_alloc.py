"""The allocation-free decode entry point against the workspace entry point.

lrkv_decode_static_scratch serves callers that cannot allocate device memory
when they call into the library (for example a plugin whose host runtime owns
every device allocation, or a serving path that must not allocate mid-request):
it takes its workspace from an array compiled into the library.  These tests
call it through the C ABI twice in a row and compare each result with
lrkv_decode on a caller-allocated workspace, within the bf16 tolerance the
decode parity tests use.  The file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from _lib_util import assert_decode_close, ensure_built
from compressed_cache_decode_gb300 import inputs, lrkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    lrkv.load()


def _workspace_path(d, dims):
    ws = lrkv.decode_workspace(dims, "cuda")
    out = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    st = lrkv.lrkv_decode(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                          d["seq_lens"], out, lse, ws, ws.numel())
    assert st == lrkv.LRKV_OK, lrkv.status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _static_path(d, dims):
    out = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    st = lrkv.lrkv_decode_static_scratch(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"],
                                         d["b_k"], d["b_v"], d["seq_lens"], out, lse)
    assert st == lrkv.LRKV_OK, lrkv.status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def test_static_scratch_matches_workspace_entry_point_twice():
    cases = [
        inputs.random_decode_case(seed=11, batch=3, heads=16, head_dim=64, rank=28, max_len=300,
                                  dtype="bf16", lens=[300, 1, 129]),
        inputs.random_decode_case(seed=12, batch=2, heads=32, head_dim=128, rank=48, max_len=200,
                                  dtype="bf16", lens=[200, 77]),
    ]
    for case in cases:  # two calls in a row, different shapes, same array
        d = {k: v.cuda() for k, v in case.items()}
        B, H, dh = case["q"].shape
        dims = lrkv.make_dims(B, H, dh, case["z_k"].shape[-1], case["k_s"].shape[1], torch.bfloat16)
        ref_o, ref_l = _workspace_path(d, dims)
        out, lse = _static_path(d, dims)
        assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
        assert_decode_close(out, lse, ref_o.astype(np.float64), ref_l.astype(np.float64), "bf16",
                            what="static scratch vs workspace")


def test_static_scratch_fp32_and_status():
    # the fp32 path (tile-synchronous kernels: its absorb kernel writes q B^K
    # and clears the status word in the array), then the status reader
    case = inputs.random_decode_case(seed=13, batch=1, heads=4, head_dim=16, rank=4, max_len=64, dtype="f32",
                                     lens=[64])
    d = {k: v.cuda() for k, v in case.items()}
    dims = lrkv.make_dims(1, 4, 16, 4, 64, torch.float32)
    ref_o, ref_l = _workspace_path(d, dims)
    out, lse = _static_path(d, dims)
    assert_decode_close(out, lse, ref_o.astype(np.float64), ref_l.astype(np.float64), "f32",
                        what="static scratch vs workspace (fp32)")
    assert lrkv.lrkv_read_static_scratch_status() == lrkv.LRKV_OK
    # a length past max_len is clamped and reported through the array's status word
    d["seq_lens"][0] = 65
    _static_path(d, dims)
    assert lrkv.lrkv_read_static_scratch_status() == lrkv.LRKV_ERR_DEVICE_BOUNDS


def test_static_scratch_back_to_back_on_one_stream():
    # two calls enqueued with no synchronisation between them (the second
    # call's scan is launched while the first call's merge may still run),
    # separate outputs, one synchronisation, both compared with the workspace path
    cases = [inputs.random_decode_case(seed=20 + i, batch=4, heads=16, head_dim=64, rank=28, max_len=1024,
                                       dtype="bf16", lens=[1024, 700, 33, 512]) for i in range(2)]
    devs = [{k: v.cuda() for k, v in c.items()} for c in cases]
    dims = lrkv.make_dims(4, 16, 64, 28, 1024, torch.bfloat16)
    refs = [_workspace_path(d, dims) for d in devs]
    outs = []
    for d in devs:
        out = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        st = lrkv.lrkv_decode_static_scratch(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"],
                                             d["b_k"], d["b_v"], d["seq_lens"], out, lse)
        assert st == lrkv.LRKV_OK, lrkv.status_string(st)
        outs.append((out, lse))
    torch.cuda.synchronize()
    for (out, lse), (ref_o, ref_l) in zip(outs, refs):
        assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o.astype(np.float64),
                            ref_l.astype(np.float64), "bf16", what="back-to-back static scratch")
    assert lrkv.lrkv_read_static_scratch_status() == lrkv.LRKV_OK


def test_static_scratch_rejects_oversized_workspace():
    # 4096 sequences x 64K rows of H=64 heads needs far more than the array holds
    dims = lrkv.make_dims(4096, 64, 64, 8, 65536, torch.bfloat16)
    assert lrkv.lrkv_decode_workspace_size(dims) > 16 * 1024 * 1024
    fake = 1 << 20  # never dereferenced: the size check comes first
    st = lrkv.load().lrkv_decode_static_scratch(
        ctypes.byref(dims), fake, fake, fake, fake, fake, fake, fake, fake, fake, None, None)
    assert st == lrkv.LRKV_ERR_WORKSPACE
