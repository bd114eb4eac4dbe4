"""Canary regions around every output buffer of the compute calls.

Each output (and workspace) is the middle of a larger buffer whose first and
last 256 elements hold a NaN bit pattern no kernel produces; after the call
(synchronised) the guards must be bit-identical, and an output the call
writes in full must no longer hold the pattern anywhere.  Covers the decode
(bf16, fp32, paged, normalised keys, full RoPE, the decode step), the
prefill, the append, the key scales and the comparison decodes.
"""
import math

import numpy as np
import pytest
import torch

from _lib_util import ensure_built
from compressed_cache_decode_gb300 import inputs, lrkv

pytestmark = pytest.mark.gpu

G = 256                  # guard elements on each side
CANARY32 = 0x7FC0BEEF    # fp32 NaN with a payload
CANARY16 = 0x7FC5        # bf16 NaN with a payload


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    lrkv.load()


class Guarded:
    """A tensor of `shape` inside a buffer with G canary elements on each side."""

    def __init__(self, shape, dtype, fill=None):
        n = math.prod(shape)
        if dtype in (torch.float32, torch.int32):
            self.raw = torch.full((n + 2 * G,), CANARY32, dtype=torch.int32, device="cuda")
            self.canary = CANARY32
        elif dtype == torch.bfloat16:
            self.raw = torch.full((n + 2 * G,), CANARY16, dtype=torch.int16, device="cuda")
            self.canary = CANARY16
        else:
            raise TypeError(dtype)
        self.n = n
        self.t = self.raw[G:G + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, written_in_full=False, what=""):
        torch.cuda.synchronize()
        raw = self.raw.cpu().numpy()
        assert np.all(raw[:G] == np.array(self.canary, dtype=raw.dtype)), f"{what}: guard before overwritten"
        assert np.all(raw[G + self.n:] == np.array(self.canary, dtype=raw.dtype)), f"{what}: guard after overwritten"
        if written_in_full:
            assert not np.any(raw[G:G + self.n] == np.array(self.canary, dtype=raw.dtype)), f"{what}: not written"


def _dev(case):
    return {k: v.cuda() for k, v in case.items()}


def _decode_outputs(B, H, dh):
    return Guarded((B, H, dh), torch.float32), Guarded((B, H), torch.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode(dtype):
    shape = (3, 32, 128, 48, 300, [300, 1, 129]) if dtype == "bf16" else (1, 4, 16, 4, 64, [64])
    B, H, dh, r, L, lens = shape
    d = _dev(inputs.random_decode_case(seed=40, batch=B, heads=H, head_dim=dh, rank=r, max_len=L, dtype=dtype,
                                       lens=lens))
    dims = lrkv.make_dims(B, H, dh, r, L, torch.bfloat16 if dtype == "bf16" else torch.float32)
    nbytes = lrkv.lrkv_decode_workspace_size(dims)
    ws = Guarded(((nbytes + 1) // 2,), torch.bfloat16)  # the workspace's bytes as 2-byte elements
    out, lse = _decode_outputs(B, H, dh)
    st = lrkv.lrkv_decode(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], d["seq_lens"],
                          out.t, lse.t, ws.t, nbytes)
    assert st == lrkv.LRKV_OK
    out.check(True, "out")
    lse.check(True, "lse")
    ws.check(False, "workspace")


def test_decode_paged_and_normed():
    B, H, dh, r, L = 2, 16, 64, 28, 512
    case = inputs.random_decode_case(seed=41, batch=B, heads=H, head_dim=dh, rank=r, max_len=L, dtype="bf16",
                                     lens=[512, 200])
    d = _dev(case)
    paged = _dev(inputs.paged_from_contiguous(case, page_size=64, seed=3))
    out, lse = _decode_outputs(B, H, dh)
    lrkv.decode_paged(paged["q"], paged["k_s"], paged["v_s"], paged["z_k"], paged["z_v"], paged["b_k"],
                      paged["b_v"], paged["block_table"], paged["seq_lens"], out=out.t, lse=lse.t)
    out.check(True, "paged out")
    lse.check(True, "paged lse")
    ks = Guarded((B, H, L), torch.float32)
    lrkv.key_scales(d["k_s"], d["z_k"], d["b_k"], torch.zeros(B, dtype=torch.int32, device="cuda"), L, ks.t)
    ks.check(True, "key scales")
    out, lse = _decode_outputs(B, H, dh)
    lrkv.decode_normed(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], ks.t, d["seq_lens"],
                       out=out.t, lse=lse.t)
    out.check(True, "normed out")
    lse.check(True, "normed lse")


def test_decode_step_writes_only_its_rows_and_outputs():
    B, H, dh, r, L, dm = 2, 16, 64, 28, 256, 256
    case = inputs.random_decode_case(seed=42, batch=B, heads=H, head_dim=dh, rank=r, max_len=L, dtype="bf16",
                                     lens=[256, 100])
    d = _dev(case)
    gen = torch.Generator(device="cuda").manual_seed(5)
    w = [(torch.randn(n, dm, generator=gen, device="cuda") * dm ** -0.5).to(torch.bfloat16)
         for n in (dh, dh, H * r, H * r)]
    x = torch.randn(B, dm, generator=gen, device="cuda").to(torch.bfloat16)
    caches = {k: Guarded(tuple(d[k].shape), torch.bfloat16, fill=d[k]) for k in ("k_s", "v_s", "z_k", "z_v")}
    out, lse = _decode_outputs(B, H, dh)
    lrkv.decode_step(x, *w, d["q"], caches["k_s"].t, caches["v_s"].t, caches["z_k"].t, caches["z_v"].t, d["b_k"],
                     d["b_v"], d["seq_lens"], out=out.t, lse=lse.t)
    out.check(True, "step out")
    lse.check(True, "step lse")
    for k, g in caches.items():
        g.check(False, f"step cache {k}")


def test_decode_rope_and_comparisons():
    B, H, dh, r, L = 2, 16, 64, 32, 256
    d = _dev(inputs.random_decode_case(seed=43, batch=B, heads=H, head_dim=dh, rank=r, max_len=L, dtype="bf16",
                                       lens=[256, 31]))
    cs = lrkv.rope_table(L, dh)
    out, lse = _decode_outputs(B, H, dh)
    lrkv.decode_rope(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], cs, d["seq_lens"],
                     out=out.t, lse=lse.t)
    out.check(True, "rope out")
    lse.check(True, "rope lse")
    dd = _dev(inputs.random_dense_case(seed=44, batch=B, heads=H, kv_heads=2, head_dim=128, max_len=L,
                                       lens=[256, 77]))
    out, lse = _decode_outputs(B, H, 128)
    lrkv.dense_decode(dd["q"], dd["k"], dd["v"], dd["seq_lens"], out=out.t, lse=lse.t)
    out.check(True, "dense out")
    lse.check(True, "dense lse")
    md = _dev(inputs.random_mla_case(seed=45, batch=B, heads=H, head_dim=128, latent_dim=512, max_len=L,
                                     lens=[256, 77]))
    out, lse = _decode_outputs(B, H, 128)
    lrkv.mla_decode(md["q"], md["c"], md["w_uk"], md["w_uv"], md["seq_lens"], out=out.t, lse=lse.t)
    out.check(True, "mla out")
    lse.check(True, "mla lse")


def test_prefill_and_append():
    B, Tq, H, dh, r, L = 2, 130, 4, 128, 64, 300
    d = _dev(inputs.random_prefill_case(seed=46, batch=B, q_len=Tq, heads=H, head_dim=dh, rank=r, max_len=L,
                                        lens=[300, 180]))
    out = Guarded((B, Tq, H, dh), torch.float32)
    lse = Guarded((B, H, Tq), torch.float32)
    lrkv.prefill(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], d["seq_lens"],
                 out=out.t, lse=lse.t)
    out.check(True, "prefill out")
    lse.check(True, "prefill lse")
    # append 96 rows at rows 64.. of both sequences; the rest of each cache keeps its contents
    dm, n_new = 256, 96
    gen = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn(B, n_new, dm, generator=gen, device="cuda").to(torch.bfloat16)
    w = [(torch.randn(n, dm, generator=gen, device="cuda") * dm ** -0.5).to(torch.bfloat16)
         for n in (dh, dh, H * r, H * r)]
    caches = {k: Guarded(tuple(d[k].shape), torch.bfloat16, fill=d[k]) for k in ("k_s", "v_s", "z_k", "z_v")}
    status = lrkv.append(x, *w, torch.full((B,), 64, dtype=torch.int32, device="cuda"), caches["k_s"].t,
                         caches["v_s"].t, caches["z_k"].t, caches["z_v"].t)
    assert status == lrkv.LRKV_OK
    for k, g in caches.items():
        g.check(False, f"append cache {k}")
