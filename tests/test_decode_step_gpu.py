"""Decode step parity: the new token's cache rows from x (review §3 Algorithm
1 for one token) and the decode over the cache that holds them (Algorithm 2),
against the fp64 oracle.  Rows: within one bf16 ulp of the float64 product plus
the fp32 accumulation bound (as for the append); outputs: the bf16 decode bar,
evaluated on the GPU-written cache."""
import numpy as np
import pytest
import torch

from _lib_util import assert_decode_close, ensure_built
from compressed_cache_decode_gb300 import inputs, lrkv
from oracle import lrkv_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    lrkv.load()


def _ulp_bf16(x):
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def _weights(seed, B, d, H, dh, r):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, d, generator=g).to(torch.bfloat16)
    w = [(torch.randn(n, d, generator=g) / d ** 0.5).to(torch.bfloat16) for n in (dh, dh, H * r, H * r)]
    return x, w


def _run_step(case, x, w):
    dev = {k: v.cuda() for k, v in case.items()}
    xd = x.cuda()
    wd = [t.cuda() for t in w]
    out, lse = lrkv.decode_step(xd, *wd, dev["q"], dev["k_s"], dev["v_s"], dev["z_k"], dev["z_v"],
                                dev["b_k"], dev["b_v"], dev["seq_lens"])
    torch.cuda.synchronize()
    cache = {k: dev[k].cpu() for k in ("k_s", "v_s", "z_k", "z_v")}
    return out.cpu().numpy(), lse.cpu().numpy(), cache


def _check_rows(cache, case, x, w, lens, H):
    ref = O.append_reference(x[:, None, :], w[0].t(), w[1].t(), w[2].t(), w[3].t(), H)
    ab = O.append_reference(x.abs()[:, None, :], w[0].abs().t(), w[1].abs().t(), w[2].abs().t(),
                            w[3].abs().t(), H)
    d = x.shape[-1]
    for b, L in enumerate(lens):
        for name, rf, a in zip(("k_s", "v_s", "z_k", "z_v"), ref, ab):
            before = case[name][b]
            after = cache[name][b]
            if L >= 1:
                got = after[L - 1].float().numpy().astype(np.float64)
                err = np.abs(got - rf[b, 0])
                tol = _ulp_bf16(rf[b, 0]) * 1.0000001 + d * 2.0 ** -24 * a[b, 0]
                assert (err <= tol).all(), f"{name} seq {b}: worst {err.max():.3e}"
            keep = torch.ones(before.shape[0], dtype=torch.bool)
            if L >= 1:
                keep[L - 1] = False
            assert torch.equal(before[keep], after[keep]), f"{name} seq {b}: other rows changed"


@pytest.mark.parametrize("shape", [
    # B, H, d_h, r, d_model, max_len, lengths (including the new token)
    (3, 4, 64, 16, 256, 200, [57, 120, 1]),
    (2, 8, 128, 32, 512, 300, [300, 129]),        # the row at the last cache position
    (4, 16, 64, 28, 1024, 4096, [4096, 3000, 17, 2048]),
    (12, 4, 64, 16, 256, 96, [5, 96, 1, 40, 77, 12, 64, 65, 3, 90, 33, 18]),   # 16 sequences per pass
    (20, 4, 64, 16, 128, 64, list(range(1, 21))),                         # two passes over the weights
])
def test_decode_step_matches_oracle(shape):
    B, H, dh, r, d, Lm, lens = shape
    case = inputs.random_decode_case(seed=B * 31 + d, batch=B, heads=H, head_dim=dh, rank=r, max_len=Lm,
                                     dtype="bf16", lens=lens)
    x, w = _weights(B + d, B, d, H, dh, r)
    out, lse, cache = _run_step(case, x, w)
    _check_rows(cache, case, x, w, lens, H)
    ref_o, ref_l = O.decode_reference(case["q"], cache["k_s"], cache["v_s"], cache["z_k"], cache["z_v"],
                                      case["b_k"], case["b_v"], case["seq_lens"])
    assert_decode_close(out, lse, ref_o, ref_l, "bf16", what=f"decode step {shape}")


def test_decode_step_empty_sequence_writes_nothing():
    B, H, dh, r, d, Lm = 2, 4, 64, 16, 128, 64
    lens = [0, 40]
    case = inputs.random_decode_case(seed=9, batch=B, heads=H, head_dim=dh, rank=r, max_len=Lm,
                                     dtype="bf16", lens=lens)
    x, w = _weights(9, B, d, H, dh, r)
    out, lse, cache = _run_step(case, x, w)
    _check_rows(cache, case, x, w, lens, H)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
