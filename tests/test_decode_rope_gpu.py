"""Full-RoPE decode parity: the CUDA path (through the C ABI) against the
fp64 oracle's decode_reference_rope on seeded inputs ("Low-Rank Key Value
Attention | What a shared cache can preserve", §8, "Full RoPE needs a
stronger identity").  The cache holds unrotated rows; the query is given
rotated; the library's rotation table is checked against cos and sin of
j theta_k computed here in fp64.  Small cases compare every output; the
long-context workload compares sampled (sequence, head) pairs in the launch
configuration the bench times."""
import math

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


def test_rotation_table_matches_fp64_cos_sin():
    for max_pos, dh, base in ((4096, 128, 10000.0), (300, 64, 500.0)):
        t = lrkv.rope_table(max_pos, dh, base).cpu().numpy().astype(np.float64)
        k = np.arange(dh // 2)
        ang = np.outer(np.arange(max_pos), base ** (-2.0 * k / dh))
        assert np.max(np.abs(t[:, 0::2] - np.cos(ang))) <= 1e-7
        assert np.max(np.abs(t[:, 1::2] - np.sin(ang))) <= 1e-7


def _run(case, table, stream=None):
    d = {k: v.cuda() for k, v in case.items()}
    out, lse = lrkv.decode_rope(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], table,
                                d["seq_lens"], stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("shape", [
    # (B, H, d_h, r, max_len, lens)
    (2, 16, 64, 32, 300, [300, 77]),
    (3, 32, 128, 48, 500, [500, 1, 257]),
    (2, 8, 128, 64, 200, [200, 0]),          # an empty history
    (1, 8, 64, 16, 40, [40]),
    (5, 16, 128, 48, 90, [1, 2, 3, 90, 89]),  # many short pieces in one range
])
def test_rope_random_shapes(shape):
    B, H, dh, r, L, lens = shape
    case = inputs.random_decode_case(seed=B * 100 + H + r + L, batch=B, heads=H, head_dim=dh, rank=r, max_len=L,
                                     dtype="bf16", lens=lens)
    table = lrkv.rope_table(L, dh)
    out, lse = _run(case, table)
    ref_o, ref_l = O.decode_reference_rope(*(case[k] for k in ("q", "k_s", "v_s", "z_k", "z_v", "b_k", "b_v",
                                                              "seq_lens")))
    assert_decode_close(out, lse, ref_o, ref_l, "bf16", what=f"rope {shape}")
    for b, Lb in enumerate(lens):
        if Lb == 0:
            assert np.all(out[b] == 0.0)
    # the rotation matters: the plain decode of the same inputs differs
    if max(lens) > 8:
        plain_o, _ = O.decode_reference(*(case[k] for k in ("q", "k_s", "v_s", "z_k", "z_v", "b_k", "b_v",
                                                           "seq_lens")))
        assert np.max(np.abs(plain_o - ref_o)) > 10 * (1e-2 * np.max(np.abs(ref_o)) + 1e-3)


def test_rope_long_context_sampled_pairs():
    """The long-context workload (4 x 65,536 rows, 32 heads, d_h 128, rank 48,
    5% of the shared key rows x8) with a rotated query, on sampled pairs."""
    w = inputs.WORKLOADS["decode_bf16_b4_h32_d128_r48_L65536_outliers"]
    case = inputs.make_decode_inputs(w, seed=0)
    table = lrkv.rope_table(w.max_len, w.head_dim)
    out, lse = _run(case, table)
    rng = np.random.default_rng(3)
    pairs = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, w.batch, 6), rng.integers(0, w.heads, 6))}
                   | {(0, 0), (w.batch - 1, w.heads - 1)})
    ref_o, ref_l = O.decode_reference_rope(*(case[k] for k in ("q", "k_s", "v_s", "z_k", "z_v", "b_k", "b_v",
                                                              "seq_lens")), pairs=pairs)
    mask = np.zeros((w.batch, w.heads), dtype=bool)
    for b, h in pairs:
        mask[b, h] = True
    assert_decode_close(out, lse, ref_o, ref_l, "bf16", mask=mask, what="rope long context")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_rope_workspace_too_small_enqueues_nothing():
    case = inputs.random_decode_case(seed=9, batch=1, heads=8, head_dim=64, rank=32, max_len=64, dtype="bf16")
    d = {k: v.cuda() for k, v in case.items()}
    dims = lrkv.make_dims(1, 8, 64, 32, 64, torch.bfloat16)
    n = lrkv.lrkv_decode_rope_workspace_size(dims)
    ws = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    table = lrkv.rope_table(64, 64)
    out = torch.full((1, 8, 64), 3.0, device="cuda")
    st = lrkv.lrkv_decode_rope(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], table, 64,
                               d["seq_lens"], out, None, ws, n - 16)
    torch.cuda.synchronize()
    assert st == lrkv.LRKV_ERR_WORKSPACE and bool(torch.all(out == 3.0))
