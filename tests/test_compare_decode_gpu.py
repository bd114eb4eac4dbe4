"""Parity of the comparison decodes on the same box (review §4-§5): dense
MHA/GQA/MQA over materialised K/V against the oracle's
dense_decode_reference, and absorbed MLA against mla_decode_reference (keys
and values rebuilt from the latent rows), through the C ABI, on seeded
inputs including ragged and empty histories."""
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


@pytest.mark.parametrize("shape", [
    # (B, H, H_kv, d, max_len, lens)
    (2, 8, 8, 128, 300, [300, 77]),          # MHA
    (3, 16, 4, 64, 257, [257, 0, 100]),      # GQA, group 4, an empty history
    (2, 32, 16, 128, 200, [200, 33]),        # GQA, group 2
    (2, 32, 4, 128, 150, [150, 149]),        # GQA, group 8
    (4, 8, 1, 64, 90, [1, 2, 90, 89]),       # MQA, short pieces
])
def test_dense_decode_matches_oracle(shape):
    B, H, Hkv, d, L, lens = shape
    case = inputs.random_dense_case(seed=B + H + Hkv + d + L, batch=B, heads=H, kv_heads=Hkv, head_dim=d, max_len=L,
                                    lens=lens)
    dv = {k: t.cuda() for k, t in case.items()}
    out, lse, ws = lrkv.dense_decode(dv["q"], dv["k"], dv["v"], dv["seq_lens"])
    torch.cuda.synchronize()
    ref_o, ref_l = O.dense_decode_reference(case["q"], case["k"], case["v"], case["seq_lens"])
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", what=f"dense {shape}")
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK


@pytest.mark.parametrize("shape", [
    # (B, H, d_h, d_c, max_len, lens)
    (2, 32, 128, 512, 300, [300, 77]),
    (3, 16, 64, 256, 200, [200, 0, 17]),     # an empty history
    (2, 8, 128, 512, 1000, [1000, 999]),
])
def test_mla_decode_matches_oracle(shape):
    B, H, dh, dc, L, lens = shape
    case = inputs.random_mla_case(seed=B + H + dh + dc + L, batch=B, heads=H, head_dim=dh, latent_dim=dc, max_len=L,
                                  lens=lens)
    dv = {k: t.cuda() for k, t in case.items()}
    out, lse, ws = lrkv.mla_decode(dv["q"], dv["c"], dv["w_uk"], dv["w_uv"], dv["seq_lens"])
    torch.cuda.synchronize()
    ref_o, ref_l = O.mla_decode_reference(case["q"], case["c"], case["w_uk"], case["w_uv"], case["seq_lens"])
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", what=f"mla {shape}")
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK


def test_compare_long_context_sampled_pairs():
    """The long-context batch and length (4 x 65,536 rows) for GQA-8 and MLA-512,
    sampled (sequence, head) pairs."""
    rng = np.random.default_rng(5)
    pairs = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, 4, 5), rng.integers(0, 32, 5))} | {(3, 31)})
    mask = np.zeros((4, 32), dtype=bool)
    for b, h in pairs:
        mask[b, h] = True
    case = inputs.random_dense_case(seed=1, batch=4, heads=32, kv_heads=8, head_dim=128, max_len=65536,
                                    lens=[65536] * 4)
    dv = {k: t.cuda() for k, t in case.items()}
    out, lse, _ = lrkv.dense_decode(dv["q"], dv["k"], dv["v"], dv["seq_lens"])
    torch.cuda.synchronize()
    ref_o, ref_l = O.dense_decode_reference(case["q"], case["k"], case["v"], case["seq_lens"], pairs=pairs)
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", mask=mask, what="gqa long")
    del case, dv
    mcase = inputs.random_mla_case(seed=2, batch=4, heads=32, head_dim=128, latent_dim=512, max_len=65536,
                                   lens=[65536] * 4)
    mv = {k: t.cuda() for k, t in mcase.items()}
    out, lse, _ = lrkv.mla_decode(mv["q"], mv["c"], mv["w_uk"], mv["w_uv"], mv["seq_lens"])
    torch.cuda.synchronize()
    ref_o, ref_l = O.mla_decode_reference(mcase["q"], mcase["c"], mcase["w_uk"], mcase["w_uv"], mcase["seq_lens"],
                                          pairs=pairs)
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", mask=mask, what="mla long")
