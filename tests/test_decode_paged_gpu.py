"""Decode and causal prefill over a paged factored cache against the fp64 oracle: the cache rows
of every sequence sit in pages of a shared pool in a seeded random order
(unused pages and rows hold NaN), a block table maps each sequence's blocks;
the result must match the decode over the logical rows and the
contiguous-cache decode of the same rows (the bf16 decode bar); a block table
entry outside the pool is flagged and leaves the other sequences correct."""
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
    # B, H, d_h, r, page_size, max_len, lengths
    (3, 16, 64, 28, 16, 320, [300, 1, 77]),
    (2, 32, 128, 48, 64, 512, [500, 129]),          # two row tiles, a partial last page
    (4, 8, 64, 8, 256, 1024, [1000, 0, 256, 257]),  # an empty history, a page boundary +-1
    (5, 18, 64, 8, 32, 96, [1, 2, 3, 96, 65]),      # several pieces per CTA, a partial row tile
])
def test_paged_decode_matches_oracle(shape):
    B, H, dh, r, ps, Lm, lens = shape
    case = inputs.random_decode_case(seed=B * 17 + ps, batch=B, heads=H, head_dim=dh, rank=r, max_len=Lm,
                                     dtype="bf16", lens=lens)
    paged = inputs.paged_from_contiguous(case, page_size=ps, seed=ps + B)
    d = {k: v.cuda() for k, v in paged.items()}
    out, lse, ws = lrkv.decode_paged(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                                     d["block_table"], d["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    ref_o, ref_l = O.decode_reference_paged(paged["q"], paged["k_s"], paged["v_s"], paged["z_k"], paged["z_v"],
                                            paged["b_k"], paged["b_v"], paged["block_table"], ps,
                                            paged["seq_lens"])
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", what=f"paged {shape}")
    # the same rows in a contiguous cache decode to the same result within the
    # bf16 bar (a paged call lays its first tiles on the 16-row grid of each
    # sequence, so the summation order can differ)
    c = {k: v.cuda() for k, v in case.items()}
    out_c, lse_c = lrkv.decode(c["q"], c["k_s"], c["v_s"], c["z_k"], c["z_v"], c["b_k"], c["b_v"], c["seq_lens"])
    torch.cuda.synchronize()
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), out_c.cpu().numpy().astype(np.float64),
                        lse_c.cpu().numpy().astype(np.float64), "bf16", what=f"paged vs contiguous {shape}")


def test_paged_decode_flags_a_page_outside_the_pool():
    B, H, dh, r, ps, Lm = 2, 16, 64, 28, 32, 128
    case = inputs.random_decode_case(seed=3, batch=B, heads=H, head_dim=dh, rank=r, max_len=Lm, dtype="bf16",
                                     lens=[100, 40])
    paged = inputs.paged_from_contiguous(case, page_size=ps, seed=4)
    d = {k: v.cuda() for k, v in paged.items()}
    d["block_table"][1, 0] = d["k_s"].shape[0] + 5          # past the pool
    out, lse, ws = lrkv.decode_paged(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                                     d["block_table"], d["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_ERR_DEVICE_BOUNDS
    assert torch.isfinite(out[0]).all()                       # the other sequence is unaffected
    ref_o, ref_l = O.decode_reference(paged["q"][:1], case["k_s"][:1], case["v_s"][:1], case["z_k"][:1],
                                      case["z_v"][:1], case["b_k"], case["b_v"], case["seq_lens"][:1])
    assert_decode_close(out[:1].cpu().numpy(), lse[:1].cpu().numpy(), ref_o, ref_l, "bf16", what="valid sequence")


@pytest.mark.parametrize("shape", [
    # B, q_len, H, page_size, max_len, lengths
    (2, 200, 3, 128, 512, [200, 450]),        # a prefix of 250 cached rows before the second chunk
    (1, 128, 2, 256, 512, [384]),             # the chunk starts on a page boundary
    (2, 512, 40, 128, 768, [512, 700]),       # more items than SMs
])
def test_paged_prefill_matches_oracle(shape):
    B, Tq, H, ps, Lm, lens = shape
    case = inputs.random_prefill_case(seed=B * 3 + Tq, batch=B, q_len=Tq, heads=H, head_dim=128, rank=64,
                                      max_len=Lm, lens=lens)
    paged = inputs.paged_from_contiguous(case, page_size=ps, seed=Tq + ps)
    d = {k: v.cuda() for k, v in paged.items()}
    out, lse, ws = lrkv.prefill_paged(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                                      d["block_table"], d["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    ref_o, ref_l = O.prefill_reference_paged(paged["q"], paged["k_s"], paged["v_s"], paged["z_k"], paged["z_v"],
                                             paged["b_k"], paged["b_v"], paged["block_table"], ps,
                                             paged["seq_lens"])
    o, l_ = out.cpu().numpy(), lse.cpu().numpy()
    assert_decode_close(o.reshape(-1, o.shape[-1]), l_.transpose(0, 2, 1).reshape(-1),
                        ref_o.reshape(-1, ref_o.shape[-1]), ref_l.transpose(0, 2, 1).reshape(-1), "bf16",
                        what=f"paged prefill {shape}")
