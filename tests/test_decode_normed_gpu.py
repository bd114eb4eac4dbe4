"""Post-projection RMSNorm of the keys (review §8, "Post-projection
normalization has a cache cost") against the fp64 oracle: the cached joint
reciprocal scales (fp32; relative error from the fp32 rebuild of each key),
the decode and the causal prefill that multiply each summed score by its
key's scale (the bf16 decode bar)."""
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
    # B, H, d_h, r, max_len, start positions, n_new, eps
    (2, 4, 64, 16, 200, [0, 37], 150, 1e-6),
    (1, 8, 128, 64, 130, [0], 130, 1e-3),     # two 64-token blocks + a ragged one
    (3, 16, 64, 28, 96, [5, 90, 0], 20, 0.0),  # rows past max_len skipped
    (2, 36, 128, 48, 700, [0, 250], 512, 1e-6),  # rank padded to 64 by the copy, a partial head group
])
@pytest.mark.parametrize("tc", ["1", "0"])  # the tcgen05 form (where it applies) and the mma.sync form
def test_key_scales_match_oracle(shape, tc, monkeypatch):
    monkeypatch.setenv("LRKV_KEY_SCALE_TC", tc)
    B, H, dh, r, Lm, start, n_new, eps = shape
    case = inputs.random_decode_case(seed=B * 11 + dh, batch=B, heads=H, head_dim=dh, rank=r, max_len=Lm,
                                     dtype="bf16")
    dev = {k: v.cuda() for k, v in case.items()}
    ks = torch.full((B, H, Lm), -1.0, dtype=torch.float32, device="cuda")
    sp = torch.tensor(start, dtype=torch.int32, device="cuda")
    lrkv.key_scales(dev["k_s"], dev["z_k"], dev["b_k"], sp, n_new, ks, eps=eps)
    torch.cuda.synchronize()
    got = ks.cpu().numpy().transpose(0, 2, 1)           # [B, L, H] like the oracle
    ref = O.key_rms_scales(case["k_s"], case["z_k"], case["b_k"], eps)
    for b in range(B):
        lo, hi = max(start[b], 0), min(start[b] + n_new, Lm)
        rel = np.abs(got[b, lo:hi] - ref[b, lo:hi]) / np.abs(ref[b, lo:hi])
        assert rel.max() <= 2e-5, f"seq {b}: worst relative error {rel.max():.2e}"
        assert np.all(got[b, :lo] == -1.0) and np.all(got[b, hi:] == -1.0), f"seq {b}: rows outside written"


@pytest.mark.parametrize("shape", [
    # B, H, d_h, r, max_len, lengths
    (3, 4, 64, 16, 200, [57, 120, 1]),
    (2, 8, 128, 32, 300, [300, 129]),
    (4, 16, 64, 28, 4096, [4096, 3000, 17, 0]),
    (6, 18, 64, 8, 80, [1, 2, 3, 80, 79, 5]),     # several pieces per CTA, a partial row tile
    (2, 32, 128, 48, 1024, [1024, 777]),          # two row tiles; scales staged with the tiles
    (2, 16, 64, 28, 301, [301, 150]),             # max_len not a multiple of 4: per-lane scale loads
])
def test_decode_normed_matches_oracle(shape):
    B, H, dh, r, Lm, lens = shape
    eps = 1e-6
    case = inputs.random_decode_case(seed=B * 13 + Lm, batch=B, heads=H, head_dim=dh, rank=r, max_len=Lm,
                                     dtype="bf16", lens=lens)
    dev = {k: v.cuda() for k, v in case.items()}
    ks = torch.empty((B, H, Lm), dtype=torch.float32, device="cuda")
    lrkv.key_scales(dev["k_s"], dev["z_k"], dev["b_k"], torch.zeros(B, dtype=torch.int32, device="cuda"), Lm, ks,
                    eps=eps)
    out, lse = lrkv.decode_normed(dev["q"], dev["k_s"], dev["v_s"], dev["z_k"], dev["z_v"], dev["b_k"], dev["b_v"],
                                  ks, dev["seq_lens"])
    torch.cuda.synchronize()
    ref_o, ref_l = O.decode_reference_normed(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"],
                                             case["b_k"], case["b_v"], case["seq_lens"], eps)
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16",
                        what=f"normed decode {shape}")
    # the normalisation matters here: the plain decode is far from the normed reference
    plain, _ = lrkv.decode(dev["q"], dev["k_s"], dev["v_s"], dev["z_k"], dev["z_v"], dev["b_k"], dev["b_v"],
                           dev["seq_lens"])
    live = np.asarray(lens) > 1
    assert np.abs(plain.cpu().numpy()[live] - ref_o[live]).max() > 1e-2


@pytest.mark.parametrize("shape", [
    # B, q_len, H, L per sequence, max_len
    (1, 128, 2, [128], 128),
    (2, 200, 3, [200, 450], 452),        # partial query tile, history before the queries, a key
                                         # tile past max_len (vector and shuffled scale reads)
    (1, 130, 2, [301], 301),             # max_len not a multiple of 4: shuffled scale reads only
    (2, 512, 40, [512, 700], 768),       # more items than SMs: several per persistent CTA
])
def test_prefill_normed_matches_oracle(shape):
    B, Tq, H, lens, Lm = shape
    eps = 1e-6
    case = inputs.random_prefill_case(seed=B * 7 + Tq, batch=B, q_len=Tq, heads=H, head_dim=128, rank=64,
                                      max_len=Lm, lens=lens)
    dev = {k: v.cuda() for k, v in case.items()}
    ks = torch.empty((B, H, Lm), dtype=torch.float32, device="cuda")
    lrkv.key_scales(dev["k_s"], dev["z_k"], dev["b_k"], torch.zeros(B, dtype=torch.int32, device="cuda"), Lm, ks,
                    eps=eps)
    for b, L in enumerate(lens):
        ks[b, :, L:] = float("nan")      # scales past the history are never used
    out, lse, ws = lrkv.prefill_normed(dev["q"], dev["k_s"], dev["v_s"], dev["z_k"], dev["z_v"], dev["b_k"],
                                       dev["b_v"], ks, dev["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    ref_o, ref_l = O.prefill_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"],
                                       case["b_k"], case["b_v"], case["seq_lens"], rms_eps=eps)
    o, l_ = out.cpu().numpy(), lse.cpu().numpy()
    assert_decode_close(o.reshape(-1, o.shape[-1]), l_.transpose(0, 2, 1).reshape(-1),
                        ref_o.reshape(-1, ref_o.shape[-1]), ref_l.transpose(0, 2, 1).reshape(-1), "bf16",
                        what=f"normed prefill {shape}")
    plain, _, _ = lrkv.prefill(dev["q"], dev["k_s"], dev["v_s"], dev["z_k"], dev["z_v"], dev["b_k"], dev["b_v"],
                               dev["seq_lens"])
    assert np.abs(plain.cpu().numpy()[:, 1:] - ref_o[:, 1:]).max() > 1e-2


def test_prefill_normed_needs_scales():
    B, Tq, H, Lm = 1, 128, 1, 128
    case = inputs.random_prefill_case(seed=3, batch=B, q_len=Tq, heads=H, head_dim=128, rank=64, max_len=Lm,
                                      lens=[128])
    dev = {k: v.cuda() for k, v in case.items()}
    dims = lrkv.make_dims(B, H, 128, 64, Lm, torch.bfloat16)
    out = torch.empty((B, Tq, H, 128), dtype=torch.float32, device="cuda")
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    st = lrkv.lrkv_prefill_normed(dims, Tq, dev["q"], dev["k_s"], dev["v_s"], dev["z_k"], dev["z_v"],
                                  dev["b_k"], dev["b_v"], None, dev["seq_lens"], out, None, ws, 16)
    assert st == lrkv.LRKV_ERR_INVALID_ARG
