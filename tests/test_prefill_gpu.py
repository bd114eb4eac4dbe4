"""Causal prefill parity: the tcgen05 flash kernel against the fp64 oracle
(bottom-right causal alignment; bf16 inputs, fp32 accumulation; q_h B_h^K
enters its contraction with the latents as two bf16 parts)."""
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


def _check(out, lse, ref_o, ref_l, what):
    # out [B, Tq, H, dh], lse [B, H, Tq]: compare as (B*Tq*H) rows
    B, Tq, H, dh = out.shape
    o = out.reshape(B * Tq * H, dh)
    ro = ref_o.reshape(B * Tq * H, dh)
    l_ = lse.transpose(0, 2, 1).reshape(-1)
    rl = ref_l.transpose(0, 2, 1).reshape(-1)
    keep = ~np.isnan(rl)
    assert_decode_close(o[keep], l_[keep], ro[keep], rl[keep], "bf16", what=what)


@pytest.mark.parametrize("shape", [
    # B, q_len, H, L per sequence, max_len
    (1, 128, 2, [128], 128),
    (2, 256, 2, [256, 300], 320),        # extra history before the queries, ragged key tile
    (1, 200, 1, [200], 256),             # partial query tile and key tile
    (2, 64, 3, [64, 500], 512),          # short block after a long history
    # more (sequence, head, query tile) items than SMs: each persistent CTA
    # runs several items back to back, of different sequences and lengths
    (2, 512, 48, [512, 700], 768),
])
def test_prefill_matches_oracle(shape):
    B, Tq, H, lens, Lm = shape
    case = inputs.random_prefill_case(seed=B * 100 + Tq, batch=B, q_len=Tq, heads=H, head_dim=128,
                                      rank=64, max_len=Lm, lens=lens)
    d = {k: v.cuda() for k, v in case.items()}
    out, lse, ws = lrkv.prefill(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                                d["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    ref_o, ref_l = O.prefill_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"],
                                       case["b_k"], case["b_v"], case["seq_lens"])
    _check(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, f"prefill {shape}")


def test_prefill_garbage_rows_past_history_are_ignored():
    """Cache rows past seq_lens hold NaN: outputs stay finite and equal."""
    B, Tq, H, Lm = 1, 100, 2, 256
    case = inputs.random_prefill_case(seed=5, batch=B, q_len=Tq, heads=H, head_dim=128, rank=64,
                                      max_len=Lm, lens=[150])
    d = {k: v.cuda() for k, v in case.items()}
    for k in ("k_s", "v_s", "z_k", "z_v"):
        d[k][:, 150:] = float("nan")
    out, lse, _ = lrkv.prefill(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                               d["seq_lens"])
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    ref_o, ref_l = O.prefill_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"],
                                       case["b_k"], case["b_v"], case["seq_lens"])
    _check(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "nan past history")


def test_prefill_full_size_on_gpu_written_cache():
    """The prefill workload end to end on the GPU: append builds the cache from
    x, then causal prefill; sampled (sequence, head, query) rows against the
    oracle evaluated on the GPU-written cache."""
    w = inputs.WORKLOADS[inputs.PREFILL_WORKLOAD]
    c = inputs.make_prefill_inputs(w, seed=0)
    dev = {k: v.cuda() for k, v in c.items()}
    B, T, H, dh, r = w.batch, w.q_len, w.heads, w.head_dim, w.rank
    k_s = torch.empty((B, T, dh), dtype=torch.bfloat16, device="cuda")
    v_s = torch.empty_like(k_s)
    z_k = torch.empty((B, T, H, r), dtype=torch.bfloat16, device="cuda")
    z_v = torch.empty_like(z_k)
    assert lrkv.append(dev["x"], dev["w_sk"], dev["w_sv"], dev["u_k"], dev["u_v"], dev["start_pos"],
                       k_s, v_s, z_k, z_v) == lrkv.LRKV_OK
    out, lse, ws = lrkv.prefill(dev["q"], k_s, v_s, z_k, z_v, dev["b_k"], dev["b_v"],
                                dev["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    cache = {k: t.cpu() for k, t in dict(k_s=k_s, v_s=v_s, z_k=z_k, z_v=z_v).items()}
    rng = np.random.default_rng(3)
    pairs = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, B, 6), rng.integers(0, H, 6))}
                   | {(0, 0), (B - 1, H - 1)})
    rows = sorted(set(rng.integers(0, T, 12).tolist()) | {0, 1, 127, 128, T - 1})
    ref_o, ref_l = O.prefill_reference(c["q"], cache["k_s"], cache["v_s"], cache["z_k"], cache["z_v"],
                                       c["b_k"], c["b_v"], c["seq_lens"], pairs=pairs, rows=rows)
    o = out.cpu().numpy()
    l_ = lse.cpu().numpy()
    for b, h in pairs:
        assert_decode_close(o[b, rows, h], l_[b, h, rows], ref_o[b, rows, h], ref_l[b, h, rows],
                            "bf16", what=f"prefill full b={b} h={h}")
