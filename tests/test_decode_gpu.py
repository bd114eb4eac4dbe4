"""Decode parity: the CUDA path (through the C ABI) against the fp64 oracle on
seeded inputs.  Small cases compare every output; the full-size workloads
compare sampled (sequence, head) pairs that the oracle computes one by one,
in the same launch configuration the bench times."""
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


def _to_dev(case):
    return {k: v.cuda() for k, v in case.items()}


def _run(case, scale=0.0, stream=None):
    d = _to_dev(case)
    out, lse = lrkv.decode(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                           d["seq_lens"], scale=scale, stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), d


def _oracle(case, pairs=None, scale=None):
    return O.decode_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"],
                              case["b_k"], case["b_v"], case["seq_lens"], scale=scale, pairs=pairs)


def test_tiny_fp32_workload_full():
    w = inputs.WORKLOADS["decode_f32_b1_h4_d16_r4_L64"]
    case = inputs.make_decode_inputs(w, seed=0)
    out, lse, _ = _run(case)
    ref_o, ref_l = _oracle(case)
    assert_decode_close(out, lse, ref_o, ref_l, "f32", what=w.name)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [
    # (B, H, d_h, r, max_len, lens)
    (3, 4, 16, 4, 200, [200, 1, 77]),
    (2, 16, 64, 28, 300, [300, 129]),
    (4, 32, 128, 48, 97, [97, 0, 33, 64]),      # an empty history
    (2, 32, 128, 56, 150, [150, 17]),
    (2, 8, 64, 0, 130, [130, 5]),                # rank 0: MQA
    (1, 18, 64, 8, 90, [90]),                    # heads not a multiple of 16
    (5, 16, 64, 8, 70, [1, 2, 3, 70, 69]),       # many short pieces in one CTA
])
def test_random_shapes(dtype, shape):
    B, H, dh, r, L, lens = shape
    if dtype == "bf16" and dh % 16:
        pytest.skip("bf16 needs head_dim % 16 == 0")
    case = inputs.random_decode_case(seed=B * 1000 + H * 10 + r + L, batch=B, heads=H, head_dim=dh,
                                     rank=r, max_len=L, dtype=dtype, lens=lens)
    if dtype == "f32" and dh > 64 and H >= 32:
        # the fp32 tile kernel keeps (d_h + r) / (lanes per head) value columns
        # per thread: these shapes are refused on the host, nothing enqueued
        d = _to_dev(case)
        dims = lrkv.make_dims(B, H, dh, r, L, torch.float32)
        ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        out = torch.full((B, H, dh), 7.0, dtype=torch.float32, device="cuda")
        lse = torch.full((B, H), 7.0, dtype=torch.float32, device="cuda")
        st = lrkv.lrkv_decode(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                              d["seq_lens"], out, lse, ws, ws.numel())
        torch.cuda.synchronize()
        assert st == lrkv.LRKV_ERR_UNSUPPORTED
        assert bool(torch.all(out == 7.0)) and bool(torch.all(lse == 7.0))
        return
    out, lse, _ = _run(case)
    ref_o, ref_l = _oracle(case)
    assert_decode_close(out, lse, ref_o, ref_l, dtype, what=f"{dtype}{shape}")
    for b, Lb in enumerate(lens):
        if Lb == 0:
            assert np.all(out[b] == 0.0)


@pytest.mark.parametrize("shape", [
    (2, 16, 64, 28, 300, [300, 129]),
    (4, 32, 128, 48, 97, [97, 0, 33, 64]),
    (8, 16, 64, 28, 4096, [4096, 4000, 1, 2048, 3333, 17, 4096, 640]),
])
def test_narrow_merge_tuning(monkeypatch, shape):
    """LRKV_DECODE_WIDE_MERGE=0: a small cache's merge runs one warp per pair on
    SMs the scan leaves free; same results as the default wide merge."""
    B, H, dh, r, L, lens = shape
    case = inputs.random_decode_case(seed=B * 7 + L, batch=B, heads=H, head_dim=dh, rank=r, max_len=L,
                                     dtype="bf16", lens=lens)
    wide_o, wide_l, _ = _run(case)
    monkeypatch.setenv("LRKV_DECODE_WIDE_MERGE", "0")
    out, lse, _ = _run(case)
    ref_o, ref_l = _oracle(case)
    assert_decode_close(out, lse, ref_o, ref_l, "bf16", what=f"narrow{shape}")
    assert_decode_close(wide_o, wide_l, ref_o, ref_l, "bf16", what=f"wide{shape}")


def test_explicit_scale():
    case = inputs.random_decode_case(seed=3, batch=2, heads=16, head_dim=64, rank=28, max_len=100,
                                     dtype="bf16", lens=[100, 40])
    out, lse, _ = _run(case, scale=0.3)
    ref_o, ref_l = _oracle(case, scale=0.3)
    assert_decode_close(out, lse, ref_o, ref_l, "bf16", what="scale=0.3")


def test_large_logits_stay_finite():
    """Scores of magnitude ~100: the online softmax must not overflow."""
    case = inputs.random_decode_case(seed=4, batch=2, heads=16, head_dim=64, rank=28, max_len=257,
                                     dtype="bf16", lens=[257, 200], q_scale=12.0)
    out, lse, _ = _run(case)
    ref_o, ref_l = _oracle(case)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    assert_decode_close(out, lse, ref_o, ref_l, "bf16", what="large logits")


def test_out_of_range_lengths_are_clamped_and_reported():
    case = inputs.random_decode_case(seed=5, batch=2, heads=16, head_dim=64, rank=28, max_len=64,
                                     dtype="bf16", lens=[64, 10])
    d = _to_dev(case)
    d["seq_lens"] = torch.tensor([1000, -3], dtype=torch.int32, device="cuda")
    dims = lrkv.make_dims(2, 16, 64, 28, 64, torch.bfloat16)
    ws = lrkv.decode_workspace(dims, "cuda")
    out, lse = lrkv.decode(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                           d["seq_lens"], ws=ws)
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_ERR_DEVICE_BOUNDS
    case["seq_lens"] = torch.tensor([64, 0], dtype=torch.int32)
    ref_o, ref_l = _oracle(case)
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", what="clamped")
    # a clean call resets the status word
    lrkv.decode(d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                torch.tensor([64, 10], dtype=torch.int32, device="cuda"), ws=ws)
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK


def test_repeatable_and_on_a_side_stream():
    case = inputs.random_decode_case(seed=6, batch=3, heads=32, head_dim=128, rank=56, max_len=333,
                                     dtype="bf16")
    out1, lse1, _ = _run(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out2, lse2, _ = _run(case, stream=s)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_workspace_too_small():
    case = inputs.random_decode_case(seed=7, batch=1, heads=16, head_dim=64, rank=28, max_len=64,
                                     dtype="bf16")
    d = _to_dev(case)
    dims = lrkv.make_dims(1, 16, 64, 28, 64, torch.bfloat16)
    n = lrkv.lrkv_decode_workspace_size(dims)
    ws = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    out = torch.empty((1, 16, 64), dtype=torch.float32, device="cuda")
    st = lrkv.lrkv_decode(dims, d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"],
                          d["seq_lens"], out, None, ws, n - 16)
    assert st == lrkv.LRKV_ERR_WORKSPACE


# ------------------------------------------------------- full-size workloads --

def _sampled_pairs(B, H, lens, n, seed):
    rng = np.random.default_rng(seed)
    pairs = {(int(b), int(h)) for b, h in zip(rng.integers(0, B, n), rng.integers(0, H, n))}
    pairs.add((0, 0))
    pairs.add((B - 1, H - 1))
    return sorted(pairs)


@pytest.mark.parametrize("name,n_pairs", [
    ("decode_bf16_b8_h16_d64_r28_L4096", None),                # every pair
    ("decode_bf16_b32_h32_d128_r56_ragged1k-8k", 40),
    ("decode_bf16_b4_h32_d128_r48_L65536_outliers", 12),
])
def test_full_size_workloads(name, n_pairs):
    w = inputs.WORKLOADS[name]
    case = inputs.make_decode_inputs(w, seed=0)
    out, lse, _ = _run(case)
    B, H = w.batch, w.heads
    pairs = None if n_pairs is None else _sampled_pairs(B, H, case["seq_lens"], n_pairs, 1)
    ref_o, ref_l = _oracle(case, pairs=pairs)
    if pairs is None:
        assert_decode_close(out, lse, ref_o, ref_l, "bf16", what=name)
    else:
        mask = np.zeros((B, H), dtype=bool)
        for b, h in pairs:
            mask[b, h] = True
        assert_decode_close(out, lse, ref_o, ref_l, "bf16", mask=mask, what=name)
    # properties that hold at any size, for every pair: finite outputs, lse at
    # least the log of the history length minus the score spread is not NaN
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
