"""Append parity: the tcgen05 GEMM that builds the factored cache rows
(review §3 Algorithm 1) against the fp64 oracle.  Each stored bf16 element
must be within one bf16 ulp of the float64 product plus the fp32 accumulation
bound K * 2^-24 * sum_i |x_i w_i| (the standard dot-product error bound; it
only matters where the product nearly cancels)."""
import numpy as np
import pytest
import torch

from _lib_util import ensure_built
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
    """One bf16 ulp at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def _check(got, ref, what, absdot=None, K=0):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    tol = _ulp_bf16(ref) * 1.0000001
    if absdot is not None:
        tol = tol + K * 2.0 ** -24 * absdot
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond 1 ulp; worst {err[bad].max():.3e}"


def _run(B, T, d, H, dh, r, max_len, start, seed):
    w = inputs.Workload("t", "prefill", B, H, dh, r, max_len, "bf16", q_len=T, d_model=d)
    c = inputs.make_prefill_inputs(w, seed=seed, batch=B, q_len=T, d_model=d)
    dev = {k: v.cuda() for k, v in c.items()}
    k_s = torch.zeros((B, max_len, dh), dtype=torch.bfloat16, device="cuda")
    v_s = torch.zeros_like(k_s)
    z_k = torch.zeros((B, max_len, H, r), dtype=torch.bfloat16, device="cuda")
    z_v = torch.zeros_like(z_k)
    sp = torch.tensor(start, dtype=torch.int32, device="cuda")
    status = lrkv.append(dev["x"], dev["w_sk"], dev["w_sv"], dev["u_k"], dev["u_v"], sp,
                         k_s, v_s, z_k, z_v)
    assert status == lrkv.LRKV_OK
    ref = O.append_reference(c["x"], c["w_sk"].t(), c["w_sv"].t(), c["u_k"].t(), c["u_v"].t(), H)
    absref = O.append_reference(c["x"].abs(), c["w_sk"].abs().t(), c["w_sv"].abs().t(),
                                c["u_k"].abs().t(), c["u_v"].abs().t(), H)
    return [t.cpu() for t in (k_s, v_s, z_k, z_v)], ref, absref


@pytest.mark.parametrize("shape", [
    # B, T, d, H, dh, r, max_len, start positions
    (1, 128, 64, 2, 64, 32, 128, [0]),
    (2, 77, 256, 4, 64, 16, 200, [3, 120]),       # ragged tail rows, offsets
    (2, 300, 512, 8, 128, 64, 400, [0, 100]),      # several N tiles, K loop of 8
])
def test_append_matches_oracle(shape):
    B, T, d, H, dh, r, L, start = shape
    got, ref, absref = _run(B, T, d, H, dh, r, L, start, seed=B * 7 + T)
    names = ["k_s", "v_s", "z_k", "z_v"]
    for b in range(B):
        rows = slice(start[b], start[b] + T)
        for name, g, rf, ab in zip(names, got, ref, absref):
            _check(g[b, rows].float().numpy(), rf[b], f"{name} seq {b}", ab[b], d)
        # rows outside the appended range stay untouched (zero)
        for g in got:
            assert torch.all(g[b, :start[b]] == 0) and torch.all(g[b, start[b] + T:] == 0)


def test_append_out_of_range_start_is_reported():
    B, T, d, H, dh, r, L = 1, 16, 64, 2, 64, 32, 20
    w = inputs.Workload("t", "prefill", B, H, dh, r, L, "bf16", q_len=T, d_model=d)
    c = inputs.make_prefill_inputs(w, seed=1, batch=B, q_len=T, d_model=d)
    dev = {k: v.cuda() for k, v in c.items()}
    k_s = torch.zeros((B, L, dh), dtype=torch.bfloat16, device="cuda")
    v_s = torch.zeros_like(k_s)
    z_k = torch.zeros((B, L, H, r), dtype=torch.bfloat16, device="cuda")
    z_v = torch.zeros_like(z_k)
    sp = torch.tensor([10], dtype=torch.int32, device="cuda")  # rows 10..25 of 20
    status = lrkv.append(dev["x"], dev["w_sk"], dev["w_sv"], dev["u_k"], dev["u_v"], sp,
                         k_s, v_s, z_k, z_v)
    assert status == lrkv.LRKV_ERR_DEVICE_BOUNDS
    ref = O.append_reference(c["x"], c["w_sk"].t(), c["w_sv"].t(), c["u_k"].t(), c["u_v"].t(), H)
    ab = O.append_reference(c["x"].abs(), c["w_sk"].abs().t(), c["w_sv"].abs().t(),
                            c["u_k"].abs().t(), c["u_v"].abs().t(), H)
    _check(k_s[0, 10:20].cpu().float().numpy(), ref[0][0, :10], "in-range rows still written",
           ab[0][0, :10], d)


def test_append_full_size_sampled_rows():
    """The prefill workload's append (8192 x 4096 x 4352): sampled rows against
    the oracle, the rest checked for finiteness."""
    w = inputs.WORKLOADS[inputs.PREFILL_WORKLOAD]
    c = inputs.make_prefill_inputs(w, seed=0)
    dev = {k: v.cuda() for k, v in c.items()}
    B, T, H, dh, r = w.batch, w.q_len, w.heads, w.head_dim, w.rank
    k_s = torch.empty((B, T, dh), dtype=torch.bfloat16, device="cuda")
    v_s = torch.empty_like(k_s)
    z_k = torch.empty((B, T, H, r), dtype=torch.bfloat16, device="cuda")
    z_v = torch.empty_like(z_k)
    status = lrkv.append(dev["x"], dev["w_sk"], dev["w_sv"], dev["u_k"], dev["u_v"],
                         dev["start_pos"], k_s, v_s, z_k, z_v)
    assert status == lrkv.LRKV_OK
    rng = np.random.default_rng(0)
    rows = sorted(set(rng.integers(0, T, 24).tolist()) | {0, T - 1})
    for b in range(B):
        xb = c["x"][b:b + 1, rows]
        ref = O.append_reference(xb, c["w_sk"].t(), c["w_sv"].t(), c["u_k"].t(), c["u_v"].t(), H)
        ab = O.append_reference(xb.abs(), c["w_sk"].abs().t(), c["w_sv"].abs().t(),
                                c["u_k"].abs().t(), c["u_v"].abs().t(), H)
        for g, rf, a, name in zip((k_s, v_s, z_k, z_v), ref, ab, ["k_s", "v_s", "z_k", "z_v"]):
            _check(g[b, rows].cpu().float().numpy(), rf[0], f"{name} seq {b}", a[0], w.d_model)
    for g in (k_s, v_s, z_k, z_v):
        assert torch.isfinite(g.float()).all()
