"""Appends into a paged factored cache against the fp64 oracle: the append
GEMM writing logical rows start_pos[b] + t through a block table (starting
mid-page, crossing page boundaries), and the decode step writing the new
token's rows through it before decoding the paged cache.  Rows within one
bf16 ulp of the float64 product plus the fp32 accumulation bound (as for the
contiguous append); pool pages and rows not written stay as they were;
decode outputs within the bf16 decode bar on the GPU-written pools."""
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


def _check_rows(got, ref, absref, K, what):
    err = np.abs(got.astype(np.float64) - ref)
    tol = _ulp_bf16(ref) * 1.0000001 + K * 2.0 ** -24 * absref
    assert (err <= tol).all(), f"{what}: worst {err.max():.3e}"


def _same(a, b):
    """Equal, NaN included (bytes of bf16 tensors)."""
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("shape", [
    # B, T, d, H, dh, r, page_size, max_len, start positions
    (2, 77, 256, 4, 64, 16, 32, 256, [3, 120]),       # mid-page starts, three page boundaries
    (1, 128, 512, 8, 128, 64, 64, 256, [64]),         # page-aligned start (a prefill of 64 before it)
])
def test_append_paged_matches_oracle(shape):
    B, T, d, H, dh, r, ps, L, start = shape
    w = inputs.Workload("t", "prefill", B, H, dh, r, L, "bf16", q_len=T, d_model=d)
    c = inputs.make_prefill_inputs(w, seed=B * 5 + T, batch=B, q_len=T, d_model=d)
    dev = {k: v.cuda() for k, v in c.items()}
    nb = L // ps
    n_pages = B * nb + 3
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(T)).to(torch.int32)
    table = perm[:B * nb].reshape(B, nb).contiguous()
    pools = [torch.zeros((n_pages, ps, dh), dtype=torch.bfloat16, device="cuda") for _ in range(2)] + \
            [torch.zeros((n_pages, ps, H, r), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sp = torch.tensor(start, dtype=torch.int32, device="cuda")
    ws = lrkv.append_paged(dev["x"], dev["w_sk"], dev["w_sv"], dev["u_k"], dev["u_v"], sp, table.cuda(), *pools,
                           heads=H)
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    ref = O.append_reference(c["x"], c["w_sk"].t(), c["w_sv"].t(), c["u_k"].t(), c["u_v"].t(), H)
    absref = O.append_reference(c["x"].abs(), c["w_sk"].abs().t(), c["w_sv"].abs().t(), c["u_k"].abs().t(),
                                c["u_v"].abs().t(), H)
    for name, pool, rf, ab in zip(("k_s", "v_s", "z_k", "z_v"), pools, ref, absref):
        logical = O.gather_paged(pool.cpu().float(), table.numpy(), ps, L)
        for b in range(B):
            rows = slice(start[b], start[b] + T)
            _check_rows(logical[b, rows], rf[b], ab[b], d, f"{name} seq {b}")
            assert np.all(logical[b, :start[b]] == 0) and np.all(logical[b, start[b] + T:] == 0)
        unused = perm[B * nb:].long()
        assert torch.all(pool[unused.cuda()] == 0), f"{name}: pages outside the table written"


def test_append_paged_unmapped_block_is_reported():
    B, T, d, H, dh, r, ps, L = 1, 64, 64, 2, 64, 32, 16, 128
    w = inputs.Workload("t", "prefill", B, H, dh, r, L, "bf16", q_len=T, d_model=d)
    c = inputs.make_prefill_inputs(w, seed=2, batch=B, q_len=T, d_model=d)
    dev = {k: v.cuda() for k, v in c.items()}
    table = torch.arange(L // ps, dtype=torch.int32).reshape(1, -1).contiguous()
    table[0, 2] = -1                                               # rows 32..47 have no page
    n_pages = L // ps
    pools = [torch.zeros((n_pages, ps, dh), dtype=torch.bfloat16, device="cuda") for _ in range(2)] + \
            [torch.zeros((n_pages, ps, H, r), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sp = torch.tensor([16], dtype=torch.int32, device="cuda")      # rows 16..79
    ws = lrkv.append_paged(dev["x"], dev["w_sk"], dev["w_sv"], dev["u_k"], dev["u_v"], sp, table.cuda(), *pools,
                           heads=H)
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_ERR_DEVICE_BOUNDS
    ref = O.append_reference(c["x"], c["w_sk"].t(), c["w_sv"].t(), c["u_k"].t(), c["u_v"].t(), H)
    ab = O.append_reference(c["x"].abs(), c["w_sk"].abs().t(), c["w_sv"].abs().t(), c["u_k"].abs().t(),
                            c["u_v"].abs().t(), H)
    logical = O.gather_paged(pools[0].cpu().float(), table.numpy(), ps, L)
    _check_rows(logical[0, 16:32], ref[0][0, :16], ab[0][0, :16], d, "rows before the unmapped block")
    _check_rows(logical[0, 48:80], ref[0][0, 32:], ab[0][0, 32:], d, "rows after it")
    assert torch.all(pools[0][2] == 0)                             # page 2 is not in the table


@pytest.mark.parametrize("shape", [
    # B, H, d_h, r, d_model, page_size, max_len, lengths (including the new token)
    (3, 16, 64, 28, 256, 16, 128, [57, 128, 1]),
    (4, 8, 64, 16, 512, 64, 256, [64, 65, 200, 0]),   # the new token opens a page / ends one
])
def test_decode_step_paged_matches_oracle(shape):
    B, H, dh, r, d, ps, L, lens = shape
    case = inputs.random_decode_case(seed=B * 23 + d, batch=B, heads=H, head_dim=dh, rank=r, max_len=L,
                                     dtype="bf16", lens=lens)
    paged = inputs.paged_from_contiguous(case, page_size=ps, seed=d + ps)
    g = torch.Generator().manual_seed(B + d)
    x = torch.randn(B, d, generator=g).to(torch.bfloat16)
    wts = [(torch.randn(n, d, generator=g) / d ** 0.5).to(torch.bfloat16) for n in (dh, dh, H * r, H * r)]
    dev = {k: v.cuda() for k, v in paged.items()}
    before = {k: dev[k].clone() for k in ("k_s", "v_s", "z_k", "z_v")}
    out, lse, ws = lrkv.decode_step_paged(x.cuda(), *[t.cuda() for t in wts], dev["q"], dev["k_s"], dev["v_s"],
                                          dev["z_k"], dev["z_v"], dev["b_k"], dev["b_v"], dev["block_table"],
                                          dev["seq_lens"])
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    bt = paged["block_table"].numpy()
    ref = O.append_reference(x[:, None, :], wts[0].t(), wts[1].t(), wts[2].t(), wts[3].t(), H)
    ab = O.append_reference(x.abs()[:, None, :], wts[0].abs().t(), wts[1].abs().t(), wts[2].abs().t(),
                            wts[3].abs().t(), H)
    for name, rf, a in zip(("k_s", "v_s", "z_k", "z_v"), ref, ab):
        pool = dev[name]
        logical = O.gather_paged(pool.cpu().float(), bt, ps, L)
        for b, Lb in enumerate(lens):
            if Lb >= 1:
                _check_rows(logical[b, Lb - 1], rf[b, 0], a[b, 0], d, f"{name} seq {b}")
        # everything else in the pool is as it was: restore the new rows and compare bytes
        restored = pool.clone()
        for b, Lb in enumerate(lens):
            if Lb >= 1:
                pg, rw = int(bt[b, (Lb - 1) // ps]), (Lb - 1) % ps
                restored[pg, rw] = before[name][pg, rw]
        assert _same(restored, before[name]), f"{name}: other rows changed"
    g_cache = [O.gather_paged(dev[k].cpu(), bt, ps, L) for k in ("k_s", "v_s", "z_k", "z_v")]
    ref_o, ref_l = O.decode_reference(paged["q"], *g_cache, paged["b_k"], paged["b_v"], paged["seq_lens"])
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", what=f"paged step {shape}")
