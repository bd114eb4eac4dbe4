"""Bounded device waits that run out.

Every wait of the bf16 decode scan for one of its copies is bounded; with the
bound cut to one SM cycle (LRKV_WAIT_LIMIT_CYCLES, read by the library at each
call) the waits give up at once.  The scan must then skip the work that
depended on them, still wait at the full bound for every copy it issued (so
no copy lands in shared memory after the block exits), return, and record
LRKV_ERR_TIMEOUT in the call's status word.  The next call on the same
workspace with the default bound returns LRKV_OK and matches the oracle.  The
call runs with L2 flushed and caches larger than L2, so that its copies come
from HBM and the ring streams at the HBM rate: the warps must wait for copies
in flight (with every row already in L2 a copy may land before anyone waits
for it, and nothing times out).  A 16-head row tile, and 32 heads (two row
tiles, B^K staged through the ring)."""
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


@pytest.mark.parametrize("shape", [(4, 16, 64, 28, 32768, [32768, 32768, 9000, 32768]),
                                   (2, 32, 128, 48, 32768, [32768, 20000])])
def test_decode_wait_timeout_is_reported_and_the_next_call_recovers(shape, monkeypatch):
    B, H, dh, r, L, lens = shape
    case = inputs.random_decode_case(seed=31 + H, batch=B, heads=H, head_dim=dh, rank=r, max_len=L,
                                     dtype="bf16", lens=lens)
    d = {k: v.cuda() for k, v in case.items()}
    dims = lrkv.make_dims(B, H, dh, r, L, torch.bfloat16)
    ws = lrkv.decode_workspace(dims, "cuda")
    args = (d["q"], d["k_s"], d["v_s"], d["z_k"], d["z_v"], d["b_k"], d["b_v"], d["seq_lens"])

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    flush.fill_(1)  # evicts the cache rows the copies to the device left in L2
    monkeypatch.setenv("LRKV_WAIT_LIMIT_CYCLES", "1")
    lrkv.decode(*args, ws=ws)
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_ERR_TIMEOUT

    monkeypatch.delenv("LRKV_WAIT_LIMIT_CYCLES")
    out, lse = lrkv.decode(*args, ws=ws)
    torch.cuda.synchronize()
    assert lrkv.lrkv_read_device_status(ws) == lrkv.LRKV_OK
    ref_o, ref_l = O.decode_reference(*(case[k] for k in ("q", "k_s", "v_s", "z_k", "z_v", "b_k", "b_v",
                                                         "seq_lens")))
    assert_decode_close(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16", what="after a timeout")
    assert np.all(np.isfinite(out.cpu().numpy()))
