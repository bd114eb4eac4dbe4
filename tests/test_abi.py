"""The C-ABI library loads and exports every symbol include/lrkv.h declares,
and its host-side checks reject bad arguments before touching a GPU.  No
compute call is made here (these run without a GPU)."""
import ctypes

import pytest

from _lib_util import ensure_built, header_symbols
from compressed_cache_decode_gb300 import lrkv


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    return lrkv.load()


def test_exports_every_declared_symbol(lib):
    declared = header_symbols()
    assert declared, "no declarations parsed"
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/lrkv.h but not exported"
    assert set(declared) == set(lrkv.EXPORTED), "binding and header disagree"


def test_version_and_status_strings(lib):
    assert lib.lrkv_abi_version() == 1
    for code, name in [(0, "LRKV_OK"), (1, "LRKV_ERR_INVALID_ARG"), (2, "LRKV_ERR_UNSUPPORTED"),
                       (3, "LRKV_ERR_WORKSPACE"), (4, "LRKV_ERR_CUDA"), (5, "LRKV_ERR_TIMEOUT"),
                       (6, "LRKV_ERR_DEVICE_BOUNDS")]:
        assert lrkv.status_string(code) == name
    assert lrkv.status_string(99) == "LRKV_ERR_UNKNOWN"


def test_cache_elems_per_token(lib):
    # 2 (d_h + H r): 4608 -> 2236 at H=18, d_h=128, r=55 (reading notes §2.5)
    assert lrkv.lrkv_cache_elems_per_token(18, 128, 55) == 2236
    assert lrkv.lrkv_cache_elems_per_token(16, 64, 28) == 1024
    assert lrkv.lrkv_cache_elems_per_token(4, 16, 0) == 32
    assert lrkv.lrkv_cache_elems_per_token(-1, 16, 0) == 0


def _call(dims, **kw):
    args = dict(q=None, k_s=None, v_s=None, z_k=None, z_v=None, b_k=None, b_v=None,
                seq_lens=None, out=None, lse=None, ws=None, ws_bytes=0)
    args.update(kw)
    lib = lrkv.load()
    return lib.lrkv_decode(None if dims is None else ctypes.byref(dims), args["q"], args["k_s"],
                           args["v_s"], args["z_k"], args["z_v"], args["b_k"], args["b_v"],
                           args["seq_lens"], args["out"], args["lse"], args["ws"],
                           args["ws_bytes"], None)


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on these paths


def test_rejects_bad_dims_without_gpu(lib):
    good = dict(q=FAKE, k_s=FAKE, v_s=FAKE, z_k=FAKE, z_v=FAKE, b_k=FAKE, b_v=FAKE,
                seq_lens=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 30)
    assert _call(None, **good) == lrkv.LRKV_ERR_INVALID_ARG
    for bad in [lrkv.make_dims(0, 16, 64, 28, 64, "bf16"), lrkv.make_dims(1, 0, 64, 28, 64, "bf16"),
                lrkv.make_dims(1, 16, 0, 28, 64, "bf16"), lrkv.make_dims(1, 16, 64, -1, 64, "bf16"),
                lrkv.make_dims(1, 16, 64, 28, 0, "bf16"), lrkv.make_dims(1, 16, 64, 28, 64, 7)]:
        assert _call(bad, **good) == lrkv.LRKV_ERR_INVALID_ARG
    nan_scale = lrkv.make_dims(1, 16, 64, 28, 64, "bf16", scale=float("nan"))
    assert _call(nan_scale, **good) == lrkv.LRKV_ERR_INVALID_ARG


def test_rejects_unsupported_shapes_without_gpu(lib):
    good = dict(q=FAKE, k_s=FAKE, v_s=FAKE, z_k=FAKE, z_v=FAKE, b_k=FAKE, b_v=FAKE,
                seq_lens=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 30)
    for dims in [lrkv.make_dims(1, 16, 60, 28, 64, "bf16"),     # row not a multiple of 16 B
                 lrkv.make_dims(1, 6, 128, 46, 64, "bf16"),     # H*r*2 = 552 B
                 lrkv.make_dims(1, 16, 64, 72, 64, "bf16"),     # rank above 64
                 lrkv.make_dims(5000, 16, 64, 28, 64, "bf16"),  # batch above 4096
                 lrkv.make_dims(1, 16, 24, 28, 64, "bf16")]:    # bf16 head_dim % 16
        assert _call(dims, **good) == lrkv.LRKV_ERR_UNSUPPORTED


def test_rejects_null_and_misaligned_pointers_without_gpu(lib):
    dims = lrkv.make_dims(2, 16, 64, 28, 128, "bf16")
    base = dict(q=FAKE, k_s=FAKE, v_s=FAKE, z_k=FAKE, z_v=FAKE, b_k=FAKE, b_v=FAKE,
                seq_lens=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 30)
    for key in ["q", "k_s", "v_s", "z_k", "z_v", "b_k", "b_v", "seq_lens", "out"]:
        args = dict(base)
        args[key] = None
        assert _call(dims, **args) == lrkv.LRKV_ERR_INVALID_ARG, key
    for key in ["q", "k_s", "v_s", "z_k", "z_v"]:
        args = dict(base)
        args[key] = FAKE + 8
        assert _call(dims, **args) == lrkv.LRKV_ERR_INVALID_ARG, key
    args = dict(base)
    args["ws"] = None
    assert _call(dims, **args) == lrkv.LRKV_ERR_WORKSPACE
    # rank 0 (MQA) needs no latents or bases
    dims0 = lrkv.make_dims(2, 16, 64, 0, 128, "bf16")
    args = dict(base, z_k=None, z_v=None, b_k=None, b_v=None, ws=None)
    assert _call(dims0, **args) == lrkv.LRKV_ERR_WORKSPACE


def test_workspace_size_checks_arguments(lib):
    n = ctypes.c_size_t(0)
    assert lib.lrkv_decode_workspace_size(None, ctypes.byref(n)) == lrkv.LRKV_ERR_INVALID_ARG
    d = lrkv.make_dims(1, 16, 64, 28, 64, "bf16")
    assert lib.lrkv_decode_workspace_size(ctypes.byref(d), None) == lrkv.LRKV_ERR_INVALID_ARG
    bad = lrkv.make_dims(1, 16, 60, 28, 64, "bf16")
    assert lib.lrkv_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == lrkv.LRKV_ERR_UNSUPPORTED


def test_new_entries_reject_bad_arguments_without_gpu(lib):
    """The decode step, the key scales and the normalised decode and prefill
    check dtype, rank, sizes and pointers on the host before any launch."""
    f32 = lrkv.make_dims(2, 4, 64, 16, 128, None)
    f32.dtype = lrkv.LRKV_F32
    bf = lrkv.make_dims(2, 4, 64, 16, 128, None)
    bf.dtype = lrkv.LRKV_BF16
    fake = ctypes.c_void_p(4096)  # aligned, never dereferenced: the checks fail first
    args_scales = (0.0, 8, fake, fake, fake, fake, fake, None)
    assert lib.lrkv_key_scales(ctypes.byref(f32), *args_scales) == lrkv.LRKV_ERR_UNSUPPORTED
    assert lib.lrkv_key_scales(ctypes.byref(bf), -1.0, 8, fake, fake, fake, fake, fake, None) == \
        lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_key_scales(ctypes.byref(bf), 0.0, 8, None, fake, fake, fake, fake, None) == \
        lrkv.LRKV_ERR_INVALID_ARG
    normed = (fake,) * 7 + (fake, fake, fake, fake, fake, 1 << 20, None)
    assert lib.lrkv_decode_normed(ctypes.byref(f32), *normed) == lrkv.LRKV_ERR_UNSUPPORTED
    assert lib.lrkv_decode_normed(ctypes.byref(bf), *((fake,) * 7), None, fake, fake, fake, fake, 1 << 20,
                                  None) == lrkv.LRKV_ERR_INVALID_ARG
    pre = (fake,) * 7     # q, the cache, the bases
    assert lib.lrkv_prefill_normed(ctypes.byref(bf), 128, *pre, None, fake, fake, fake, fake, 1 << 20,
                                   None) == lrkv.LRKV_ERR_INVALID_ARG      # no key scales
    pbf = lrkv.make_dims(1, 2, 128, 64, 128, "bf16")
    assert lib.lrkv_prefill_normed(ctypes.byref(pbf), 256, *pre, fake, fake, fake, fake, fake, 1 << 20,
                                   None) == lrkv.LRKV_ERR_UNSUPPORTED      # q_len > max_len
    ptrs = (fake,) * 15   # x, the weights, q, the cache, the bases, seq_lens, out, lse
    assert lib.lrkv_decode_step(ctypes.byref(f32), 64, *ptrs, fake, 1 << 20, None) == lrkv.LRKV_ERR_UNSUPPORTED
    assert lib.lrkv_decode_step(ctypes.byref(bf), 60, *ptrs, fake, 1 << 20, None) == \
        lrkv.LRKV_ERR_UNSUPPORTED       # d_model not a multiple of 8


def test_paged_decode_rejects_bad_paging_without_gpu(lib):
    """Page size, pool size and table are checked on the host before any launch."""
    bf = lrkv.make_dims(2, 16, 64, 28, 256, "bf16")
    fake = ctypes.c_void_p(4096)  # aligned, never dereferenced: the checks fail first
    rest = (fake,) * 7 + (fake, fake, fake, fake, 1 << 24, None)  # q .. b_v, seq_lens, out, lse, ws, bytes, stream
    call = lib.lrkv_decode_paged
    assert call(ctypes.byref(bf), 24, 8, fake, *rest) == lrkv.LRKV_ERR_INVALID_ARG    # not a power of two
    assert call(ctypes.byref(bf), 8, 8, fake, *rest) == lrkv.LRKV_ERR_INVALID_ARG     # below one 16-token tile
    assert call(ctypes.byref(bf), 512, 8, fake, *rest) == lrkv.LRKV_ERR_INVALID_ARG   # max_len not a multiple
    assert call(ctypes.byref(bf), 64, 0, fake, *rest) == lrkv.LRKV_ERR_INVALID_ARG    # empty pool
    assert call(ctypes.byref(bf), 64, 8, None, *rest) == lrkv.LRKV_ERR_INVALID_ARG    # no block table
    f32 = lrkv.make_dims(2, 16, 64, 28, 256, None)
    f32.dtype = lrkv.LRKV_F32
    assert call(ctypes.byref(f32), 64, 8, fake, *rest) == lrkv.LRKV_ERR_UNSUPPORTED   # bf16 streaming only
    pre = lrkv.make_dims(1, 2, 128, 64, 512, "bf16")
    prest = (fake,) * 6 + (fake, fake, fake, fake, 1 << 20, None)  # k_s .. b_v, seq_lens, out, lse, ws, bytes, stream
    assert lib.lrkv_prefill_paged(ctypes.byref(pre), 128, fake, 64, 8, fake, *prest) == \
        lrkv.LRKV_ERR_INVALID_ARG                                                     # a key tile spans pages


def test_paged_appends_reject_bad_paging_without_gpu(lib):
    """The paged append and decode step check the paging before any launch."""
    bf = lrkv.make_dims(2, 4, 64, 16, 256, "bf16")
    fake = ctypes.c_void_p(4096)
    w = (fake,) * 5                                     # x and the four weights
    cache = (fake,) * 4
    # append: (dims, d_model, n_new, x, w_sk, w_sv, u_k, u_v, start_pos, page_size, num_pages, table, cache.., ws..)
    assert lib.lrkv_append_paged(ctypes.byref(bf), 256, 8, *w, fake, 24, 8, fake, *cache, fake, 16, None) == \
        lrkv.LRKV_ERR_INVALID_ARG                       # page size not a power of two
    assert lib.lrkv_append_paged(ctypes.byref(bf), 256, 8, *w, fake, 64, 8, None, *cache, fake, 16, None) == \
        lrkv.LRKV_ERR_INVALID_ARG                       # no block table
    # decode step: (dims, d_model, x, w.., q, page_size, num_pages, table, cache.., b_k, b_v, seq_lens, out, lse, ws..)
    assert lib.lrkv_decode_step_paged(ctypes.byref(bf), 256, *w, fake, 512, 8, fake, *cache, fake, fake, fake,
                                      fake, fake, fake, 1 << 20, None) == lrkv.LRKV_ERR_INVALID_ARG  # > max_len
    assert lib.lrkv_decode_step_paged(ctypes.byref(bf), 256, *w, fake, 64, 0, fake, *cache, fake, fake, fake,
                                      fake, fake, fake, 1 << 20, None) == lrkv.LRKV_ERR_INVALID_ARG  # no pages


def test_prefill_workspace_size_and_rejection_without_gpu(lib):
    """The prefill's workspace query checks the shape like the prefill does,
    and a prefill given fewer bytes is rejected before any launch."""
    n = ctypes.c_size_t(0)
    d = lrkv.make_dims(2, 32, 128, 64, 4096, "bf16")
    assert lib.lrkv_prefill_workspace_size(ctypes.byref(d), 4096, ctypes.byref(n)) == lrkv.LRKV_OK
    assert n.value == 16 == lrkv.lrkv_prefill_workspace_size(d, 4096)
    assert lib.lrkv_prefill_workspace_size(None, 16, ctypes.byref(n)) == lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_prefill_workspace_size(ctypes.byref(d), 16, None) == lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_prefill_workspace_size(ctypes.byref(d), 0, ctypes.byref(n)) == lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_prefill_workspace_size(ctypes.byref(d), 8192, ctypes.byref(n)) == \
        lrkv.LRKV_ERR_UNSUPPORTED                                          # q_len > max_len
    other = lrkv.make_dims(2, 32, 64, 64, 4096, "bf16")
    assert lib.lrkv_prefill_workspace_size(ctypes.byref(other), 16, ctypes.byref(n)) == lrkv.LRKV_ERR_UNSUPPORTED
    fake = ctypes.c_void_p(4096)  # aligned, never dereferenced: the checks fail first
    pre = (fake,) * 8             # q, the cache, the bases, seq_lens
    need = lrkv.lrkv_prefill_workspace_size(d, 128)
    for call, extra in ((lib.lrkv_prefill, ()), (lib.lrkv_prefill_normed, None)):
        args = pre if extra is not None else (fake,) * 7 + (fake, fake)   # normed: + key_scale before seq_lens
        assert call(ctypes.byref(d), 128, *args, fake, fake, fake, need - 1, None) == lrkv.LRKV_ERR_WORKSPACE
        assert call(ctypes.byref(d), 128, *args, fake, fake, None, need, None) == lrkv.LRKV_ERR_WORKSPACE
        assert call(ctypes.byref(d), 128, *args, fake, fake, ctypes.c_void_p(4096 + 8), need, None) == \
            lrkv.LRKV_ERR_INVALID_ARG                                      # misaligned workspace
    paged = (fake,) * 6 + (fake,)  # k_s .. b_v, seq_lens
    assert lib.lrkv_prefill_paged(ctypes.byref(d), 128, fake, 128, 64, fake, *paged, fake, fake, fake, need - 1,
                                  None) == lrkv.LRKV_ERR_WORKSPACE


def test_rope_entries_reject_bad_arguments_without_gpu(lib):
    """The full-RoPE table and decode check shapes, the table length and the
    workspace on the host before any launch."""
    fake = ctypes.c_void_p(4096)
    assert lib.lrkv_rope_table(0, 128, 10000.0, fake, None) == lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_rope_table(16, 127, 10000.0, fake, None) == lrkv.LRKV_ERR_INVALID_ARG   # odd head_dim
    assert lib.lrkv_rope_table(16, 128, 1.0, fake, None) == lrkv.LRKV_ERR_INVALID_ARG      # base must exceed 1
    assert lib.lrkv_rope_table(16, 128, 10000.0, None, None) == lrkv.LRKV_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    for dims, want in [(lrkv.make_dims(2, 16, 64, 28, 64, "bf16"), lrkv.LRKV_ERR_UNSUPPORTED),    # rank % 16
                       (lrkv.make_dims(2, 12, 64, 32, 64, "bf16"), lrkv.LRKV_ERR_UNSUPPORTED),    # heads % 8
                       (lrkv.make_dims(2, 16, 96, 32, 64, "bf16"), lrkv.LRKV_ERR_UNSUPPORTED),    # head_dim
                       (lrkv.make_dims(2, 16, 64, 32, 64, "f32"), lrkv.LRKV_ERR_UNSUPPORTED),
                       (lrkv.make_dims(0, 16, 64, 32, 64, "bf16"), lrkv.LRKV_ERR_INVALID_ARG)]:
        assert lib.lrkv_decode_rope_workspace_size(ctypes.byref(dims), ctypes.byref(n)) == want
    ok = lrkv.make_dims(2, 16, 64, 32, 64, "bf16")
    args = (fake,) * 8   # q~, the cache, the bases, the table
    # a table shorter than the cache, a missing pointer, a missing workspace
    assert lib.lrkv_decode_rope(ctypes.byref(ok), *args, 63, fake, fake, fake, fake, 1 << 20, None) == \
        lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_decode_rope(ctypes.byref(ok), *args[:7], None, 64, fake, fake, fake, fake, 1 << 20, None) == \
        lrkv.LRKV_ERR_INVALID_ARG
    assert lib.lrkv_decode_rope(ctypes.byref(ok), *args, 64, fake, fake, fake, None, 1 << 20, None) == \
        lrkv.LRKV_ERR_WORKSPACE


def test_comparison_entries_reject_bad_arguments_without_gpu(lib):
    """The dense and MLA comparison decodes check shapes before any launch."""
    n = ctypes.c_size_t(0)
    dd = lrkv.lrkv_dense_dims
    for dims, want in [(dd(2, 32, 2, 128, 64, 0.0), lrkv.LRKV_ERR_UNSUPPORTED),   # group of 16
                       (dd(2, 8, 8, 96, 64, 0.0), lrkv.LRKV_ERR_UNSUPPORTED),     # head_dim 96
                       (dd(2, 8, 3, 64, 64, 0.0), lrkv.LRKV_ERR_INVALID_ARG),     # 3 does not divide 8
                       (dd(0, 8, 8, 64, 64, 0.0), lrkv.LRKV_ERR_INVALID_ARG)]:
        assert lib.lrkv_dense_decode_workspace_size(ctypes.byref(dims), ctypes.byref(n)) == want
    md = lrkv.lrkv_mla_dims
    for dims, want in [(md(2, 32, 128, 384, 64, 0.0), lrkv.LRKV_ERR_UNSUPPORTED),   # latent width
                       (md(2, 12, 128, 512, 64, 0.0), lrkv.LRKV_ERR_UNSUPPORTED),    # 12 heads
                       (md(2, 32, 256, 512, 64, 0.0), lrkv.LRKV_ERR_UNSUPPORTED),    # head_dim
                       (md(2, 32, 128, 512, 0, 0.0), lrkv.LRKV_ERR_INVALID_ARG)]:
        assert lib.lrkv_mla_decode_workspace_size(ctypes.byref(dims), ctypes.byref(n)) == want
    fake = ctypes.c_void_p(4096)
    ok = dd(2, 8, 8, 64, 64, 0.0)
    assert lib.lrkv_dense_decode(ctypes.byref(ok), fake, fake, fake, fake, fake, None, None, 1 << 20, None) == \
        lrkv.LRKV_ERR_WORKSPACE
    okm = md(2, 8, 64, 256, 64, 0.0)
    assert lib.lrkv_mla_decode(ctypes.byref(okm), fake, ctypes.c_void_p(4096 + 8), fake, fake, fake, fake, None,
                               fake, 1 << 20, None) == lrkv.LRKV_ERR_INVALID_ARG   # c not 16-byte aligned
