"""Pins for the oracle's comparison decodes (review §4 "Weight count and the
two decode regimes", §5 on absorbed MLA and optimized GQA): dense grouped
attention against torch's SDPA in fp64 with the KV heads repeated, the MQA
endpoint against the LRKV decode at rank 0, the MHA endpoint against the LRKV
decode with full-rank residuals, and MLA against its absorbed form and its
identity-projection endpoint.  Planted mistakes (a wrong head grouping, keys
for values, a transposed projection) fail a pin.  No CUDA library calls."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import lrkv_oracle as O


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _sdpa_grouped(q, k, v, lens):
    B, H, d = q.shape
    g = H // k.shape[2]
    out = np.zeros((B, H, d))
    for b in range(B):
        L = lens[b]
        for h in range(H):
            t = lambda a: torch.tensor(a, dtype=torch.float64)[None, None]  # noqa: E731
            out[b, h] = F.scaled_dot_product_attention(t(q[b, h][None]), t(k[b, :L, h // g]), t(v[b, :L, h // g]),
                                                       scale=1 / math.sqrt(d))[0, 0, 0].numpy()
    return out


def _dense_case(seed, B=2, H=8, Hkv=2, d=16, L=11):
    rng = np.random.default_rng(seed)
    return (_rand(rng, B, H, d), _rand(rng, B, L, Hkv, d), _rand(rng, B, L, Hkv, d), [L, L - 4])


def _check_dense_sdpa():
    ok = True
    for Hkv in (8, 2, 1):   # MHA, GQA, MQA
        q, k, v, lens = _dense_case(10 + Hkv, Hkv=Hkv)
        o, _ = O.dense_decode_reference(q, k, v, lens)
        ok = ok and np.allclose(o, _sdpa_grouped(q, k, v, lens), atol=1e-12, rtol=0)
    return ok


def _check_mqa_is_lrkv_rank0():
    """One KV head for all query heads equals the LRKV decode at rank 0 (the
    shared rows alone; notes §2.1, review §3)."""
    q, k, v, lens = _dense_case(20, Hkv=1)
    o1, l1 = O.dense_decode_reference(q, k, v, lens)
    B, H, d = q.shape
    z = np.zeros((B, k.shape[1], H, 0))
    o2, l2 = O.decode_reference(q, k[:, :, 0], v[:, :, 0], z, z, np.zeros((H, d, 0)), np.zeros((H, d, 0)), lens)
    return np.allclose(o1, o2, atol=1e-12, rtol=0) and np.allclose(l1, l2, atol=1e-12, rtol=0)


def _check_mha_is_lrkv_full_rank():
    """Every head its own KV equals the LRKV decode whose full-rank residuals
    reproduce the heads (shared rows zero, B_h = I; notes §2.1)."""
    q, k, v, lens = _dense_case(30, H=4, Hkv=4, d=8)
    o1, l1 = O.dense_decode_reference(q, k, v, lens)
    B, L = k.shape[:2]
    eye = np.stack([np.eye(8)] * 4)
    o2, l2 = O.decode_reference(q, np.zeros((B, L, 8)), np.zeros((B, L, 8)), k, v, eye, eye, lens)
    return np.allclose(o1, o2, atol=1e-12, rtol=0) and np.allclose(l1, l2, atol=1e-12, rtol=0)


def _mla_case(seed, B=2, H=4, dh=8, dc=12, L=10):
    rng = np.random.default_rng(seed)
    return (_rand(rng, B, H, dh), _rand(rng, B, L, dc), _rand(rng, H, dh, dc, std=1 / math.sqrt(dc)),
            _rand(rng, H, dh, dc, std=1 / math.sqrt(dc)), [L, L - 3])


def _check_mla_absorbed():
    """The absorbed contraction equals the rebuilt keys and values."""
    c = _mla_case(40)
    o1, l1 = O.mla_decode_reference(*c)
    o2, l2 = O.mla_decode_absorbed(*c)
    return np.allclose(o1, o2, atol=1e-12, rtol=0) and np.allclose(l1, l2, atol=1e-12, rtol=0)


def _check_mla_identity_is_mqa():
    """W_uk = W_uv = I (d_c = d_h): every head reads the latent rows as its
    keys and values, i.e. MQA on them."""
    rng = np.random.default_rng(50)
    B, H, d, L = 2, 3, 6, 9
    q, c = _rand(rng, B, H, d), _rand(rng, B, L, d)
    eye = np.stack([np.eye(d)] * H)
    o1, _ = O.mla_decode_reference(q, c, eye, eye, [L, 4])
    o2, _ = O.dense_decode_reference(q, c[:, :, None, :], c[:, :, None, :], [L, 4])
    return np.allclose(o1, o2, atol=1e-12, rtol=0)


_PINS = [_check_dense_sdpa, _check_mqa_is_lrkv_rank0, _check_mha_is_lrkv_full_rank, _check_mla_absorbed,
         _check_mla_identity_is_mqa]


@pytest.mark.parametrize("pin", _PINS, ids=lambda f: f.__name__)
def test_compare_pin_holds(pin):
    assert pin()


def test_empty_history():
    q, k, v, _ = _dense_case(60)
    o, l = O.dense_decode_reference(q, k, v, [0, 3])
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))


@pytest.mark.parametrize("mutant", ["wrong_grouping", "keys_for_values", "transposed_projection"])
def test_compare_planted_mistakes_are_caught(mutant, monkeypatch):
    real_dense, real_mla = O.dense_decode_reference, O.mla_decode_reference
    if mutant == "wrong_grouping":
        def bad(q, k, v, lens, scale=None, pairs=None):   # query head h reads KV head h % H_kv
            q, k, v = (np.asarray(a, float) for a in (q, k, v))
            H, Hkv = q.shape[1], k.shape[2]
            perm = [(h % Hkv) * (H // Hkv) + h // Hkv for h in range(H)]
            o, l = real_dense(q[:, perm], k, v, lens, scale, pairs)
            inv = np.argsort(perm)
            return o[:, inv], l[:, inv]
        monkeypatch.setattr(O, "dense_decode_reference", bad)
    elif mutant == "keys_for_values":
        monkeypatch.setattr(O, "dense_decode_reference", lambda q, k, v, lens, scale=None, pairs=None:
                            real_dense(q, k, k, lens, scale, pairs))
    elif mutant == "transposed_projection":
        def bad_mla(q, c, w_uk, w_uv, lens, scale=None, pairs=None):
            w = np.asarray(w_uv, float)
            w2 = np.stack([np.resize(w[h].T.reshape(-1), w[h].shape) for h in range(w.shape[0])])
            return real_mla(q, c, w_uk, w2, lens, scale, pairs)
        monkeypatch.setattr(O, "mla_decode_reference", bad_mla)
    assert not all(p() for p in _PINS), mutant
