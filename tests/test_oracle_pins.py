"""Pins for the fp64 oracle against what the LRKV pages and mathematics fix.

Nothing here calls the CUDA library.  Each pin is chosen so that a plausible
mistake in the oracle (a dropped latent term, a transposed basis, the wrong
scale, two softmaxes, a shifted causal mask) fails at least one of them; the
mutation tests at the bottom plant such mistakes and check that they are
caught.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import read_golden
from oracle import lrkv_oracle as O


def _sdpa(q, K, V, scale, mask=None):
    """torch's scaled_dot_product_attention in float64 on CPU: an independent
    textbook attention used as the reference for the MQA/MHA endpoints."""
    q, K, V = (torch.tensor(np.array(a), dtype=torch.float64) for a in (q, K, V))
    m = None if mask is None else torch.as_tensor(mask)
    return F.scaled_dot_product_attention(q, K, V, attn_mask=m, scale=scale).numpy()


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


# --------------------------------------------------------------------------
# Worked examples printed on the pages
# --------------------------------------------------------------------------

def test_hand_calculation_score_decomposition():
    """review §3 hand calculation: q=(2,1), k_s=(1,3), z=4, B=(1,-1)^T gives
    the materialised key (5,-1) and the dot product 9 = 5 + 1*4."""
    kv, _ = read_golden("review_s3_hand_calculation.txt")
    q = np.array(kv["query"]).reshape(1, 1, 2)
    k_s = np.array(kv["shared_key"]).reshape(1, 1, 2)
    z_k = np.array(kv["private_key_latent"]).reshape(1, 1, 1, 1)
    b_k = np.array(kv["basis_column"]).reshape(1, 2, 1)
    K = O.reconstruct_head(k_s[0], z_k[0, :, 0, :], b_k[0])
    assert np.array_equal(K[0], np.array(kv["materialised_key"]))
    zeros_v = np.zeros((1, 1, 2))
    zeros_zv = np.zeros((1, 1, 1, 1))
    # One visible row: lse equals the single (unscaled here) logit.
    _, lse = O.decode_reference(q, k_s, zeros_v, z_k, zeros_zv, b_k, b_k, [1], scale=1.0)
    assert lse[0, 0] == kv["full_dot"][0]
    _, lse_f = O.decode_factored(q, k_s, zeros_v, z_k, zeros_zv, b_k, b_k, [1], scale=1.0)
    assert lse_f[0, 0] == kv["full_dot"][0]
    # the two terms of Eq. (6) separately
    assert float(q[0, 0] @ k_s[0, 0]) == kv["shared_dot"][0]
    assert float((q[0, 0] @ b_k[0])[0]) == kv["projected_query"][0]


def test_hand_calculation_value_decomposition():
    """review §3 hand calculation: weights (1/4, 3/4) on private value
    coordinates (2, 6) give 5, which contributes (5,-5) through B=(1,-1)^T."""
    kv, _ = read_golden("review_s3_hand_calculation.txt")
    w = kv["value_weights"]
    # logits 0 and ln(w1/w0) give exactly those weights; keys carry them
    q = np.array([1.0, 0.0]).reshape(1, 1, 2)
    k_s = np.array([[0.0, 0.0], [math.log(w[1] / w[0]), 0.0]]).reshape(1, 2, 2)
    z_k = np.zeros((1, 2, 1, 1))
    v_s = np.zeros((1, 2, 2))
    z_v = np.array(kv["private_value_latents"]).reshape(1, 2, 1, 1)
    b = np.array(kv["basis_column"]).reshape(1, 2, 1)
    for fn in (O.decode_reference, O.decode_factored):
        out, _ = fn(q, k_s, v_s, z_k, z_v, b, b, [2], scale=1.0)
        np.testing.assert_allclose(out[0, 0], kv["private_value_contribution"], rtol=0, atol=1e-13)
    assert w[0] * kv["private_value_latents"][0] + w[1] * kv["private_value_latents"][1] == \
        kv["weighted_private_latent"][0]


def test_single_softmax_over_summed_logits():
    """review §2: shared logits (2,0) plus private logits (0,2) give uniform
    weights; either branch normalised alone concentrates on one token."""
    kv, _ = read_golden("review_s2_summed_logits.txt")
    q = np.array([1.0, 0.0]).reshape(1, 1, 2)
    k_s = np.array([[kv["shared_logits"][0], 0.0], [kv["shared_logits"][1], 0.0]]).reshape(1, 2, 2)
    b_k = np.array([1.0, 0.0]).reshape(1, 2, 1)                 # p = q B = 1
    z_k = np.array(kv["private_logits"]).reshape(1, 2, 1, 1)
    v_s = np.eye(2).reshape(1, 2, 2)                            # o = the weights
    z_v = np.zeros((1, 2, 1, 1))
    out, _ = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_k, [2], scale=1.0)
    np.testing.assert_allclose(out[0, 0], kv["summed_weights"], atol=1e-15)
    # the wrong reading: normalise each branch and add (or average) them
    e_s = np.exp(kv["shared_logits"]) / np.exp(kv["shared_logits"]).sum()
    assert abs(e_s[0] - 0.5) > 0.3


# --------------------------------------------------------------------------
# Endpoints of the rank (notes §2.1; review §3): r=0 is MQA, r=d_h reaches MHA
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1])
def test_rank_zero_is_mqa(seed):
    rng = np.random.default_rng(seed)
    B, H, dh, L = 2, 3, 8, 11
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    empty = np.zeros((B, L, H, 0))
    b0 = np.zeros((H, dh, 0))
    lens = [L, 7]
    out, lse = O.decode_reference(q, k_s, v_s, empty, empty, b0, b0, lens)
    for b in range(B):
        Lb = lens[b]
        ref = _sdpa(q[b][:, None, :], np.broadcast_to(k_s[b, :Lb], (H, Lb, dh)),
                    np.broadcast_to(v_s[b, :Lb], (H, Lb, dh)), 1 / math.sqrt(dh))[:, 0]
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)
        s = (q[b] @ k_s[b, :Lb].T) / math.sqrt(dh)
        np.testing.assert_allclose(lse[b], np.log(np.exp(s).sum(-1)), rtol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_full_rank_reproduces_mha(seed):
    """Given arbitrary per-head K_h, V_h, pick any S and invertible B_h and set
    z = (K_h - S) B_h^{-T}; the LRKV head then equals MHA on K_h, V_h."""
    rng = np.random.default_rng(seed)
    B, H, dh, L = 2, 4, 6, 9
    r = dh
    q = _rand(rng, B, H, dh)
    Kmha, Vmha = _rand(rng, B, H, L, dh), _rand(rng, B, H, L, dh)
    S_k, S_v = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    Bk = _rand(rng, H, dh, r) + 3 * np.eye(dh)
    Bv = _rand(rng, H, dh, r) + 3 * np.eye(dh)
    z_k = np.empty((B, L, H, r))
    z_v = np.empty((B, L, H, r))
    for h in range(H):
        z_k[:, :, h, :] = np.linalg.solve(Bk[h], (Kmha[:, h] - S_k).reshape(-1, dh).T).T.reshape(B, L, r)
        z_v[:, :, h, :] = np.linalg.solve(Bv[h], (Vmha[:, h] - S_v).reshape(-1, dh).T).T.reshape(B, L, r)
    out, _ = O.decode_reference(q, S_k, S_v, z_k, z_v, Bk, Bv, [L, L])
    ref = _sdpa(q[:, :, None, :], Kmha, Vmha, 1 / math.sqrt(dh))[:, :, 0]
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-10)


def test_zero_basis_is_mqa():
    """B_h = 0 removes every private term whatever the latents hold."""
    rng = np.random.default_rng(5)
    B, H, dh, r, L = 1, 3, 8, 4, 10
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b0 = np.zeros((H, dh, r))
    out, _ = O.decode_reference(q, k_s, v_s, z_k, z_v, b0, b0, [L])
    ref = _sdpa(q[0][:, None, :], np.broadcast_to(k_s[0], (H, L, dh)),
                np.broadcast_to(v_s[0], (H, L, dh)), 1 / math.sqrt(dh))[:, 0]
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Exactness of the associative form (notes §2.4; review §3 Algorithm 2)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_factored_equals_reconstructed(seed):
    rng = np.random.default_rng(100 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    dh, r, L = int(rng.integers(2, 9)), int(rng.integers(1, 5)), 16
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    lens = rng.integers(0, L + 1, size=B)
    o1, l1 = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, lens)
    o2, l2 = O.decode_factored(q, k_s, v_s, z_k, z_v, b_k, b_v, lens)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)


def test_near_cancelling_key_terms():
    """Shared and private key parts that nearly cancel (review §9 proposes this
    case): the full key is a small difference of large terms."""
    rng = np.random.default_rng(7)
    B, H, dh, r, L = 1, 2, 4, 4, 12
    q = _rand(rng, B, H, dh)
    b_k = np.stack([np.eye(dh)] * H)
    big = 1e3 * _rand(rng, B, L, dh)
    k_s = big.copy()
    z_k = np.stack([-big[0] + 1e-3 * _rand(rng, L, dh) for _ in range(H)], axis=1)[None]
    v_s, z_v = _rand(rng, B, L, dh), _rand(rng, B, L, H, r)
    o1, l1 = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_k, [L])
    o2, l2 = O.decode_factored(q, k_s, v_s, z_k, z_v, b_k, b_k, [L])
    np.testing.assert_allclose(o1, o2, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(l1, l2, rtol=1e-9, atol=1e-9)


def test_gauge_invariance():
    """U_h -> U_h C, B_h -> B_h C^{-T} leaves the residual unchanged
    (notes §4.6): on cached latents, z -> z C, B -> B C^{-T}."""
    rng = np.random.default_rng(11)
    B, H, dh, r, L = 2, 3, 8, 4, 10
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    C = _rand(rng, H, r, r) + 2 * np.eye(r)
    Cinv_T = np.linalg.inv(C).transpose(0, 2, 1)
    z_k2 = np.einsum("blhc,hcd->blhd", z_k, C)
    z_v2 = np.einsum("blhc,hcd->blhd", z_v, C)
    b_k2 = np.einsum("hdc,hce->hde", b_k, Cinv_T)
    b_v2 = np.einsum("hdc,hce->hde", b_v, Cinv_T)
    o1, l1 = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [L, 6])
    o2, l2 = O.decode_reference(q, k_s, v_s, z_k2, z_v2, b_k2, b_v2, [L, 6])
    np.testing.assert_allclose(o1, o2, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(l1, l2, rtol=1e-10, atol=1e-10)


# --------------------------------------------------------------------------
# Closed forms of softmax attention
# --------------------------------------------------------------------------

def test_single_row_history():
    rng = np.random.default_rng(3)
    B, H, dh, r = 1, 2, 8, 3
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, 1, dh), _rand(rng, B, 1, dh)
    z_k, z_v = _rand(rng, B, 1, H, r), _rand(rng, B, 1, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    out, lse = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [1])
    for h in range(H):
        Vh = v_s[0, 0] + b_v[h] @ z_v[0, 0, h]
        Kh = k_s[0, 0] + b_k[h] @ z_k[0, 0, h]
        np.testing.assert_allclose(out[0, h], Vh, rtol=1e-14, atol=1e-14)
        assert abs(lse[0, h] - q[0, h] @ Kh / math.sqrt(dh)) < 1e-13


def test_zero_query_averages_values():
    rng = np.random.default_rng(4)
    B, H, dh, r, L = 1, 2, 8, 3, 13
    q = np.zeros((B, H, dh))
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    out, lse = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [L])
    for h in range(H):
        mean_v = v_s[0].mean(0) + b_v[h] @ z_v[0, :, h].mean(0)
        np.testing.assert_allclose(out[0, h], mean_v, rtol=1e-13, atol=1e-13)
        assert abs(lse[0, h] - math.log(L)) < 1e-13


def test_logit_shift_invariance():
    """Adding u with q.u = c to every shared key shifts all logits by
    c*scale: o is unchanged, lse moves by exactly that amount."""
    rng = np.random.default_rng(6)
    B, H, dh, r, L = 1, 1, 8, 3, 9
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    u = q[0, 0] / (q[0, 0] @ q[0, 0]) * 2.5           # q.u = 2.5
    o1, l1 = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [L])
    o2, l2 = O.decode_reference(q, k_s + u, v_s, z_k, z_v, b_k, b_v, [L])
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    assert abs((l2 - l1)[0, 0] - 2.5 / math.sqrt(dh)) < 1e-12


def test_empty_history():
    rng = np.random.default_rng(8)
    B, H, dh, r, L = 2, 2, 4, 2, 5
    args = [_rand(rng, B, H, dh), _rand(rng, B, L, dh), _rand(rng, B, L, dh),
            _rand(rng, B, L, H, r), _rand(rng, B, L, H, r), _rand(rng, H, dh, r), _rand(rng, H, dh, r)]
    out, lse = O.decode_reference(*args, [0, L])
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


# --------------------------------------------------------------------------
# Prefill (causal) against torch SDPA with an explicit mask
# --------------------------------------------------------------------------

@pytest.mark.parametrize("extra", [0, 5])
def test_prefill_matches_masked_sdpa(extra):
    """Queries are the last q_len tokens of the history; query i at position
    L - q_len + i sees keys j <= that position."""
    rng = np.random.default_rng(9 + extra)
    B, H, dh, r, Tq = 1, 2, 8, 3, 7
    L = Tq + extra
    q = _rand(rng, B, Tq, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    out, lse = O.prefill_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [L])
    mask = np.zeros((Tq, L), dtype=bool)
    for i in range(Tq):
        mask[i, : L - Tq + i + 1] = True
    for h in range(H):
        Kh = k_s[0] + z_k[0, :, h] @ b_k[h].T
        Vh = v_s[0] + z_v[0, :, h] @ b_v[h].T
        ref = _sdpa(q[0, :, h], Kh, Vh, 1 / math.sqrt(dh), mask=mask)
        np.testing.assert_allclose(out[0, :, h], ref, rtol=1e-12, atol=1e-12)
    # the last query row equals a decode step over the whole history
    od, ld = O.decode_reference(q[:, -1], k_s, v_s, z_k, z_v, b_k, b_v, [L])
    np.testing.assert_allclose(out[0, -1], od[0], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse[0, :, -1], ld[0], rtol=1e-13, atol=1e-13)
    # the first query of a square prefill sees only key 0
    if extra == 0:
        for h in range(H):
            np.testing.assert_allclose(out[0, 0, h], v_s[0, 0] + b_v[h] @ z_v[0, 0, h], atol=1e-13)


# --------------------------------------------------------------------------
# Append (Algorithm 1): the cached rows rebuild X W_h exactly
# --------------------------------------------------------------------------

def test_append_rebuilds_effective_projection():
    """X W_h = X W_s + (X U_h) B_h^T (review §3; notes §2.1): the cached rows
    and B_h must rebuild the un-factored projection of each head."""
    rng = np.random.default_rng(12)
    B, T, d, H, dh, r = 2, 5, 16, 3, 4, 2
    x = _rand(rng, B, T, d)
    w_sk, w_sv = _rand(rng, d, dh), _rand(rng, d, dh)
    u_k, u_v = _rand(rng, d, H * r), _rand(rng, d, H * r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    k_s, v_s, z_k, z_v = O.append_reference(x, w_sk, w_sv, u_k, u_v, H)
    for h in range(H):
        Wk = w_sk + u_k[:, h * r:(h + 1) * r] @ b_k[h].T
        Wv = w_sv + u_v[:, h * r:(h + 1) * r] @ b_v[h].T
        np.testing.assert_allclose(k_s + z_k[:, :, h] @ b_k[h].T, x @ Wk, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(v_s + z_v[:, :, h] @ b_v[h].T, x @ Wv, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(O.effective_projection(w_sk, u_k, b_k, h), Wk, atol=1e-14)


def test_append_small_integers():
    """Exact integer case: one token, d=2, d_h=1, H=2, r=1."""
    x = np.array([[[1.0, 2.0]]])
    w_sk = np.array([[3.0], [4.0]])               # k_s = 1*3 + 2*4 = 11
    w_sv = np.array([[1.0], [-1.0]])              # v_s = -1
    u_k = np.array([[1.0, 0.0], [0.0, 1.0]])      # z_k = (1, 2): head 0 -> 1, head 1 -> 2
    u_v = np.array([[2.0, 1.0], [1.0, 2.0]])      # z_v = (4, 5)
    k_s, v_s, z_k, z_v = O.append_reference(x, w_sk, w_sv, u_k, u_v, heads=2)
    assert k_s[0, 0, 0] == 11 and v_s[0, 0, 0] == -1
    assert list(z_k[0, 0, :, 0]) == [1, 2] and list(z_v[0, 0, :, 0]) == [4, 5]


# --------------------------------------------------------------------------
# Mutation checks: plant a mistake in the oracle, see at least one pin fail
# --------------------------------------------------------------------------

def _check_mha_endpoint():
    rng = np.random.default_rng(21)
    B, H, dh, L = 1, 2, 4, 6
    q = _rand(rng, B, H, dh)
    Kmha, Vmha = _rand(rng, B, H, L, dh), _rand(rng, B, H, L, dh)
    S = np.zeros((B, L, dh))
    Bk = _rand(rng, H, dh, dh) + 3 * np.eye(dh)
    z_k = np.empty((B, L, H, dh))
    z_v = np.empty((B, L, H, dh))
    for h in range(H):
        z_k[0, :, h] = np.linalg.solve(Bk[h], Kmha[0, h].T).T
        z_v[0, :, h] = np.linalg.solve(Bk[h], Vmha[0, h].T).T
    ref = _sdpa(q[:, :, None, :], Kmha, Vmha, 1 / math.sqrt(dh))[:, :, 0]
    out, _ = O.decode_reference(q, S, S, z_k, z_v, Bk, Bk, [L])
    return np.allclose(out, ref, rtol=1e-9, atol=1e-9)


def _check_single_row_scale():
    rng = np.random.default_rng(22)
    B, H, dh, r = 1, 1, 8, 3
    q = _rand(rng, B, H, dh)
    k_s, v_s = _rand(rng, B, 1, dh), _rand(rng, B, 1, dh)
    z_k, z_v = _rand(rng, B, 1, H, r), _rand(rng, B, 1, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    _, lse = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [1])
    Kh = k_s[0, 0] + b_k[0] @ z_k[0, 0, 0]
    return abs(lse[0, 0] - q[0, 0] @ Kh / math.sqrt(dh)) < 1e-12


def _check_summed_logits():
    q = np.array([1.0, 0.0]).reshape(1, 1, 2)
    k_s = np.array([[2.0, 0.0], [0.0, 0.0]]).reshape(1, 2, 2)
    b_k = np.array([1.0, 0.0]).reshape(1, 2, 1)
    z_k = np.array([0.0, 2.0]).reshape(1, 2, 1, 1)
    out, _ = O.decode_reference(q, k_s, np.eye(2).reshape(1, 2, 2), z_k, np.zeros((1, 2, 1, 1)),
                                b_k, b_k, [2], scale=1.0)
    return np.allclose(out[0, 0], [0.5, 0.5], atol=1e-12)


def _check_prefill_mask():
    rng = np.random.default_rng(23)
    B, H, dh, r, Tq, L = 1, 1, 4, 2, 5, 8
    q = _rand(rng, B, Tq, H, dh)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    out, _ = O.prefill_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, [L])
    mask = np.tril(np.ones((Tq, L), dtype=bool), k=L - Tq)
    Kh = k_s[0] + z_k[0, :, 0] @ b_k[0].T
    Vh = v_s[0] + z_v[0, :, 0] @ b_v[0].T
    ref = _sdpa(q[0, :, 0], Kh, Vh, 1 / math.sqrt(dh), mask=mask)
    return np.allclose(out[0, :, 0], ref, rtol=1e-10, atol=1e-10)


_PINS = [_check_mha_endpoint, _check_single_row_scale, _check_summed_logits, _check_prefill_mask]


def test_pins_pass_on_the_oracle():
    assert all(c() for c in _PINS)


@pytest.mark.parametrize("mutant", ["transposed_basis", "dropped_latent", "sqrt_r_scale",
                                    "two_softmaxes", "shifted_mask", "sign_flip"])
def test_planted_mistakes_are_caught(mutant, monkeypatch):
    if mutant == "transposed_basis":
        monkeypatch.setattr(O, "reconstruct_head", lambda s, z, b: s + (z @ b if z.shape[1] == b.shape[0] else z @ b.T * 1.5))
    elif mutant == "dropped_latent":
        monkeypatch.setattr(O, "reconstruct_head", lambda s, z, b: s)
    elif mutant == "sign_flip":
        monkeypatch.setattr(O, "reconstruct_head", lambda s, z, b: s - z @ b.T)
    elif mutant == "sqrt_r_scale":
        monkeypatch.setattr(O, "default_scale", lambda dh: 1.0 / math.sqrt(3))
    elif mutant == "two_softmaxes":
        real = O.decode_reference

        def two(q, k_s, v_s, z_k, z_v, b_k, b_v, lens, scale=None, pairs=None):
            zero_b = np.zeros_like(np.asarray(b_k, float))
            zero_s = np.zeros_like(np.asarray(k_s, float))
            o1, _ = real(q, k_s, v_s, z_k, z_v, zero_b, b_v, lens, scale)   # shared logits only
            o2, _ = real(q, zero_s, v_s, z_k, z_v, b_k, b_v, lens, scale)   # private logits only
            return 0.5 * (o1 + o2), None
        monkeypatch.setattr(O, "decode_reference", two)
    elif mutant == "shifted_mask":
        orig = O._softmax_attend
        monkeypatch.setattr(O, "_softmax_attend",
                            lambda s, V: orig(s[:-1], V[:-1]) if len(s) > 1 else orig(s, V))
    assert not all(c() for c in _PINS), mutant


# --------------------------------------------------------------------------
# Post-projection RMSNorm of the keys (review §8, "Post-projection
# normalization has a cache cost"): the oracle's joint reciprocal scale and
# the normalised decode.

def _norm_case(seed):
    rng = np.random.default_rng(seed)
    B, H, dh, r, L = 2, 3, 8, 4, 7
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r), _rand(rng, H, dh, r)
    # head 0 of sequence 0: shared part nearly cancelling the private one, so
    # the cross term of the expansion carries the norm
    k_s[0] = -(z_k[0, :, 0, :] @ b_k[0].T) + 1e-3 * _rand(rng, L, dh)
    q = _rand(rng, B, H, dh)
    return q, k_s, v_s, z_k, z_v, b_k, b_v, [L, L - 2]


def _check_norm_expansion():
    """The scale from the rebuilt key equals the review's expansion
    |s|^2 + 2 s B z^T + z B^T B z^T (with and without eps)."""
    _, k_s, _, z_k, _, b_k, _, _ = _norm_case(31)
    ok = True
    for eps in (0.0, 1e-3):
        a = O.key_rms_scales(k_s, z_k, b_k, eps)
        e = O.key_rms_scales_expanded(k_s, z_k, b_k, eps)
        ok = ok and np.allclose(a, e, rtol=1e-6, atol=0)
    return ok


def _check_norm_unit_rms_is_plain():
    """Keys whose rows already have RMS 1 (eps 0): the normalised decode equals
    the plain one."""
    q, k_s, v_s, z_k, z_v, b_k, b_v, lens = _norm_case(32)
    H = 1
    q, z_k, z_v, b_k, b_v = q[:, :H], z_k[:, :, :H], z_v[:, :, :H], b_k[:H], b_v[:H]
    K = k_s + np.einsum("blc,dc->bld", z_k[:, :, 0, :], b_k[0])
    c = 1.0 / np.sqrt(np.mean(K * K, axis=2))           # per (b, j): scales s_j and z_j together
    k_s, z_k = k_s * c[:, :, None], z_k * c[:, :, None, None]
    plain, _ = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, lens)
    normed, _ = O.decode_reference_normed(q, k_s, v_s, z_k, z_v, b_k, b_v, lens, 0.0)
    return np.allclose(plain, normed, rtol=1e-10, atol=1e-12)


def _check_norm_scale_invariance():
    """eps 0: scaling every key (shared and private parts) by 3.7 changes
    nothing after the norm, while the plain decode changes."""
    q, k_s, v_s, z_k, z_v, b_k, b_v, lens = _norm_case(33)
    a, la = O.decode_reference_normed(q, k_s, v_s, z_k, z_v, b_k, b_v, lens, 0.0)
    b, lb = O.decode_reference_normed(q, 3.7 * k_s, v_s, 3.7 * z_k, z_v, b_k, b_v, lens, 0.0)
    p1, _ = O.decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, lens)
    p2, _ = O.decode_reference(q, 3.7 * k_s, v_s, 3.7 * z_k, z_v, b_k, b_v, lens)
    return np.allclose(a, b, rtol=1e-10, atol=1e-12) and np.allclose(la, lb) and not np.allclose(p1, p2)


def _check_norm_single_row():
    """One visible row: lse = scale q . k / rms(k) for the rebuilt key."""
    q, k_s, v_s, z_k, z_v, b_k, b_v, _ = _norm_case(34)
    eps = 1e-2
    _, lse = O.decode_reference_normed(q, k_s, v_s, z_k, z_v, b_k, b_v, [1, 1], eps)
    k = k_s[1, 0] + b_k[2] @ z_k[1, 0, 2]
    want = q[1, 2] @ k / math.sqrt(np.mean(k * k) + eps) / math.sqrt(k_s.shape[2])
    return abs(lse[1, 2] - want) < 1e-12


def _check_norm_prefill_rows_are_decodes():
    """Normalised causal prefill: query i (absolute position p_i) gives the
    normalised decode of the same query over the first p_i + 1 rows; the rows
    at the end of the history are normalised by their own key only."""
    q, k_s, v_s, z_k, z_v, b_k, b_v, lens = _norm_case(35)
    rng = np.random.default_rng(36)
    B, H, dh = q.shape
    Tq = 4
    qp = _rand(rng, B, Tq, H, dh)
    eps = 1e-3
    out, lse = O.prefill_reference(qp, k_s, v_s, z_k, z_v, b_k, b_v, lens, rms_eps=eps)
    ok = True
    for i in range(Tq):
        pos = [L - Tq + i + 1 for L in lens]
        o, l = O.decode_reference_normed(qp[:, i], k_s, v_s, z_k, z_v, b_k, b_v, pos, eps)
        ok = ok and np.allclose(out[:, i], o, rtol=1e-10, atol=1e-12) and np.allclose(lse[:, :, i], l)
    plain, _ = O.prefill_reference(qp, k_s, v_s, z_k, z_v, b_k, b_v, lens)
    return ok and not np.allclose(plain, out)


_NORM_PINS = [_check_norm_expansion, _check_norm_unit_rms_is_plain, _check_norm_scale_invariance,
              _check_norm_single_row, _check_norm_prefill_rows_are_decodes]


def test_norm_pins_pass_on_the_oracle():
    assert all(c() for c in _NORM_PINS)


@pytest.mark.parametrize("mutant", ["no_sqrt", "sum_not_mean", "eps_outside", "dropped_latent"])
def test_norm_planted_mistakes_are_caught(mutant, monkeypatch):
    if mutant == "no_sqrt":
        monkeypatch.setattr(O, "_rms", lambda K, eps: np.mean(K * K, axis=1) + eps)
    elif mutant == "sum_not_mean":
        monkeypatch.setattr(O, "_rms", lambda K, eps: np.sqrt(np.sum(K * K, axis=1) + eps))
    elif mutant == "eps_outside":
        monkeypatch.setattr(O, "_rms", lambda K, eps: np.sqrt(np.mean(K * K, axis=1)) + eps)
    elif mutant == "dropped_latent":
        monkeypatch.setattr(O, "reconstruct_head", lambda s, z, b: s)
    assert not all(c() for c in _NORM_PINS), mutant


# --------------------------------------------------------------------------
# Paged cache: the oracle's gather through the block table against the cache
# the pages were scattered from (by the input generator, written apart from
# the oracle), and the paged decode against the contiguous one.

def test_paged_gather_round_trip():
    from compressed_cache_decode_gb300 import inputs
    case = inputs.random_decode_case(seed=5, batch=3, heads=2, head_dim=8, rank=4, max_len=48, dtype="f32",
                                     lens=[48, 1, 20])
    ps = 16
    paged = inputs.paged_from_contiguous(case, page_size=ps, seed=1)
    bt = paged["block_table"].numpy()
    assert len(set(bt[bt >= 0].tolist())) == (bt >= 0).sum()  # distinct pages
    for name in ("k_s", "v_s", "z_k", "z_v"):
        g = O.gather_paged(paged[name], bt, ps, 48)
        ref = case[name].double().numpy()
        for b, L in enumerate(case["seq_lens"].tolist()):
            nblk = -(-L // ps)
            assert np.array_equal(g[b, :nblk * ps], ref[b, :nblk * ps]), (name, b)
            assert np.isnan(g[b, nblk * ps:]).all()
    o1, l1 = O.decode_reference_paged(case["q"], paged["k_s"], paged["v_s"], paged["z_k"], paged["z_v"],
                                      case["b_k"], case["b_v"], bt, ps, case["seq_lens"])
    o2, l2 = O.decode_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"], case["b_k"],
                                case["b_v"], case["seq_lens"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_gather_catches_a_wrong_row_order(monkeypatch):
    """A gather that takes the block index and the row in page the wrong way
    round fails the round trip."""
    from compressed_cache_decode_gb300 import inputs
    case = inputs.random_decode_case(seed=6, batch=2, heads=1, head_dim=4, rank=2, max_len=32, dtype="f32",
                                     lens=[32, 17])
    paged = inputs.paged_from_contiguous(case, page_size=16, seed=2)
    bt = paged["block_table"].numpy()

    def bad_gather(pool, block_table, page_size, max_len):
        pool = np.asarray(pool, dtype=np.float64)
        out = np.full((block_table.shape[0], max_len) + pool.shape[2:], np.nan)
        for b in range(block_table.shape[0]):
            for t in range(max_len):
                pg = block_table[b, t % block_table.shape[1]]
                if pg >= 0:
                    out[b, t] = pool[pg, t // block_table.shape[1] % page_size]
        return out

    monkeypatch.setattr(O, "gather_paged", bad_gather)
    o1, _ = O.decode_reference_paged(case["q"], paged["k_s"], paged["v_s"], paged["z_k"], paged["z_v"],
                                     case["b_k"], case["b_v"], bt, 16, case["seq_lens"])
    o2, _ = O.decode_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"], case["b_k"],
                               case["b_v"], case["seq_lens"])
    assert not np.allclose(np.nan_to_num(o1), o2)


def test_paged_prefill_round_trip():
    """The paged prefill over the gathered logical rows equals the prefill on
    the contiguous cache the pages were scattered from."""
    from compressed_cache_decode_gb300 import inputs
    case = inputs.random_prefill_case(seed=8, batch=2, q_len=20, heads=2, head_dim=8, rank=4, max_len=64,
                                      lens=[20, 50], dtype="f32")
    paged = inputs.paged_from_contiguous(case, page_size=16, seed=3)
    o1, l1 = O.prefill_reference_paged(case["q"], paged["k_s"], paged["v_s"], paged["z_k"], paged["z_v"],
                                       case["b_k"], case["b_v"], paged["block_table"].numpy(), 16, case["seq_lens"])
    o2, l2 = O.prefill_reference(case["q"], case["k_s"], case["v_s"], case["z_k"], case["z_v"], case["b_k"],
                                 case["b_v"], case["seq_lens"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
