"""Pins for the oracle's full-RoPE decode (review §8, "Full RoPE needs a
stronger identity"; notes §2.7): the review's counterexample, the identity
rotation, an independent complex-number formulation against torch's
attention in fp64, the review's position-specific contraction, and the
relative-position property.  Mutation tests plant plausible mistakes (a
reversed turn, rotated values, rotation in rank space, an off-by-one
position, the half-split pairing) in the oracle and check that a pin fails.
Nothing here calls the CUDA library."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import read_golden
from oracle import lrkv_oracle as O


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _case(seed, B=2, H=3, dh=8, r=4, L=9, lens=None):
    rng = np.random.default_rng(seed)
    k_s, v_s = _rand(rng, B, L, dh), _rand(rng, B, L, dh)
    z_k, z_v = _rand(rng, B, L, H, r), _rand(rng, B, L, H, r)
    b_k, b_v = _rand(rng, H, dh, r, std=1 / math.sqrt(r)), _rand(rng, H, dh, r, std=1 / math.sqrt(r))
    q = _rand(rng, B, H, dh)
    # near-cancelling keys on (0, 0): the shared row undoes most of the private one
    k_s[0] = -(z_k[0, :, 0, :] @ b_k[0].T) + 1e-3 * _rand(rng, L, dh)
    return q, k_s, v_s, z_k, z_v, b_k, b_v, (lens or [L, L - 3])


def _complex_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, lens, theta):
    """Independent formulation: the rebuilt key's pairs as complex numbers
    multiplied by exp(i j theta_k) (numpy complex arithmetic), then torch's
    scaled_dot_product_attention in float64 with the unrotated values."""
    B, H, dh = q.shape
    out = np.zeros((B, H, dh))
    lse = np.zeros((B, H))
    for b in range(B):
        L = lens[b]
        for h in range(H):
            K = np.einsum("lr,dr->ld", z_k[b, :L, h], b_k[h]) + k_s[b, :L]
            V = np.einsum("lr,dr->ld", z_v[b, :L, h], b_v[h]) + v_s[b, :L]
            kc = (K[:, 0::2] + 1j * K[:, 1::2]) * np.exp(1j * np.outer(np.arange(L), theta))
            Kr = np.empty_like(K)
            Kr[:, 0::2], Kr[:, 1::2] = kc.real, kc.imag
            scale = 1 / math.sqrt(dh)
            t = lambda a: torch.tensor(a, dtype=torch.float64)[None, None]  # noqa: E731
            out[b, h] = F.scaled_dot_product_attention(t(q[b, h][None]), t(Kr), t(V), scale=scale)[0, 0, 0].numpy()
            s = scale * (Kr @ q[b, h])
            lse[b, h] = float(torch.logsumexp(torch.tensor(s), 0))
    return out, lse


# --------------------------------------------------------------------------
# pins, each returning True when it holds (the mutation tests reuse them)

def _check_counterexample():
    """review §8 / Figure 9: B_h^T = (1, 0), z = 1, a quarter turn; the
    rotated private key is (0, 1) and its score against q = (0, 1) is 1, while
    any rank-space transform of z scores 0."""
    kv, _ = read_golden("review_s8_rope_counterexample.txt")
    q = np.array(kv["query"]).reshape(1, 1, 2)
    b_k = np.array(kv["basis_transposed"]).reshape(1, 2, 1)
    z_k = np.array(kv["latent"]).reshape(1, 1, 1, 1)
    zero_s = np.zeros((1, 1, 2))
    theta = [kv["angle"][0]]
    key = O.rope_rotate_rows(O.reconstruct_head(zero_s[0], z_k[0, :, 0, :], b_k[0]), [1], theta)
    if not np.allclose(key[0], kv["rotated_private_key"], atol=1e-15):
        return False
    # the single cache row sits at position 1 (one quarter turn)
    _, lse = O.decode_reference_rope(q, zero_s, zero_s, z_k, z_k, b_k, b_k, [1], theta=theta, pos_offset=1,
                                     scale=1.0)
    rank_space = [float(q[0, 0] @ (e * b_k[0][:, 0])) for e in (-2.0, 0.5, 1.0, 3.0)]
    return (abs(lse[0, 0] - kv["score_rotated_key"][0]) < 1e-12
            and all(abs(v - kv["score_rank_space"][0]) < 1e-15 for v in rank_space))


def _check_identity_rotation():
    """theta = 0 turns nothing: the plain decode on the same query."""
    c = _case(1)
    o1, l1 = O.decode_reference_rope(*c, theta=np.zeros(4))
    o2, l2 = O.decode_reference(*c)
    return np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


def _check_complex_formulation():
    """Against complex multiplication by exp(i j theta) and torch's attention,
    at the standard frequencies and at a large base."""
    ok = True
    for seed, base in ((2, 10000.0), (3, 50.0)):
        c = _case(seed, dh=8, r=4, L=11)
        th = O.rope_frequencies(8, base)
        o, l = O.decode_reference_rope(*c, base=base)
        o_ref, l_ref = _complex_reference(*c, th)
        ok = ok and np.allclose(o, o_ref, rtol=0, atol=1e-10) and np.allclose(l, l_ref, rtol=0, atol=1e-10)
    return ok


def _check_position_specific_contraction():
    """The review's exact option (q~ D_j^T B_h) z_j^T, never rebuilding K,
    equals the rebuilt-and-rotated definition."""
    c = _case(4, B=2, H=4, dh=8, r=4, L=13)
    o1, l1 = O.decode_reference_rope(*c)
    o2, l2 = O.decode_rope_factored(*c)
    return np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


def _check_relative_positions():
    """Scores depend only on relative positions: shifting every key by 37
    positions and turning the query 37 positions further changes nothing."""
    q, k_s, v_s, z_k, z_v, b_k, b_v, lens = _case(5)
    th = O.rope_frequencies(q.shape[2])
    q2 = np.stack([O.rope_rotate_rows(q[b], [37] * q.shape[1], th) for b in range(q.shape[0])])
    o1, l1 = O.decode_reference_rope(q, k_s, v_s, z_k, z_v, b_k, b_v, lens)
    o2, l2 = O.decode_reference_rope(q2, k_s, v_s, z_k, z_v, b_k, b_v, lens, pos_offset=37)
    return np.allclose(o1, o2, rtol=0, atol=1e-10) and np.allclose(l1, l2, rtol=0, atol=1e-10)


_PINS = [_check_counterexample, _check_identity_rotation, _check_complex_formulation,
         _check_position_specific_contraction, _check_relative_positions]


@pytest.mark.parametrize("pin", _PINS, ids=lambda f: f.__name__)
def test_rope_pin_holds(pin):
    assert pin()


def test_rope_rotation_keeps_pair_norms_and_empty_history():
    """Rotation keeps the norm of every key pair (a rotation), and an empty
    history gives out = 0 and lse = -inf."""
    c = _case(6)
    th = O.rope_frequencies(8)
    K = _rand(np.random.default_rng(0), 5, 8)
    Kr = O.rope_rotate_rows(K, np.arange(5) * 1000, th)
    assert np.allclose(K[:, 0::2] ** 2 + K[:, 1::2] ** 2, Kr[:, 0::2] ** 2 + Kr[:, 1::2] ** 2, atol=1e-12)
    o, l = O.decode_reference_rope(*c[:7], [0, 3])
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))


@pytest.mark.parametrize("mutant", ["reversed_turn", "rotated_values", "rank_space_rotation",
                                    "off_by_one_position", "half_split_pairs"])
def test_rope_planted_mistakes_are_caught(mutant, monkeypatch):
    real_rot = O.rope_rotate_rows
    real_dec = O.decode_reference_rope
    if mutant == "reversed_turn":
        monkeypatch.setattr(O, "rope_rotate_rows", lambda X, p, th: real_rot(X, -np.asarray(p, float), th))
    elif mutant == "off_by_one_position":
        monkeypatch.setattr(O, "rope_rotate_rows", lambda X, p, th: real_rot(X, np.asarray(p, float) + 1, th))
    elif mutant == "half_split_pairs":
        def half(X, p, th):
            X = np.asarray(X, float)
            d = X.shape[1]
            perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])  # (k, k + d/2) become a pair
            inv = np.argsort(perm)
            return real_rot(X[:, inv], p, th)[:, perm]
        monkeypatch.setattr(O, "rope_rotate_rows", half)
    elif mutant == "rotated_values":
        def rv(q, k_s, v_s, z_k, z_v, b_k, b_v, lens, base=10000.0, theta=None, pos_offset=0, scale=None,
               pairs=None):
            th = O.rope_frequencies(q.shape[2], base) if theta is None else theta
            L = np.asarray(v_s).shape[1]
            vr = np.stack([real_rot(O.reconstruct_head(np.asarray(v_s[b], float), np.asarray(z_v[b, :, 0], float) * 0,
                                                        np.zeros((q.shape[2], z_v.shape[-1]))),
                                    np.arange(L) + pos_offset, th) for b in range(q.shape[0])])
            return real_dec(q, k_s, vr, z_k, z_v, b_k, b_v, lens, base, theta, pos_offset, scale, pairs)
        monkeypatch.setattr(O, "decode_reference_rope", rv)
    elif mutant == "rank_space_rotation":
        # the commute the review rejects: turn the shared row at full width but
        # the latent only in rank space (pairs of latent coordinates; a single
        # latent coordinate is left as it is)
        def rank_space(q, k_s, v_s, z_k, z_v, b_k, b_v, lens, base=10000.0, theta=None, pos_offset=0, scale=None,
                       pairs=None):
            q, k_s, v_s, z_k, z_v, b_k, b_v = (np.asarray(a, float) for a in (q, k_s, v_s, z_k, z_v, b_k, b_v))
            B, H, dh = q.shape
            r = z_k.shape[-1]
            th = O.rope_frequencies(dh, base) if theta is None else np.asarray(theta, float)
            scale = 1 / math.sqrt(dh) if scale is None else scale
            out, lse = np.zeros((B, H, dh)), np.zeros((B, H))
            for b in range(B):
                L = lens[b]
                pos = np.arange(L) + pos_offset
                for h in range(H):
                    zr = real_rot(z_k[b, :L, h], pos, th[: r // 2]) if r >= 2 else z_k[b, :L, h]
                    K = real_rot(k_s[b, :L], pos, th) + zr @ b_k[h].T
                    V = v_s[b, :L] + z_v[b, :L, h] @ b_v[h].T
                    s = scale * (K @ q[b, h])
                    m = s.max()
                    w = np.exp(s - m)
                    out[b, h], lse[b, h] = (w @ V) / w.sum(), m + math.log(w.sum())
            return out, lse
        monkeypatch.setattr(O, "decode_reference_rope", rank_space)
    assert not all(c() for c in _PINS), mutant
