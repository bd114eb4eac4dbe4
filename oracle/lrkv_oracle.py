"""Plain fp64 CPU oracle for Low-Rank Key-Value attention (LRKV).

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the bench's
CPU-baseline leg may import this module.  It shares no code with the CUDA
library: it never imports the package, its binding or its kernels.

Sources, cited by page title and section:
  * "Low-Rank Key Value Attention：中文研读笔记" (reading notes, below "notes"):
    §2.1 Eqs. (2)-(5) factorisation; §2.3 decode-time cache rows; §2.4 Eqs.
    (6)-(7) associative logits/values; §2.5 Eqs. (8)-(9) cache accounting;
    §2.6 Eq. (10) K/V parameter count.
  * "Low-Rank Key Value Attention | What a shared cache can preserve"
    (technical review, below "review"): §2 attention definition with the
    causal mask; §3 Algorithm 1 (construct the factored cache), Algorithm 2
    (decode against the factored history) and the hand calculation; §4 cache
    ceiling, 2.5B byte example, TP replication.

What it computes is the plain definition: each head's full K_h and V_h are
rebuilt explicitly as K_h = S_K + R_h^K (B_h^K)^T (notes §2.1; review §3), and
then textbook masked softmax attention runs on them (review §2).  The method is
exact in real arithmetic (notes §2.4 closing remark; review §3 Algorithm 2
preamble), so the result of the factored computation must equal this one up to
rounding order.  Inputs are promoted exactly to float64 (bf16 and fp32 are
exactly representable).

Readings where the pages leave a step open:
  * scale: one 1/sqrt(d_h) for the summed logit (review §3, "Associative
    decode"); never sqrt(r).
  * one softmax over the summed logits, never two normalised branches (review
    §2 example with logits (2,0) and (0,2)).
  * decode visibility: the new token is appended before attending, so the
    visible history of sequence b is rows [0, seq_lens[b]) (notes §2.4
    pseudocode appends first).
  * prefill: query i of q_len sits at absolute position seq_lens[b]-q_len+i
    and sees keys j <= that position (bottom-right causal alignment; the pages
    only say "causal").
  * an empty history (seq_lens[b] == 0) gives out = 0 and lse = -inf.
  * no RoPE except in the *_rope functions (notes §2.7; review §8: exact
    rotation of the rebuilt keys, see the readings there).  Post-projection RMSNorm only in the
    *_normed functions (review §8, "Post-projection normalization has a cache
    cost"): the key k_j = s_j + z_j B_h^T is divided by its joint RMS
    n_{h,j} = sqrt(mean_d k_j[d]^2 + eps) (never the two parts by separate
    norms); values are not normalised; a per-head gain is the caller's, folded
    into q (the review's remark on affine gains).
  * lse is the natural-log log-sum-exp of the scaled, masked logits.
  * paged cache (review §4 and §9, page boundaries as a serving concern; the
    pages give no layout): the rows of every sequence live in fixed-size pages
    of a shared pool; logical row t of sequence b is row t mod page_size of
    page block_table[b][t div page_size].  Attention over a paged cache is
    attention over the logical rows (gather_paged).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np


def _f64(a) -> np.ndarray:
    """Exact promotion of a torch tensor or array (fp32 / bf16) to float64."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        import torch  # local: only for dtype promotion of torch inputs
        a = a.to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def default_scale(head_dim: int) -> float:
    """1/sqrt(d_h): the summed score stands for the full-width dot product
    (review §3, "Associative decode")."""
    return 1.0 / math.sqrt(head_dim)


# --------------------------------------------------------------------------
# Factorisation and cache construction
# --------------------------------------------------------------------------

def reconstruct_head(shared: np.ndarray, latent_h: np.ndarray, basis_h: np.ndarray) -> np.ndarray:
    """Materialise one head's keys (or values): K_h = S + R_h B_h^T.

    notes §2.1 Eqs. (2)-(5); review §3 "From a weight factorization to token
    coordinates".  shared [L, d_h], latent_h [L, r], basis_h [d_h, r].
    """
    return shared + latent_h @ basis_h.T


def append_reference(x, w_sk, w_sv, u_k, u_v, heads: int) -> Tuple[np.ndarray, ...]:
    """Factored cache rows for new token activations (review §3 Algorithm 1;
    notes §2.3): S_K = X W_sK, S_V = X W_sV once, and per head
    R_K[h] = X U_K[h], R_V[h] = X U_V[h], all at the tokens' own indices.

    x [B, T, d]; w_sk, w_sv [d, d_h]; u_k, u_v [d, H*r] with head h in
    columns [h*r, (h+1)*r).  Returns k_s, v_s [B, T, d_h], z_k, z_v [B, T, H, r].
    """
    x = _f64(x)
    B, T, d = x.shape
    w_sk, w_sv, u_k, u_v = (_f64(a) for a in (w_sk, w_sv, u_k, u_v))
    r = u_k.shape[1] // heads
    k_s = x @ w_sk
    v_s = x @ w_sv
    z_k = (x @ u_k).reshape(B, T, heads, r)
    z_v = (x @ u_v).reshape(B, T, heads, r)
    return k_s, v_s, z_k, z_v


def effective_projection(w_s, u, basis, h: int) -> np.ndarray:
    """W_h = W_shared + U_h B_h^T (notes §2.1 Eq. (2)); used only to pin the
    append path against the un-factored projection."""
    w_s, u, basis = _f64(w_s), _f64(u), _f64(basis)
    r = basis.shape[2]
    return w_s + u[:, h * r:(h + 1) * r] @ basis[h].T


# --------------------------------------------------------------------------
# Attention on the reconstructed heads (the definition)
# --------------------------------------------------------------------------

def _softmax_attend(s: np.ndarray, V: np.ndarray) -> Tuple[np.ndarray, float]:
    """Textbook softmax over the visible logits s [L] and weighted sum of V
    rows (review §2).  Returns (o [d_h], lse)."""
    m = np.max(s)
    w = np.exp(s - m)
    l = np.sum(w)
    return (w @ V) / l, float(m + math.log(l))


def decode_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, scale: Optional[float] = None,
                     pairs: Optional[Iterable[Tuple[int, int]]] = None):
    """One decode step for every (sequence b, head h), or only for `pairs`.

    For each pair: rebuild K_h, V_h over rows [0, seq_lens[b]), form
    s_j = scale * q_h . K_h[j], softmax, o = sum_j a_j V_h[j] (review §3
    Algorithm 2 semantics, computed by the explicit expansion).
    Returns out [B, H, d_h] and lse [B, H] (float64); pairs not computed are NaN.
    """
    q, k_s, v_s, z_k, z_v, b_k, b_v = (_f64(a) for a in (q, k_s, v_s, z_k, z_v, b_k, b_v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    out = np.full((B, H, dh), np.nan)
    lse = np.full((B, H), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = int(lens[b])
        if L == 0:
            out[b, h] = 0.0
            lse[b, h] = -np.inf
            continue
        K = reconstruct_head(k_s[b, :L], z_k[b, :L, h, :], b_k[h])
        V = reconstruct_head(v_s[b, :L], z_v[b, :L, h, :], b_v[h])
        s = scale * (K @ q[b, h])
        out[b, h], lse[b, h] = _softmax_attend(s, V)
    return out, lse


def _rms(K: np.ndarray, rms_eps: float) -> np.ndarray:
    """Root mean square of every row of K [L, d_h] with eps inside the root
    (the review's d_h n^2 = |k|^2 + d_h eps)."""
    return np.sqrt(np.mean(K * K, axis=1) + rms_eps)


def key_rms_scales(k_s, z_k, b_k, rms_eps: float) -> np.ndarray:
    """Reciprocal post-projection RMS of every cached key (review §8,
    "Post-projection normalization has a cache cost"): k_j = s_j + z_j B_h^T
    rebuilt explicitly, n_{h,j} = sqrt(mean_d k_j[d]^2 + eps).  k_s [B, L, d_h],
    z_k [B, L, H, r], b_k [H, d_h, r]; returns 1 / n [B, L, H]."""
    k_s, z_k, b_k = (_f64(a) for a in (k_s, z_k, b_k))
    B, L, dh = k_s.shape
    H = z_k.shape[2]
    out = np.empty((B, L, H))
    for b in range(B):
        for h in range(H):
            K = reconstruct_head(k_s[b], z_k[b, :, h, :], b_k[h])
            out[b, :, h] = 1.0 / _rms(K, rms_eps)
    return out


def key_rms_scales_expanded(k_s, z_k, b_k, rms_eps: float) -> np.ndarray:
    """The same scale from the review's expansion of the squared norm,
    d_h n^2 = |s|^2 + 2 s B z^T + z B^T B z^T + d_h eps (shared, cross and
    private terms).  Used only to pin key_rms_scales."""
    k_s, z_k, b_k = (_f64(a) for a in (k_s, z_k, b_k))
    B, L, dh = k_s.shape
    H = z_k.shape[2]
    out = np.empty((B, L, H))
    for h in range(H):
        Bh = b_k[h]                                      # [d_h, r]
        G = Bh.T @ Bh                                    # [r, r]
        ss = np.einsum("bld,bld->bl", k_s, k_s)
        cross = 2.0 * np.einsum("bld,dc,blc->bl", k_s, Bh, z_k[:, :, h, :])
        priv = np.einsum("blc,ce,ble->bl", z_k[:, :, h, :], G, z_k[:, :, h, :])
        out[:, :, h] = 1.0 / np.sqrt((ss + cross + priv) / dh + rms_eps)
    return out


def decode_reference_normed(q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, rms_eps: float,
                            scale: Optional[float] = None,
                            pairs: Optional[Iterable[Tuple[int, int]]] = None):
    """decode_reference with post-projection RMSNorm of the keys (review §8):
    every rebuilt key row is divided by its RMS sqrt(mean k^2 + eps) before the
    scaled dot product with q; the softmax and the values are as in the plain
    decode."""
    q, k_s, v_s, z_k, z_v, b_k, b_v = (_f64(a) for a in (q, k_s, v_s, z_k, z_v, b_k, b_v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    out = np.full((B, H, dh), np.nan)
    lse = np.full((B, H), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = int(lens[b])
        if L == 0:
            out[b, h] = 0.0
            lse[b, h] = -np.inf
            continue
        K = reconstruct_head(k_s[b, :L], z_k[b, :L, h, :], b_k[h])
        K = K / _rms(K, rms_eps)[:, None]
        V = reconstruct_head(v_s[b, :L], z_v[b, :L, h, :], b_v[h])
        s = scale * (K @ q[b, h])
        out[b, h], lse[b, h] = _softmax_attend(s, V)
    return out, lse


def prefill_reference(q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, scale: Optional[float] = None,
                      pairs: Optional[Iterable[Tuple[int, int]]] = None,
                      rows: Optional[Sequence[int]] = None, rms_eps: Optional[float] = None):
    """Causal attention of q_len queries per sequence against the factored cache.

    q [B, q_len, H, d_h].  Query i of sequence b sits at absolute position
    p_i = seq_lens[b] - q_len + i and sees keys j <= p_i (causal mask of
    review §2; bottom-right alignment).  `rows` restricts the query indices
    computed.  With `rms_eps` given, every rebuilt key row is first divided by
    its RMS sqrt(mean k^2 + rms_eps) (post-projection RMSNorm of the keys,
    review §8, as in decode_reference_normed).  Returns out [B, q_len, H, d_h]
    and lse [B, H, q_len]; entries not computed are NaN.
    """
    q, k_s, v_s, z_k, z_v, b_k, b_v = (_f64(a) for a in (q, k_s, v_s, z_k, z_v, b_k, b_v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, Tq, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    out = np.full((B, Tq, H, dh), np.nan)
    lse = np.full((B, H, Tq), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    qi = list(range(Tq)) if rows is None else list(rows)
    for b, h in todo:
        L = int(lens[b])
        if L < Tq:
            raise ValueError("prefill needs seq_lens[b] >= q_len (queries are part of the history)")
        K = reconstruct_head(k_s[b, :L], z_k[b, :L, h, :], b_k[h])
        if rms_eps is not None:
            K = K / _rms(K, rms_eps)[:, None]
        V = reconstruct_head(v_s[b, :L], z_v[b, :L, h, :], b_v[h])
        for i in qi:
            p = L - Tq + i
            s = scale * (K[: p + 1] @ q[b, i, h])
            out[b, i, h], lse[b, h, i] = _softmax_attend(s, V[: p + 1])
    return out, lse


# --------------------------------------------------------------------------
# Second CPU path, used only to pin the definition above: the associative
# (factored) form of notes §2.4 Eqs. (6)-(7) / review §3 Algorithm 2.
# --------------------------------------------------------------------------

def decode_factored(q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, scale: Optional[float] = None):
    """Algorithm 2 of the review in its own order, in fp64, never rebuilding
    K_h or V_h: p = q B_K[h]; score_j = q.S_K[j] + p.R_K[h,j]; scale; one
    softmax; reduce S_V and R_V[h] with the same weights; map the private
    reduction through B_V[h]^T; add."""
    q, k_s, v_s, z_k, z_v, b_k, b_v = (_f64(a) for a in (q, k_s, v_s, z_k, z_v, b_k, b_v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    out = np.zeros((B, H, dh))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(H):
            p = q[b, h] @ b_k[h]                                   # step 02
            score = k_s[b, :L] @ q[b, h] + z_k[b, :L, h, :] @ p    # steps 03-04
            score = score * scale                                  # step 05
            m = np.max(score)
            w = np.exp(score - m)
            l = np.sum(w)
            a = w / l                                              # step 06
            shared = a @ v_s[b, :L]                                # step 07
            private = a @ z_v[b, :L, h, :]
            out[b, h] = shared + private @ b_v[h].T                # steps 08-09
            lse[b, h] = m + math.log(l)
    return out, lse


# --------------------------------------------------------------------------
# Full rotary position embedding on the factored cache (review §8, "Full RoPE
# needs a stronger identity"; notes §2.7).  The latents cannot be rotated in
# rank space for a generic basis, so the cache keeps unrotated rows and the
# rotation of key position j is applied to the rebuilt key.
#
# Readings (the pages fix none of these): theta_k = base^(-2k/d_h) for
# k = 0 .. d_h/2 - 1 with base 10000; the pairs are adjacent coordinates
# (2k, 2k+1) and the rotation of a row at position j multiplies each pair,
# read as the complex number x_{2k} + i x_{2k+1}, by exp(i j theta_k); cache
# row j sits at position j + pos_offset; the query arrives already rotated to
# its own position (the review's q~_i); values are not rotated.
# --------------------------------------------------------------------------

def rope_frequencies(head_dim: int, base: float = 10000.0) -> np.ndarray:
    """theta_k = base^(-2k/d_h), k = 0 .. d_h/2 - 1."""
    k = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-2.0 * k / head_dim)


def rope_rotate_rows(X, positions, theta) -> np.ndarray:
    """Row j of X [L, d_h] times D_{positions[j]} (row vectors): pair
    (2k, 2k+1) turned by the angle positions[j] * theta[k]:
    x'_{2k} = x_{2k} cos - x_{2k+1} sin, x'_{2k+1} = x_{2k} sin + x_{2k+1} cos."""
    X = _f64(X)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * np.asarray(theta, dtype=np.float64)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(X)
    out[:, 0::2] = X[:, 0::2] * c - X[:, 1::2] * s
    out[:, 1::2] = X[:, 0::2] * s + X[:, 1::2] * c
    return out


def decode_reference_rope(q_rot, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, base: float = 10000.0,
                          theta=None, pos_offset: int = 0, scale: Optional[float] = None,
                          pairs: Optional[Iterable[Tuple[int, int]]] = None):
    """Decode with full RoPE on the keys, computed by the definition: for
    each (sequence b, head h) rebuild K_h = S_K + Z_h B_h^T over rows
    [0, seq_lens[b]), rotate row j by D_{j + pos_offset}, score
    s_j = scale * q_rot . (K_h[j] D_j), one softmax, o = sum_j a_j V_h[j] with
    V_h = S_V + Z_v B_V^T unrotated.  q_rot [B, H, d_h] is the query already
    rotated to its position.  `theta` overrides the frequency schedule."""
    q, k_s, v_s, z_k, z_v, b_k, b_v = (_f64(a) for a in (q_rot, k_s, v_s, z_k, z_v, b_k, b_v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    th = rope_frequencies(dh, base) if theta is None else np.asarray(theta, dtype=np.float64)
    out = np.full((B, H, dh), np.nan)
    lse = np.full((B, H), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = int(lens[b])
        if L == 0:
            out[b, h] = 0.0
            lse[b, h] = -np.inf
            continue
        K = reconstruct_head(k_s[b, :L], z_k[b, :L, h, :], b_k[h])
        K = rope_rotate_rows(K, np.arange(L) + pos_offset, th)
        V = reconstruct_head(v_s[b, :L], z_v[b, :L, h, :], b_v[h])
        s = scale * (K @ q[b, h])
        out[b, h], lse[b, h] = _softmax_attend(s, V)
    return out, lse


def decode_rope_factored(q_rot, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, base: float = 10000.0,
                         theta=None, scale: Optional[float] = None):
    """The review's exact decode option in its own form, never rebuilding
    K_h: the query is turned back to each key position, u_j = q~ D_j^T, and
    the score is u_j . s_j + (u_j B_h) . z_j (the position-specific
    contraction (q~ D_j^T B_h) z_j^T); one softmax; the values as in
    decode_factored.  Used only to pin decode_reference_rope."""
    q, k_s, v_s, z_k, z_v, b_k, b_v = (_f64(a) for a in (q_rot, k_s, v_s, z_k, z_v, b_k, b_v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    th = rope_frequencies(dh, base) if theta is None else np.asarray(theta, dtype=np.float64)
    out = np.zeros((B, H, dh))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(H):
            U = rope_rotate_rows(np.tile(q[b, h], (L, 1)), -np.arange(L), th)   # rows q~ D_j^T = q~ D_{-j}
            score = np.sum(U * k_s[b, :L], axis=1) + np.sum((U @ b_k[h]) * z_k[b, :L, h, :], axis=1)
            score = score * scale
            m = np.max(score)
            w = np.exp(score - m)
            l = np.sum(w)
            a = w / l
            out[b, h] = a @ v_s[b, :L] + (a @ z_v[b, :L, h, :]) @ b_v[h].T
            lse[b, h] = m + math.log(l)
    return out, lse


# --------------------------------------------------------------------------
# Comparison decodes on the same box (review §4 "Weight count and the two
# decode regimes", §5 on absorbed MLA and optimized GQA): dense attention over
# materialised K/V with grouped heads, and MLA with the up-projections
# absorbed.  Readings: GQA query head h reads KV head h // (H / H_kv); MLA
# keeps one latent row c_j of width d_c per token for all heads,
# K_h = C W_uk[h]^T and V_h = C W_uv[h]^T with W_uk[h], W_uv[h] of shape
# [d_h, d_c]; one scale 1/sqrt(d_h); no position encoding on either (the same
# positional semantics as the LRKV decode).
# --------------------------------------------------------------------------

def dense_decode_reference(q, k, v, seq_lens, scale: Optional[float] = None,
                           pairs: Optional[Iterable[Tuple[int, int]]] = None):
    """Textbook decode over materialised K/V: q [B, H, d], k and v
    [B, L, H_kv, d]; query head h attends KV head h // (H / H_kv) over rows
    [0, seq_lens[b]).  Returns out [B, H, d], lse [B, H] (float64)."""
    q, k, v = (_f64(a) for a in (q, k, v))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, d = q.shape
    Hkv = k.shape[2]
    g = H // Hkv
    if scale is None:
        scale = default_scale(d)
    out = np.full((B, H, d), np.nan)
    lse = np.full((B, H), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = int(lens[b])
        if L == 0:
            out[b, h] = 0.0
            lse[b, h] = -np.inf
            continue
        K, V = k[b, :L, h // g], v[b, :L, h // g]
        out[b, h], lse[b, h] = _softmax_attend(scale * (K @ q[b, h]), V)
    return out, lse


def mla_decode_reference(q, c, w_uk, w_uv, seq_lens, scale: Optional[float] = None,
                         pairs: Optional[Iterable[Tuple[int, int]]] = None):
    """MLA decode by the definition: rebuild every head's keys and values from
    the shared latent rows, K_h = C W_uk[h]^T, V_h = C W_uv[h]^T (c [B, L, d_c],
    w_uk, w_uv [H, d_h, d_c]), then textbook softmax attention with q
    [B, H, d_h].  Returns out [B, H, d_h], lse [B, H]."""
    q, c, w_uk, w_uv = (_f64(a) for a in (q, c, w_uk, w_uv))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    out = np.full((B, H, dh), np.nan)
    lse = np.full((B, H), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = int(lens[b])
        if L == 0:
            out[b, h] = 0.0
            lse[b, h] = -np.inf
            continue
        K = c[b, :L] @ w_uk[h].T
        V = c[b, :L] @ w_uv[h].T
        out[b, h], lse[b, h] = _softmax_attend(scale * (K @ q[b, h]), V)
    return out, lse


def mla_decode_absorbed(q, c, w_uk, w_uv, seq_lens, scale: Optional[float] = None):
    """The absorbed form (review §5: (q_h A_h) Z^T for the scores, the values
    likewise): q_c = q_h W_uk[h] (d_c), scores q_c . c_j, o_c = sum_j a_j c_j,
    o_h = o_c W_uv[h]^T.  Used only to pin mla_decode_reference."""
    q, c, w_uk, w_uv = (_f64(a) for a in (q, c, w_uk, w_uv))
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, H, dh = q.shape
    if scale is None:
        scale = default_scale(dh)
    out = np.zeros((B, H, dh))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(H):
            qc = q[b, h] @ w_uk[h]
            s = scale * (c[b, :L] @ qc)
            m = np.max(s)
            w = np.exp(s - m)
            l = np.sum(w)
            out[b, h] = ((w / l) @ c[b, :L]) @ w_uv[h].T
            lse[b, h] = m + math.log(l)
    return out, lse


# --------------------------------------------------------------------------
# Cache and parameter accounting (notes §2.5-2.6; review §4)
# --------------------------------------------------------------------------

def cache_elems_per_token(heads: int, head_dim: int, rank: int) -> int:
    """Elements one token adds per layer: 2(d_h + H r) (notes §2.5 Eq. (8))."""
    return 2 * (head_dim + heads * rank)


def mha_elems_per_token(heads: int, head_dim: int) -> int:
    """Dense MHA: 2 H d_h per token per layer (notes §1 table)."""
    return 2 * heads * head_dim


def cache_fraction(heads: int, head_dim: int, rank: int) -> float:
    """rho = 1/H + r/d_h, the remaining fraction of the MHA cache
    (notes §2.5 Eq. (9))."""
    return 1.0 / heads + rank / head_dim


def cache_bytes(elem_bytes: int, layers: int, batch: int, length: int, heads: int,
                head_dim: int, rank: int) -> int:
    """2 s N b L (d_h + H r) bytes (notes §2.5; review §4 M_LRKV)."""
    return 2 * elem_bytes * layers * batch * length * (head_dim + heads * rank)


def mha_cache_bytes(elem_bytes: int, layers: int, batch: int, length: int, heads: int,
                    head_dim: int) -> int:
    """2 b N B T H d_h (review §2 "Where the bytes go")."""
    return 2 * elem_bytes * layers * batch * length * heads * head_dim


def rank_ceiling(head_dim: int, heads: int, target_fraction: float) -> int:
    """Largest rank within a cache budget c: floor(d_h (c - 1/H)) (review §4)."""
    return int(math.floor(head_dim * (target_fraction - 1.0 / heads) + 1e-12))


def saves_cache(heads: int, head_dim: int, rank: int) -> bool:
    """LRKV is smaller than MHA only if r < d_h (1 - 1/H) (notes §2.5)."""
    return rank < head_dim * (1.0 - 1.0 / heads)


def tp_replicated_fraction(shards: int, heads: int, head_dim: int, rank: int) -> float:
    """P/H + r/d_h when every tensor-parallel shard keeps its own copy of the
    shared block (review §4 "Tensor parallelism can replicate the shared
    block")."""
    return shards / heads + rank / head_dim


def kv_param_count(d_model: int, heads: int, head_dim: int, rank: int) -> int:
    """2 d d_h + 2 H r (d + d_h) K/V projection weights (notes §2.6 Eq. (10))."""
    return 2 * d_model * head_dim + 2 * heads * rank * (d_model + head_dim)


def kv_param_fraction(d_model: int, heads: int, head_dim: int, rank: int) -> float:
    """Ratio to MHA's 2 H d d_h K/V weights (notes §2.6; review §4)."""
    return kv_param_count(d_model, heads, head_dim, rank) / (2 * heads * d_model * head_dim)


def decode_flop_ratio(head_dim: int, rank: int, history: int) -> float:
    """C_LRKV / C_MHA ~= 1 + r/d_h + r/T (review §4 "Weight count and the two
    decode regimes")."""
    return 1.0 + rank / head_dim + rank / history


# --------------------------------------------------------------------------
# Paged cache: the logical rows of each sequence gathered from a page pool.

def gather_paged(pool, block_table, page_size: int, max_len: int) -> np.ndarray:
    """Logical cache [B, max_len, ...] of a page pool [num_pages, page_size,
    ...]: row t of sequence b is pool[block_table[b][t // page_size], t %
    page_size].  Blocks whose table entry is negative are left NaN (never
    visible when the lengths stay inside the mapped blocks)."""
    pool = _f64(pool)
    bt = np.asarray(block_table, dtype=np.int64)
    B = bt.shape[0]
    out = np.full((B, max_len) + pool.shape[2:], np.nan)
    for b in range(B):
        for t in range(max_len):
            pg = bt[b, t // page_size]
            if pg >= 0:
                out[b, t] = pool[pg, t % page_size]
    return out


def decode_reference_paged(q, k_s, v_s, z_k, z_v, b_k, b_v, block_table, page_size: int, seq_lens,
                           scale: Optional[float] = None, pairs: Optional[Iterable[Tuple[int, int]]] = None):
    """decode_reference over the logical rows of a paged cache (pools
    k_s, v_s [P, page_size, d_h] and z_k, z_v [P, page_size, H, r])."""
    max_len = np.asarray(block_table).shape[1] * page_size
    g = [gather_paged(t, block_table, page_size, max_len) for t in (k_s, v_s, z_k, z_v)]
    return decode_reference(q, g[0], g[1], g[2], g[3], b_k, b_v, seq_lens, scale=scale, pairs=pairs)


def prefill_reference_paged(q, k_s, v_s, z_k, z_v, b_k, b_v, block_table, page_size: int, seq_lens,
                            scale: Optional[float] = None, pairs: Optional[Iterable[Tuple[int, int]]] = None,
                            rows: Optional[Sequence[int]] = None):
    """prefill_reference over the logical rows of a paged cache."""
    max_len = np.asarray(block_table).shape[1] * page_size
    g = [gather_paged(t, block_table, page_size, max_len) for t in (k_s, v_s, z_k, z_v)]
    return prefill_reference(q, g[0], g[1], g[2], g[3], b_k, b_v, seq_lens, scale=scale, pairs=pairs, rows=rows)
