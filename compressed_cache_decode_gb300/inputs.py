"""Seeded synthetic workloads for LRKV factored-cache attention.

This module only draws random numbers and lays them out in the cache layout;
it holds none of the attention arithmetic.  The same tensors (already rounded
once to the storage dtype) feed both the CUDA library and the fp64 oracle.

Layouts (row-major, tokens contiguous per sequence):
  q        [B, H, d_h]            decode query, storage dtype
  q        [B, T, H, d_h]         prefill queries, storage dtype
  k_s, v_s [B, max_len, d_h]      shared key/value rows
  z_k, z_v [B, max_len, H, r]     per-head rank-r latents
  b_k, b_v [H, d_h, r]            per-head reconstruction bases B_h
  seq_lens [B] int32              visible history length per sequence
  x        [B, T, d]              layer input (append workload)
  w_sk, w_sv [d_h, d]; u_k, u_v [H*r, d] (output-major; row h*r+c = column c of U_h)

Workloads mirror the shapes the LRKV pages discuss: head width 128, 16-32
heads, ranks that keep the cache near half of MHA, and contexts from 4K to
64K tokens (Low-Rank Key Value Attention reading notes, §2.5 table of Table-7
ranks; technical review, §4).  Draw order is fixed: per-sequence lengths (when
ragged), then k_s, v_s, z_k, z_v, q, B^K, B^V, then workload extras.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str              # "decode" or "prefill"
    batch: int
    heads: int
    head_dim: int
    rank: int
    max_len: int
    dtype: str             # "f32" or "bf16" (storage dtype of q, cache and bases)
    ragged: Optional[tuple] = None      # (lo, hi) inclusive per-sequence lengths
    outlier_frac: float = 0.0           # fraction of k_s rows scaled by outlier_mag
    outlier_mag: float = 1.0
    q_len: int = 1                      # prefill query count
    d_model: int = 0                    # prefill: layer width d for the append GEMM

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


# The five workloads.  The first is small enough for the oracle in seconds; the
# decode bench's headline runs the largest one-GPU decode (the fourth) and
# times the other three decodes as legs of the same run.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("decode_f32_b1_h4_d16_r4_L64", "decode", 1, 4, 16, 4, 64, "f32"),
        Workload("decode_bf16_b8_h16_d64_r28_L4096", "decode", 8, 16, 64, 28, 4096, "bf16"),
        Workload("decode_bf16_b32_h32_d128_r56_ragged1k-8k", "decode", 32, 32, 128, 56, 8192,
                 "bf16", ragged=(1024, 8192)),
        Workload("decode_bf16_b4_h32_d128_r48_L65536_outliers", "decode", 4, 32, 128, 48, 65536,
                 "bf16", outlier_frac=0.05, outlier_mag=8.0),
        Workload("prefill_bf16_b2_t4096_h32_d128_r64_dmodel4096", "prefill", 2, 32, 128, 64, 4096,
                 "bf16", q_len=4096, d_model=4096),
    ]
}

DECODE_BENCH_WORKLOAD = "decode_bf16_b4_h32_d128_r48_L65536_outliers"
DECODE_LEG_WORKLOADS = ("decode_f32_b1_h4_d16_r4_L64", "decode_bf16_b8_h16_d64_r28_L4096",
                        "decode_bf16_b32_h32_d128_r56_ragged1k-8k")
PREFILL_WORKLOAD = "prefill_bf16_b2_t4096_h32_d128_r64_dmodel4096"


def _normal(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_decode_inputs(w: Workload, seed: int = 0, batch: Optional[int] = None,
                       max_len: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw one decode workload on the CPU, rounded once to the storage dtype.

    `batch`/`max_len` override the workload size (tests use smaller copies of
    the same recipe).  Cache entries and q ~ N(0,1); B^K, B^V ~ N(0, 1/r).
    """
    B = batch if batch is not None else w.batch
    L = max_len if max_len is not None else w.max_len
    H, dh, r = w.heads, w.head_dim, w.rank
    gen = torch.Generator().manual_seed(seed)
    if w.ragged is not None:
        lo, hi = w.ragged
        lo, hi = min(lo, L), min(hi, L)
        seq_lens = torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64).to(torch.int32)
    else:
        seq_lens = torch.full((B,), L, dtype=torch.int32)
    k_s = _normal(gen, (B, L, dh))
    v_s = _normal(gen, (B, L, dh))
    z_k = _normal(gen, (B, L, H, r))
    z_v = _normal(gen, (B, L, H, r))
    q = _normal(gen, (B, H, dh))
    bstd = 1.0 / math.sqrt(r) if r > 0 else 1.0
    b_k = _normal(gen, (H, dh, r), bstd)
    b_v = _normal(gen, (H, dh, r), bstd)
    if w.outlier_frac > 0.0:
        n_out = int(round(w.outlier_frac * L))
        for b in range(B):
            rows = torch.randperm(L, generator=gen)[:n_out]
            k_s[b, rows] *= w.outlier_mag
    dt = w.torch_dtype
    return dict(q=q.to(dt), k_s=k_s.to(dt), v_s=v_s.to(dt), z_k=z_k.to(dt), z_v=z_v.to(dt),
                b_k=b_k.to(dt), b_v=b_v.to(dt), seq_lens=seq_lens)


def make_prefill_inputs(w: Workload, seed: int = 0, batch: Optional[int] = None,
                        q_len: Optional[int] = None, d_model: Optional[int] = None
                        ) -> Dict[str, torch.Tensor]:
    """Draw one prefill workload: layer input x and the projection weights that
    the append step turns into the factored cache, plus the queries.

    x ~ N(0,1); W_sK, W_sV, U^K, U^V ~ N(0, 1/d); B^K, B^V ~ N(0, 1/r); q ~ N(0,1)
    drawn directly (the workload gives no W^Q).  Draw order: x, W_sK, W_sV,
    U^K, U^V, q, B^K, B^V.  The projection weights are stored output-major
    (w_sk [d_h, d], u_k [H*r, d], row h*r + c = column c of U_h), the layout
    the append entry point reads.
    """
    B = batch if batch is not None else w.batch
    T = q_len if q_len is not None else w.q_len
    d = d_model if d_model is not None else w.d_model
    H, dh, r = w.heads, w.head_dim, w.rank
    gen = torch.Generator().manual_seed(seed)
    wstd = 1.0 / math.sqrt(d)
    x = _normal(gen, (B, T, d))
    w_sk = _normal(gen, (dh, d), wstd)
    w_sv = _normal(gen, (dh, d), wstd)
    u_k = _normal(gen, (H * r, d), wstd)
    u_v = _normal(gen, (H * r, d), wstd)
    q = _normal(gen, (B, T, H, dh))
    bstd = 1.0 / math.sqrt(r) if r > 0 else 1.0
    b_k = _normal(gen, (H, dh, r), bstd)
    b_v = _normal(gen, (H, dh, r), bstd)
    dt = w.torch_dtype
    return dict(x=x.to(dt), w_sk=w_sk.to(dt), w_sv=w_sv.to(dt), u_k=u_k.to(dt), u_v=u_v.to(dt),
                q=q.to(dt), b_k=b_k.to(dt), b_v=b_v.to(dt),
                seq_lens=torch.full((B,), T, dtype=torch.int32),
                start_pos=torch.zeros((B,), dtype=torch.int32))


def random_decode_case(seed: int, batch: int, heads: int, head_dim: int, rank: int,
                       max_len: int, dtype: str, lens=None, q_scale: float = 1.0
                       ) -> Dict[str, torch.Tensor]:
    """Small randomised decode case (parity sweeps).  `lens` may list explicit
    per-sequence lengths (0 allowed); otherwise lengths are uniform in
    [1, max_len]."""
    gen = torch.Generator().manual_seed(seed)
    if lens is None:
        seq_lens = torch.randint(1, max_len + 1, (batch,), generator=gen, dtype=torch.int64)
    else:
        seq_lens = torch.tensor(lens, dtype=torch.int64)
    k_s = _normal(gen, (batch, max_len, head_dim))
    v_s = _normal(gen, (batch, max_len, head_dim))
    z_k = _normal(gen, (batch, max_len, heads, rank))
    z_v = _normal(gen, (batch, max_len, heads, rank))
    q = _normal(gen, (batch, heads, head_dim), q_scale)
    bstd = 1.0 / math.sqrt(rank) if rank > 0 else 1.0
    b_k = _normal(gen, (heads, head_dim, rank), bstd)
    b_v = _normal(gen, (heads, head_dim, rank), bstd)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    return dict(q=q.to(dt), k_s=k_s.to(dt), v_s=v_s.to(dt), z_k=z_k.to(dt), z_v=z_v.to(dt),
                b_k=b_k.to(dt), b_v=b_v.to(dt), seq_lens=seq_lens.to(torch.int32))


def paged_from_contiguous(case: Dict[str, torch.Tensor], page_size: int, seed: int,
                          extra_pages: int = 3) -> Dict[str, torch.Tensor]:
    """The cache of a contiguous case (max_len a multiple of page_size) laid
    out in a page pool: block j of sequence b goes to a page drawn by a seeded
    permutation; `extra_pages` unused pages and every page row never written
    hold NaN; the block table [B][max_len / page_size] (int32) maps the blocks
    of each sequence that hold any of its rows and is -1 past them."""
    k_s = case["k_s"]
    B, L = k_s.shape[0], k_s.shape[1]
    assert L % page_size == 0
    nb = L // page_size
    lens = case["seq_lens"].tolist()
    used = [(b, j) for b in range(B) for j in range(nb) if j * page_size < lens[b]]
    n_pages = len(used) + extra_pages
    gen = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_pages, generator=gen).tolist()
    table = torch.full((B, nb), -1, dtype=torch.int32)
    out = dict(case)
    for name in ("k_s", "v_s", "z_k", "z_v"):
        t = case[name]
        pool = torch.full((n_pages, page_size) + tuple(t.shape[2:]), float("nan"), dtype=t.dtype)
        for k, (b, j) in enumerate(used):
            pool[perm[k]] = t[b, j * page_size:(j + 1) * page_size]
        out[name] = pool
    for k, (b, j) in enumerate(used):
        table[b, j] = perm[k]
    out["block_table"] = table
    return out


def random_prefill_case(seed: int, batch: int, q_len: int, heads: int, head_dim: int, rank: int,
                        max_len: int, lens, dtype: str = "bf16") -> Dict[str, torch.Tensor]:
    """Small randomised prefill case: a cache of `max_len` rows per sequence
    (rows past each history are filled too, as garbage the kernels must
    ignore) and q [B, q_len, H, d_h]."""
    gen = torch.Generator().manual_seed(seed)
    k_s = _normal(gen, (batch, max_len, head_dim))
    v_s = _normal(gen, (batch, max_len, head_dim))
    z_k = _normal(gen, (batch, max_len, heads, rank))
    z_v = _normal(gen, (batch, max_len, heads, rank))
    q = _normal(gen, (batch, q_len, heads, head_dim))
    bstd = 1.0 / math.sqrt(rank) if rank > 0 else 1.0
    b_k = _normal(gen, (heads, head_dim, rank), bstd)
    b_v = _normal(gen, (heads, head_dim, rank), bstd)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    return dict(q=q.to(dt), k_s=k_s.to(dt), v_s=v_s.to(dt), z_k=z_k.to(dt), z_v=z_v.to(dt),
                b_k=b_k.to(dt), b_v=b_v.to(dt), seq_lens=torch.tensor(lens, dtype=torch.int32))


def random_dense_case(seed: int, batch: int, heads: int, kv_heads: int, head_dim: int, max_len: int, lens,
                      dtype=torch.bfloat16) -> Dict[str, torch.Tensor]:
    """Materialised K/V for the comparison decode: q [B, H, d], k, v
    [B, L, H_kv, d] ~ N(0,1); draw order k, v, q."""
    gen = torch.Generator().manual_seed(seed)
    k = _normal(gen, (batch, max_len, kv_heads, head_dim))
    v = _normal(gen, (batch, max_len, kv_heads, head_dim))
    q = _normal(gen, (batch, heads, head_dim))
    return dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), seq_lens=torch.tensor(lens, dtype=torch.int32))


def random_mla_case(seed: int, batch: int, heads: int, head_dim: int, latent_dim: int, max_len: int, lens,
                    dtype=torch.bfloat16) -> Dict[str, torch.Tensor]:
    """Latent rows and up-projections for the absorbed-MLA comparison
    decode: c [B, L, d_c] ~ N(0,1), q [B, H, d_h] ~ N(0,1), w_uk, w_uv
    [H, d_h, d_c] ~ N(0, 1/d_c); draw order c, q, w_uk, w_uv."""
    gen = torch.Generator().manual_seed(seed)
    c = _normal(gen, (batch, max_len, latent_dim))
    q = _normal(gen, (batch, heads, head_dim))
    wstd = 1.0 / math.sqrt(latent_dim)
    w_uk = _normal(gen, (heads, head_dim, latent_dim), wstd)
    w_uv = _normal(gen, (heads, head_dim, latent_dim), wstd)
    return dict(q=q.to(dtype), c=c.to(dtype), w_uk=w_uk.to(dtype), w_uv=w_uv.to(dtype),
                seq_lens=torch.tensor(lens, dtype=torch.int32))
