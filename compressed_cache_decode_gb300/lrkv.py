"""ctypes binding of the LRKV C ABI (include/lrkv.h).

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of `liblrkv.so`.  PyTorch is used for device memory and streams.  The
library is loaded on first use; if it has not been built, loading raises
(there is no CPU fallback).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblrkv.so")

LRKV_OK = 0
LRKV_ERR_INVALID_ARG = 1
LRKV_ERR_UNSUPPORTED = 2
LRKV_ERR_WORKSPACE = 3
LRKV_ERR_CUDA = 4
LRKV_ERR_TIMEOUT = 5
LRKV_ERR_DEVICE_BOUNDS = 6

LRKV_F32 = 0
LRKV_BF16 = 1

# Every symbol include/lrkv.h declares (checked by the ABI test).
EXPORTED = (
    "lrkv_abi_version",
    "lrkv_status_string",
    "lrkv_cache_elems_per_token",
    "lrkv_decode_workspace_size",
    "lrkv_decode",
    "lrkv_decode_profiled",
    "lrkv_decode_static_scratch",
    "lrkv_read_static_scratch_status",
    "lrkv_append",
    "lrkv_prefill",
    "lrkv_prefill_workspace_size",
    "lrkv_decode_step",
    "lrkv_key_scales",
    "lrkv_decode_normed",
    "lrkv_prefill_normed",
    "lrkv_decode_paged",
    "lrkv_append_paged",
    "lrkv_decode_step_paged",
    "lrkv_prefill_paged",
    "lrkv_rope_table",
    "lrkv_decode_rope_workspace_size",
    "lrkv_decode_rope",
    "lrkv_dense_decode_workspace_size",
    "lrkv_dense_decode",
    "lrkv_mla_decode_workspace_size",
    "lrkv_mla_decode",
    "lrkv_read_device_status",
)


class lrkv_dims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("rank", ctypes.c_int),
        ("max_len", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("scale", ctypes.c_float),
    ]


class lrkv_dense_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_len", ctypes.c_int), ("scale", ctypes.c_float)]


class lrkv_mla_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("latent_dim", ctypes.c_int), ("max_len", ctypes.c_int), ("scale", ctypes.c_float)]


class LRKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liblrkv.so (once).  Raises FileNotFoundError if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} is missing: build it with `python -m compressed_cache_decode_gb300.build` "
            "(the LRKV path has no CPU fallback)")
    lib = ctypes.CDLL(p)
    vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    dims_p = ctypes.POINTER(lrkv_dims)
    lib.lrkv_abi_version.restype = ctypes.c_int
    lib.lrkv_abi_version.argtypes = []
    lib.lrkv_status_string.restype = ctypes.c_char_p
    lib.lrkv_status_string.argtypes = [ctypes.c_int]
    lib.lrkv_cache_elems_per_token.restype = sz
    lib.lrkv_cache_elems_per_token.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.lrkv_decode_workspace_size.restype = ctypes.c_int
    lib.lrkv_decode_workspace_size.argtypes = [dims_p, ctypes.POINTER(sz)]
    lib.lrkv_decode.restype = ctypes.c_int
    lib.lrkv_decode.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.lrkv_decode_profiled.restype = ctypes.c_int
    lib.lrkv_decode_profiled.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp,
                                         vp, vp]
    lib.lrkv_decode_static_scratch.restype = ctypes.c_int
    lib.lrkv_decode_static_scratch.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp]
    lib.lrkv_append.restype = ctypes.c_int
    lib.lrkv_append.argtypes = [dims_p, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, i32p, vp, vp, vp,
                                vp, vp, sz, vp]
    lib.lrkv_key_scales.restype = ctypes.c_int
    lib.lrkv_key_scales.argtypes = [dims_p, ctypes.c_float, ctypes.c_int, vp, vp, vp, i32p, vp, vp]
    lib.lrkv_decode_normed.restype = ctypes.c_int
    lib.lrkv_decode_normed.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.lrkv_decode_step.restype = ctypes.c_int
    lib.lrkv_decode_step.argtypes = [dims_p, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     i32p, vp, vp, vp, sz, vp]
    lib.lrkv_prefill_workspace_size.restype = ctypes.c_int
    lib.lrkv_prefill_workspace_size.argtypes = [dims_p, ctypes.c_int, ctypes.POINTER(sz)]
    lib.lrkv_prefill.restype = ctypes.c_int
    lib.lrkv_prefill.argtypes = [dims_p, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz,
                                 vp]
    lib.lrkv_prefill_normed.restype = ctypes.c_int
    lib.lrkv_prefill_normed.argtypes = [dims_p, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, i32p, vp, vp,
                                        vp, sz, vp]
    lib.lrkv_decode_paged.restype = ctypes.c_int
    lib.lrkv_decode_paged.argtypes = [dims_p, ctypes.c_int, ctypes.c_int, i32p, vp, vp, vp, vp, vp, vp, vp, i32p,
                                      vp, vp, vp, sz, vp]
    lib.lrkv_append_paged.restype = ctypes.c_int
    lib.lrkv_append_paged.argtypes = [dims_p, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, i32p, ctypes.c_int,
                                      ctypes.c_int, i32p, vp, vp, vp, vp, vp, sz, vp]
    lib.lrkv_decode_step_paged.restype = ctypes.c_int
    lib.lrkv_decode_step_paged.argtypes = [dims_p, ctypes.c_int, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                           ctypes.c_int, i32p, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.lrkv_prefill_paged.restype = ctypes.c_int
    lib.lrkv_prefill_paged.argtypes = [dims_p, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, i32p, vp, vp, vp, vp,
                                       vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.lrkv_rope_table.restype = ctypes.c_int
    lib.lrkv_rope_table.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_float, vp, vp]
    lib.lrkv_decode_rope_workspace_size.restype = ctypes.c_int
    lib.lrkv_decode_rope_workspace_size.argtypes = [dims_p, ctypes.POINTER(sz)]
    lib.lrkv_decode_rope.restype = ctypes.c_int
    lib.lrkv_decode_rope.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, i32p, vp, vp, vp, sz,
                                     vp]
    ddp, mdp = ctypes.POINTER(lrkv_dense_dims), ctypes.POINTER(lrkv_mla_dims)
    lib.lrkv_dense_decode_workspace_size.restype = ctypes.c_int
    lib.lrkv_dense_decode_workspace_size.argtypes = [ddp, ctypes.POINTER(sz)]
    lib.lrkv_dense_decode.restype = ctypes.c_int
    lib.lrkv_dense_decode.argtypes = [ddp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.lrkv_mla_decode_workspace_size.restype = ctypes.c_int
    lib.lrkv_mla_decode_workspace_size.argtypes = [mdp, ctypes.POINTER(sz)]
    lib.lrkv_mla_decode.restype = ctypes.c_int
    lib.lrkv_mla_decode.argtypes = [mdp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.lrkv_read_device_status.restype = ctypes.c_int
    lib.lrkv_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.lrkv_read_static_scratch_status.restype = ctypes.c_int
    lib.lrkv_read_static_scratch_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().lrkv_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_dims(batch: int, heads: int, head_dim: int, rank: int, max_len: int, dtype,
              scale: float = 0.0) -> lrkv_dims:
    if dtype in (torch.bfloat16, "bf16", LRKV_BF16):
        dt = LRKV_BF16
    elif dtype in (torch.float32, "f32", LRKV_F32):
        dt = LRKV_F32
    else:
        dt = int(dtype) if isinstance(dtype, int) else -1
    return lrkv_dims(batch, heads, head_dim, rank, max_len, dt, float(scale))


# ------------------------------------------------------- raw ABI wrappers --

def lrkv_cache_elems_per_token(heads: int, head_dim: int, rank: int) -> int:
    return int(load().lrkv_cache_elems_per_token(heads, head_dim, rank))


def lrkv_decode_workspace_size(dims: lrkv_dims) -> int:
    n = ctypes.c_size_t(0)
    st = load().lrkv_decode_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_workspace_size")
    return int(n.value)


def lrkv_decode(dims: lrkv_dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws,
                ws_bytes: int, stream=None) -> int:
    """Direct call of the C entry point; returns its status code."""
    return int(load().lrkv_decode(ctypes.byref(dims), _ptr(q), _ptr(k_s), _ptr(v_s), _ptr(z_k),
                                  _ptr(z_v), _ptr(b_k), _ptr(b_v), _ptr(seq_lens), _ptr(out),
                                  _ptr(lse), _ptr(ws), ws_bytes, _stream_handle(stream)))


def lrkv_decode_profiled(dims: lrkv_dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws,
                         ws_bytes: int, ev_begin: "torch.cuda.Event", ev_end: "torch.cuda.Event",
                         stream=None) -> int:
    """lrkv_decode with CUDA events recorded around the split-KV kernel."""
    for ev in (ev_begin, ev_end):
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record(torch.cuda.current_stream() if stream is None else stream)
    return int(load().lrkv_decode_profiled(
        ctypes.byref(dims), _ptr(q), _ptr(k_s), _ptr(v_s), _ptr(z_k), _ptr(z_v), _ptr(b_k),
        _ptr(b_v), _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
        _stream_handle(stream), ev_begin.cuda_event, ev_end.cuda_event))


def lrkv_decode_static_scratch(dims: lrkv_dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out,
                               lse, stream=None) -> int:
    """lrkv_decode with the workspace taken from the array built into the
    library (for callers that cannot allocate device memory); returns the
    status code."""
    return int(load().lrkv_decode_static_scratch(
        ctypes.byref(dims), _ptr(q), _ptr(k_s), _ptr(v_s), _ptr(z_k), _ptr(z_v), _ptr(b_k),
        _ptr(b_v), _ptr(seq_lens), _ptr(out), _ptr(lse), _stream_handle(stream)))


def lrkv_read_static_scratch_status(stream=None) -> int:
    """Status of the last lrkv_decode_static_scratch call on the current device."""
    out = ctypes.c_int(0)
    st = load().lrkv_read_static_scratch_status(_stream_handle(stream), ctypes.byref(out))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_read_static_scratch_status")
    return int(out.value)


def lrkv_read_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int(0)
    st = load().lrkv_read_device_status(_ptr(ws), _stream_handle(stream), ctypes.byref(out))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_read_device_status")
    return int(out.value)


# ------------------------------------------------------- tensor front end --

def decode_workspace(dims: lrkv_dims, device) -> torch.Tensor:
    n = lrkv_decode_workspace_size(dims)
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode(q: torch.Tensor, k_s: torch.Tensor, v_s: torch.Tensor, z_k: torch.Tensor,
           z_v: torch.Tensor, b_k: torch.Tensor, b_v: torch.Tensor, seq_lens: torch.Tensor,
           scale: float = 0.0, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
           stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One decode step on device tensors in the layouts of include/lrkv.h.
    Allocates out/lse/workspace with torch when not given."""
    B, H, dh = q.shape
    max_len = k_s.shape[1]
    r = z_k.shape[-1] if z_k is not None else 0
    dims = make_dims(B, H, dh, r, max_len, q.dtype, scale)
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(dims, q.device)
    for t in (q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens):
        if t is not None and not t.is_contiguous():
            raise ValueError("LRKV tensors must be contiguous")
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    st = lrkv_decode(dims, q, k_s, v_s, z_k if r > 0 else None, z_v if r > 0 else None,
                     b_k if r > 0 else None, b_v if r > 0 else None, seq_lens, out, lse, ws,
                     ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode")
    return out, lse


def lrkv_append(dims: lrkv_dims, d_model: int, n_new: int, x, w_sk, w_sv, u_k, u_v, start_pos,
                k_s, v_s, z_k, z_v, ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the append entry point; returns its status code."""
    return int(load().lrkv_append(ctypes.byref(dims), d_model, n_new, _ptr(x), _ptr(w_sk),
                                  _ptr(w_sv), _ptr(u_k), _ptr(u_v), _ptr(start_pos), _ptr(k_s),
                                  _ptr(v_s), _ptr(z_k), _ptr(z_v), _ptr(ws), ws_bytes,
                                  _stream_handle(stream)))


def append(x: torch.Tensor, w_sk: torch.Tensor, w_sv: torch.Tensor, u_k: torch.Tensor,
           u_v: torch.Tensor, start_pos: torch.Tensor, k_s: torch.Tensor, v_s: torch.Tensor,
           z_k: torch.Tensor, z_v: torch.Tensor, stream=None) -> int:
    """Append x [B, n_new, d] to the cache in place (weights output-major:
    w_sk [d_h, d], u_k [H*r, d]).  Returns the device status word after a
    synchronising read."""
    B, n_new, d = x.shape
    H, r = z_k.shape[2], z_k.shape[3]
    dims = make_dims(B, H, k_s.shape[2], r, k_s.shape[1], x.dtype)
    ws = torch.zeros(16, dtype=torch.uint8, device=x.device)
    st = lrkv_append(dims, d, n_new, x, w_sk, w_sv, u_k, u_v, start_pos, k_s, v_s, z_k, z_v, ws,
                     ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_append")
    return lrkv_read_device_status(ws, stream)


def key_scales(k_s: torch.Tensor, z_k: torch.Tensor, b_k: torch.Tensor, start_pos: torch.Tensor,
               n_new: int, key_scale: torch.Tensor, eps: float = 1e-6, stream=None) -> None:
    """Reciprocal key RMS (post-projection RMSNorm) of the rows
    [start_pos[b], start_pos[b] + n_new) into key_scale [B, H, max_len] (fp32)."""
    B, L, dh = k_s.shape
    H, r = z_k.shape[2], z_k.shape[3]
    dims = make_dims(B, H, dh, r, L, k_s.dtype)
    st = int(load().lrkv_key_scales(ctypes.byref(dims), float(eps), int(n_new), _ptr(k_s), _ptr(z_k), _ptr(b_k),
                                    _ptr(start_pos), _ptr(key_scale), _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_key_scales")


def lrkv_decode_normed(dims: lrkv_dims, q, k_s, v_s, z_k, z_v, b_k, b_v, key_scale, seq_lens, out, lse,
                       ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the normalised-key decode entry point; returns its status."""
    return int(load().lrkv_decode_normed(ctypes.byref(dims), _ptr(q), _ptr(k_s), _ptr(v_s), _ptr(z_k),
                                         _ptr(z_v), _ptr(b_k), _ptr(b_v), _ptr(key_scale), _ptr(seq_lens),
                                         _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream_handle(stream)))


def decode_normed(q, k_s, v_s, z_k, z_v, b_k, b_v, key_scale, seq_lens, scale: float = 0.0, out=None,
                  lse=None, ws=None, stream=None):
    """decode with the keys' post-projection RMSNorm scales applied to the scores."""
    B, H, dh = q.shape
    dims = make_dims(B, H, dh, z_k.shape[-1], k_s.shape[1], q.dtype, scale)
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(dims, q.device)
    st = lrkv_decode_normed(dims, q, k_s, v_s, z_k, z_v, b_k, b_v, key_scale, seq_lens, out, lse, ws,
                            ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_normed")
    return out, lse


def lrkv_decode_step(dims: lrkv_dims, d_model: int, x, w_sk, w_sv, u_k, u_v, q, k_s, v_s, z_k, z_v,
                     b_k, b_v, seq_lens, out, lse, ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the decode-step entry point; returns its status code."""
    return int(load().lrkv_decode_step(ctypes.byref(dims), d_model, _ptr(x), _ptr(w_sk), _ptr(w_sv),
                                       _ptr(u_k), _ptr(u_v), _ptr(q), _ptr(k_s), _ptr(v_s), _ptr(z_k),
                                       _ptr(z_v), _ptr(b_k), _ptr(b_v), _ptr(seq_lens), _ptr(out),
                                       _ptr(lse), _ptr(ws), ws_bytes, _stream_handle(stream)))


def decode_step(x: torch.Tensor, w_sk: torch.Tensor, w_sv: torch.Tensor, u_k: torch.Tensor,
                u_v: torch.Tensor, q: torch.Tensor, k_s: torch.Tensor, v_s: torch.Tensor,
                z_k: torch.Tensor, z_v: torch.Tensor, b_k: torch.Tensor, b_v: torch.Tensor,
                seq_lens: torch.Tensor, scale: float = 0.0, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One decode step: writes the token's rows (from x [B, d]) at
    seq_lens[b] - 1, then decodes.  Allocates out/lse/workspace when not given."""
    B, H, dh = q.shape
    d = x.shape[-1]
    dims = make_dims(B, H, dh, z_k.shape[-1], k_s.shape[1], q.dtype, scale)
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(dims, q.device)
    for t in (x, w_sk, w_sv, u_k, u_v, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens):
        if not t.is_contiguous():
            raise ValueError("LRKV tensors must be contiguous")
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    st = lrkv_decode_step(dims, d, x, w_sk, w_sv, u_k, u_v, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens,
                          out, lse, ws, ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_step")
    return out, lse


def lrkv_prefill_workspace_size(dims: lrkv_dims, q_len: int) -> int:
    n = ctypes.c_size_t(0)
    st = load().lrkv_prefill_workspace_size(ctypes.byref(dims), int(q_len), ctypes.byref(n))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_prefill_workspace_size")
    return int(n.value)


def lrkv_prefill(dims: lrkv_dims, q_len: int, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse,
                 ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the prefill entry point; returns its status code."""
    return int(load().lrkv_prefill(ctypes.byref(dims), q_len, _ptr(q), _ptr(k_s), _ptr(v_s),
                                   _ptr(z_k), _ptr(z_v), _ptr(b_k), _ptr(b_v), _ptr(seq_lens),
                                   _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream_handle(stream)))


def lrkv_prefill_normed(dims: lrkv_dims, q_len: int, q, k_s, v_s, z_k, z_v, b_k, b_v, key_scale, seq_lens,
                        out, lse, ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the normalised-key prefill entry point; returns its status."""
    return int(load().lrkv_prefill_normed(ctypes.byref(dims), q_len, _ptr(q), _ptr(k_s), _ptr(v_s),
                                          _ptr(z_k), _ptr(z_v), _ptr(b_k), _ptr(b_v), _ptr(key_scale),
                                          _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                          _stream_handle(stream)))


def prefill(q: torch.Tensor, k_s: torch.Tensor, v_s: torch.Tensor, z_k: torch.Tensor,
            z_v: torch.Tensor, b_k: torch.Tensor, b_v: torch.Tensor, seq_lens: torch.Tensor,
            scale: float = 0.0, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """Causal prefill of q [B, q_len, H, d_h]; returns (out, lse, status)."""
    B, Tq, H, dh = q.shape
    r = z_k.shape[-1]
    dims = make_dims(B, H, dh, r, k_s.shape[1], q.dtype, scale)
    if out is None:
        out = torch.empty((B, Tq, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.zeros(lrkv_prefill_workspace_size(dims, Tq), dtype=torch.uint8, device=q.device)
    st = lrkv_prefill(dims, Tq, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws, ws.numel(),
                      stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_prefill")
    return out, lse, ws


def prefill_normed(q: torch.Tensor, k_s: torch.Tensor, v_s: torch.Tensor, z_k: torch.Tensor,
                   z_v: torch.Tensor, b_k: torch.Tensor, b_v: torch.Tensor, key_scale: torch.Tensor,
                   seq_lens: torch.Tensor, scale: float = 0.0, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """prefill with the keys' post-projection RMSNorm scales (key_scale
    [B, H, max_len] fp32) applied to the scores; returns (out, lse, status)."""
    B, Tq, H, dh = q.shape
    r = z_k.shape[-1]
    dims = make_dims(B, H, dh, r, k_s.shape[1], q.dtype, scale)
    if out is None:
        out = torch.empty((B, Tq, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.zeros(lrkv_prefill_workspace_size(dims, Tq), dtype=torch.uint8, device=q.device)
    st = lrkv_prefill_normed(dims, Tq, q, k_s, v_s, z_k, z_v, b_k, b_v, key_scale, seq_lens, out, lse, ws,
                             ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_prefill_normed")
    return out, lse, ws


def lrkv_decode_paged(dims: lrkv_dims, page_size: int, num_pages: int, block_table, q, k_s, v_s, z_k, z_v, b_k,
                      b_v, seq_lens, out, lse, ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the paged-cache decode entry point; returns its status."""
    return int(load().lrkv_decode_paged(ctypes.byref(dims), page_size, num_pages, _ptr(block_table), _ptr(q),
                                        _ptr(k_s), _ptr(v_s), _ptr(z_k), _ptr(z_v), _ptr(b_k), _ptr(b_v),
                                        _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                        _stream_handle(stream)))


def decode_paged(q, k_s, v_s, z_k, z_v, b_k, b_v, block_table, seq_lens, scale: float = 0.0, out=None, lse=None,
                 ws=None, stream=None):
    """decode over a paged cache: pools k_s, v_s [P, page_size, d_h] and
    z_k, z_v [P, page_size, H, r]; block_table [B, max_len / page_size] int32."""
    B, H, dh = q.shape
    num_pages, page_size = k_s.shape[0], k_s.shape[1]
    r = z_k.shape[-1]
    dims = make_dims(B, H, dh, r, block_table.shape[1] * page_size, q.dtype, scale)
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(dims, q.device)
    st = lrkv_decode_paged(dims, page_size, num_pages, block_table, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens,
                           out, lse, ws, ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_paged")
    return out, lse, ws


def append_paged(x, w_sk, w_sv, u_k, u_v, start_pos, block_table, k_s, v_s, z_k, z_v, heads: int, ws=None,
                 stream=None):
    """The factored rows of x [B, n_new, d_model] into a paged cache (pools
    k_s, v_s [P, page_size, d_h], z_k, z_v [P, page_size, H, r]) at logical
    rows start_pos[b] + t; returns the status workspace."""
    B, n_new, d = x.shape
    num_pages, page_size, dh = k_s.shape
    r = z_k.shape[-1]
    dims = make_dims(B, heads, dh, r, block_table.shape[1] * page_size, x.dtype)
    if ws is None:
        ws = torch.zeros(16, dtype=torch.uint8, device=x.device)
    st = int(load().lrkv_append_paged(ctypes.byref(dims), d, n_new, _ptr(x), _ptr(w_sk), _ptr(w_sv), _ptr(u_k),
                                      _ptr(u_v), _ptr(start_pos), page_size, num_pages, _ptr(block_table),
                                      _ptr(k_s), _ptr(v_s), _ptr(z_k), _ptr(z_v), _ptr(ws), ws.numel(),
                                      _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_append_paged")
    return ws


def decode_step_paged(x, w_sk, w_sv, u_k, u_v, q, k_s, v_s, z_k, z_v, b_k, b_v, block_table, seq_lens,
                      scale: float = 0.0, out=None, lse=None, ws=None, stream=None):
    """decode_step over a paged cache; returns (out, lse, ws)."""
    B, H, dh = q.shape
    num_pages, page_size = k_s.shape[0], k_s.shape[1]
    r = z_k.shape[-1]
    dims = make_dims(B, H, dh, r, block_table.shape[1] * page_size, q.dtype, scale)
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(dims, q.device)
    st = int(load().lrkv_decode_step_paged(ctypes.byref(dims), x.shape[-1], _ptr(x), _ptr(w_sk), _ptr(w_sv),
                                           _ptr(u_k), _ptr(u_v), _ptr(q), page_size, num_pages,
                                           _ptr(block_table), _ptr(k_s), _ptr(v_s), _ptr(z_k), _ptr(z_v),
                                           _ptr(b_k), _ptr(b_v), _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(ws),
                                           ws.numel(), _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_step_paged")
    return out, lse, ws


def prefill_paged(q, k_s, v_s, z_k, z_v, b_k, b_v, block_table, seq_lens, scale: float = 0.0, out=None, lse=None,
                  ws=None, stream=None):
    """Causal prefill of q [B, q_len, H, d_h] over a paged cache (pools k_s,
    v_s [P, page_size, d_h], z_k, z_v [P, page_size, H, r]); returns
    (out, lse, status workspace)."""
    B, Tq, H, dh = q.shape
    num_pages, page_size = k_s.shape[0], k_s.shape[1]
    r = z_k.shape[-1]
    dims = make_dims(B, H, dh, r, block_table.shape[1] * page_size, q.dtype, scale)
    if out is None:
        out = torch.empty((B, Tq, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.zeros(lrkv_prefill_workspace_size(dims, Tq), dtype=torch.uint8, device=q.device)
    st = int(load().lrkv_prefill_paged(ctypes.byref(dims), Tq, _ptr(q), page_size, num_pages, _ptr(block_table),
                                       _ptr(k_s), _ptr(v_s), _ptr(z_k), _ptr(z_v), _ptr(b_k), _ptr(b_v),
                                       _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                       _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_prefill_paged")
    return out, lse, ws


# ------------------------------------------------------------ full RoPE --

def rope_table(max_pos: int, head_dim: int, base: float = 10000.0, device="cuda", stream=None) -> torch.Tensor:
    """The rotation table [max_pos, head_dim] fp32 (cos, sin pairs) computed
    by the library."""
    t = torch.empty((max_pos, head_dim), dtype=torch.float32, device=device)
    st = int(load().lrkv_rope_table(int(max_pos), int(head_dim), float(base), _ptr(t), _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_rope_table")
    return t


def lrkv_decode_rope_workspace_size(dims: lrkv_dims) -> int:
    n = ctypes.c_size_t(0)
    st = load().lrkv_decode_rope_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_rope_workspace_size")
    return int(n.value)


def lrkv_decode_rope(dims: lrkv_dims, q_rot, k_s, v_s, z_k, z_v, b_k, b_v, cos_sin, max_pos: int, seq_lens, out,
                     lse, ws, ws_bytes: int, stream=None) -> int:
    """Direct call of the full-RoPE decode entry point; returns its status."""
    return int(load().lrkv_decode_rope(ctypes.byref(dims), _ptr(q_rot), _ptr(k_s), _ptr(v_s), _ptr(z_k),
                                       _ptr(z_v), _ptr(b_k), _ptr(b_v), _ptr(cos_sin), int(max_pos),
                                       _ptr(seq_lens), _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                       _stream_handle(stream)))


def decode_rope(q_rot, k_s, v_s, z_k, z_v, b_k, b_v, cos_sin, seq_lens, scale: float = 0.0, out=None, lse=None,
                ws=None, stream=None):
    """Decode with full RoPE of the keys: q_rot [B, H, d_h] is the query
    rotated to its position, the cache holds unrotated rows, cos_sin is a
    table from rope_table().  Returns (out, lse)."""
    B, H, dh = q_rot.shape
    dims = make_dims(B, H, dh, z_k.shape[-1], k_s.shape[1], q_rot.dtype, scale)
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q_rot.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q_rot.device)
    if ws is None:
        ws = torch.empty(lrkv_decode_rope_workspace_size(dims), dtype=torch.uint8, device=q_rot.device)
    for t in (q_rot, k_s, v_s, z_k, z_v, b_k, b_v, cos_sin, seq_lens):
        if not t.is_contiguous():
            raise ValueError("LRKV tensors must be contiguous")
    st = lrkv_decode_rope(dims, q_rot, k_s, v_s, z_k, z_v, b_k, b_v, cos_sin, cos_sin.shape[0], seq_lens, out, lse,
                          ws, ws.numel(), stream)
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_decode_rope")
    return out, lse


# ------------------------------------------------- comparison decodes --

def dense_decode(q, k, v, seq_lens, scale: float = 0.0, out=None, lse=None, ws=None, stream=None):
    """Decode over materialised K/V (MHA, GQA, MQA): q [B, H, d], k, v
    [B, L, H_kv, d] bf16.  Returns (out, lse, ws)."""
    B, H, d = q.shape
    dims = lrkv_dense_dims(B, H, k.shape[2], d, k.shape[1], float(scale))
    if out is None:
        out = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        n = ctypes.c_size_t(0)
        st = load().lrkv_dense_decode_workspace_size(ctypes.byref(dims), ctypes.byref(n))
        if st != LRKV_OK:
            raise LRKVError(st, "lrkv_dense_decode_workspace_size")
        ws = torch.empty(int(n.value), dtype=torch.uint8, device=q.device)
    st = int(load().lrkv_dense_decode(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(out),
                                      _ptr(lse), _ptr(ws), ws.numel(), _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_dense_decode")
    return out, lse, ws


def mla_decode(q, c, w_uk, w_uv, seq_lens, scale: float = 0.0, out=None, lse=None, ws=None, stream=None):
    """Absorbed MLA decode: q [B, H, d_h], c [B, L, d_c], w_uk, w_uv
    [H, d_h, d_c] bf16.  Returns (out, lse, ws)."""
    B, H, dh = q.shape
    dims = lrkv_mla_dims(B, H, dh, c.shape[2], c.shape[1], float(scale))
    if out is None:
        out = torch.empty((B, H, dh), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        n = ctypes.c_size_t(0)
        st = load().lrkv_mla_decode_workspace_size(ctypes.byref(dims), ctypes.byref(n))
        if st != LRKV_OK:
            raise LRKVError(st, "lrkv_mla_decode_workspace_size")
        ws = torch.empty(int(n.value), dtype=torch.uint8, device=q.device)
    st = int(load().lrkv_mla_decode(ctypes.byref(dims), _ptr(q), _ptr(c), _ptr(w_uk), _ptr(w_uv), _ptr(seq_lens),
                                    _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream_handle(stream)))
    if st != LRKV_OK:
        raise LRKVError(st, "lrkv_mla_decode")
    return out, lse, ws
