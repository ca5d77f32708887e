"""B300-native MLA decode over a latent KV cache with matrix absorption.

Thin Python binding of ``libmla.so`` (C ABI declared in ``include/mla.h``).  Every
step of the path runs in the library's CUDA kernels; this module only marshals
torch tensors (device memory and the current CUDA stream) into pointers and
sizes.  There is no fallback: if the library is missing or a call fails, an
exception is raised.

Pipeline of one decode step (absorbed MLA, "MLA multi-head latent attention:
low-rank compression and matrix absorption", sections 3.1-3.2 and 5.1-5.2):

    cache_append(cache, c_kv, k_r, seq_idx, pos)   # cache row = [c_KV || RoPE(k_R)]
    q_cat = absorb_q(q_nope, q_rope, q_pos, w_uk)  # [q_nope W_UK || RoPE(q_R)]
    o_lat, lse = decode_attn(q_cat, cache, seq_lens, scale, ws)
    o = out_up(o_lat, w_uv)                        # W_UV applied after attention
    gate(h, w_g, o.view(B, -1))                    # gated variant only
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MlaError", "LatentCache", "lib", "cache_append", "absorb_q", "decode_workspace",
    "decode_attn", "decode_attn_noalloc", "out_up", "gate", "get_device_error", "debug_inject_fault", "LIB_PATH",
    "PagedLatentCache", "cache_append_paged", "decode_attn_paged", "PAGE_ROWS",
    "kv_down_workspace", "kv_down_append", "absorb_q_append", "prefill_explicit_workspace", "prefill_explicit",
    "decode_attn_partial", "decode_merge",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_BF16, MLA_F32 = 0, 1
_DT = {torch.bfloat16: MLA_BF16, torch.float32: MLA_F32}


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib_handle.mla_status_string(status).decode() if _lib_handle is not None else str(status)
        super().__init__(f"{where}: {msg}")
        self.status = status


class _Cache(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("B", ctypes.c_int32),
        ("N_max", ctypes.c_int32), ("d_c", ctypes.c_int32), ("d_r", ctypes.c_int32),
        ("_pad", ctypes.c_int32), ("row_stride", ctypes.c_int64),
    ]


class _PagedCache(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("d_c", ctypes.c_int32), ("d_r", ctypes.c_int32), ("row_stride", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("B", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
    ]


PAGE_ROWS = 64

_lib_handle = None

_SIGS = {
    "mla_abi_version": (ctypes.c_int32, []),
    "mla_build_source_hash": (ctypes.c_char_p, []),
    "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mla_cache_append": (ctypes.c_int, [ctypes.POINTER(_Cache), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p]),
    "mla_absorb_q": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p]),
    "mla_absorb_q_append": (ctypes.c_int, [ctypes.POINTER(_Cache), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p]),
    "mla_absorb_q_append_paged": (ctypes.c_int, [ctypes.POINTER(_PagedCache), ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                 ctypes.c_void_p]),
    "mla_decode_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "mla_decode_attn": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(_Cache), ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "mla_prefill_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_int32]),
    "mla_prefill_attn": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(_Cache), ctypes.c_void_p, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_float, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "mla_out_up": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]),
    "mla_gate": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]),
    "mla_get_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "mla_debug_inject_fault": (ctypes.c_int, [ctypes.c_int32]),
    "mla_cache_append_paged": (ctypes.c_int, [ctypes.POINTER(_PagedCache), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                              ctypes.c_void_p]),
    "mla_decode_attn_paged": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(_PagedCache), ctypes.c_void_p,
                                             ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "mla_kv_down_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_int32, ctypes.c_int32]),
    "mla_kv_down_append": (ctypes.c_int, [ctypes.POINTER(_Cache), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                          ctypes.c_void_p]),
    "mla_kv_down_append_paged": (ctypes.c_int, [ctypes.POINTER(_PagedCache), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
                                                ctypes.c_size_t, ctypes.c_void_p]),
    "mla_prefill_explicit_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                              ctypes.c_int32]),
    "mla_prefill_explicit": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Cache),
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p]),
    "mla_decode_attn_partial": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(_Cache), ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
                                               ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "mla_decode_merge": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p]),
    "mla_decode_attn_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(_Cache), ctypes.c_void_p,
                                               ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p]),
}


def lib() -> ctypes.CDLL:
    """Load libmla.so from the package directory (raises if it was not built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmla.so not built at {LIB_PATH}; run `python -m head_latent_attention_29_b300._build`")
        h = ctypes.CDLL(LIB_PATH)
        if os.path.isdir(os.path.join(_PKG, "csrc")):
            from . import _build
            h.mla_build_source_hash.restype = ctypes.c_char_p
            have, want = h.mla_build_source_hash().decode(), _build.source_hash()
            if have != want:
                raise ImportError(f"{LIB_PATH} was built from other sources (hash {have}, sources {want}); "
                                  "rebuild it: `python -m head_latent_attention_29_b300._build`")
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MlaError(status, where)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dev_tensor(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _out_tensor(t: torch.Tensor, name: str, shape: tuple, dtype) -> torch.Tensor:
    """A caller-supplied output: a contiguous CUDA tensor of exactly this shape and
    dtype (the kernels write every element through maps built from the shape)."""
    _dev_tensor(t, name, dtype)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


class LatentCache:
    """One layer's latent cache [B, N_max, row_stride] on the device.

    Row t of sequence b holds [c_KV (d_c) || RoPE(k_R) (d_r)] (icman.com.cn MLA
    article, section 2).  ``row_stride`` defaults to d_c + d_r rounded up to 16
    bytes.  The tensor is allocated by torch and owned by this object."""

    def __init__(self, B: int, N_max: int, d_c: int, d_r: int, dtype=torch.bfloat16, device="cuda",
                 row_stride: int | None = None, data: torch.Tensor | None = None):
        esz = 2 if dtype == torch.bfloat16 else 4
        R = d_c + d_r
        if row_stride is None:
            row_stride = ((R * esz + 15) // 16) * 16 // esz
        self.B, self.N_max, self.d_c, self.d_r, self.row_stride = B, N_max, d_c, d_r, row_stride
        self.dtype = dtype
        if data is None:
            data = torch.zeros((B, N_max, row_stride), dtype=dtype, device=device)
        elif tuple(data.shape) != (B, N_max, row_stride) or data.dtype != dtype:
            raise ValueError("cache tensor shape/dtype mismatch")
        self.data = data

    @property
    def rows(self) -> torch.Tensor:
        """View [B, N_max, d_c + d_r] of the cached rows (padding excluded)."""
        return self.data[..., : self.d_c + self.d_r]

    def struct(self) -> _Cache:
        return _Cache(self.data.data_ptr(), _DT[self.dtype], self.B, self.N_max, self.d_c, self.d_r, 0,
                      self.row_stride)


def cache_append(cache: LatentCache, c_kv: torch.Tensor, k_r: torch.Tensor | None, seq_idx: torch.Tensor,
                 pos: torch.Tensor, rope_base: float = 10000.0) -> None:
    """Write T rows: cache[seq_idx[i], pos[i]] = [c_kv[i] || RoPE(k_r[i], pos[i])]."""
    _dev_tensor(c_kv, "c_kv", cache.dtype)
    if cache.d_r > 0:
        _dev_tensor(k_r, "k_r", cache.dtype)
    _dev_tensor(seq_idx, "seq_idx", torch.int32)
    _dev_tensor(pos, "pos", torch.int32)
    T = seq_idx.numel()
    st = cache.struct()
    _check(lib().mla_cache_append(ctypes.byref(st), _ptr(c_kv), _ptr(k_r if cache.d_r > 0 else None), _ptr(seq_idx),
                                  _ptr(pos), T, float(rope_base), _stream(c_kv)), "mla_cache_append")


def absorb_q(q_nope: torch.Tensor, q_rope: torch.Tensor | None, q_pos: torch.Tensor, w_uk: torch.Tensor,
             rope_base: float = 10000.0, out: torch.Tensor | None = None) -> torch.Tensor:
    """q_cat [B, H, d_c + d_r] = [q_nope W_UK || RoPE(q_rope, q_pos)] per head."""
    _dev_tensor(q_nope, "q_nope")
    B, H, d_k = q_nope.shape
    _dev_tensor(w_uk, "w_uk", q_nope.dtype)
    d_c = w_uk.shape[2]
    d_r = 0 if q_rope is None else q_rope.shape[2]
    if q_rope is not None:
        _dev_tensor(q_rope, "q_rope", q_nope.dtype)
    _dev_tensor(q_pos, "q_pos", torch.int32)
    if out is None:
        out = torch.empty((B, H, d_c + d_r), dtype=q_nope.dtype, device=q_nope.device)
    _check(lib().mla_absorb_q(_ptr(q_nope), _ptr(q_rope), _ptr(q_pos), _ptr(w_uk), _ptr(out), B, H, d_k, d_c, d_r,
                              _DT[q_nope.dtype], float(rope_base), _stream(q_nope)), "mla_absorb_q")
    return out


def absorb_q_append(cache, c_kv: torch.Tensor, k_r: torch.Tensor | None, seq_idx: torch.Tensor, pos: torch.Tensor,
                    q_nope: torch.Tensor, q_rope: torch.Tensor | None, q_pos: torch.Tensor, w_uk: torch.Tensor,
                    rope_base: float = 10000.0, out: torch.Tensor | None = None) -> torch.Tensor:
    """cache_append(cache, c_kv, k_r, seq_idx, pos) and absorb_q(q_nope, q_rope, q_pos,
    w_uk) in one call (one launch for bf16); returns q_cat [B, H, d_c + d_r].  The
    cache is a LatentCache or a PagedLatentCache."""
    _dev_tensor(q_nope, "q_nope", cache.dtype)
    B, H, d_k = q_nope.shape
    _dev_tensor(w_uk, "w_uk", cache.dtype)
    if tuple(w_uk.shape) != (H, d_k, cache.d_c):
        raise ValueError("w_uk must be [H, d_k, d_c]")
    if cache.d_r > 0:
        _dev_tensor(q_rope, "q_rope", cache.dtype)
        _dev_tensor(k_r, "k_r", cache.dtype)
    _dev_tensor(q_pos, "q_pos", torch.int32)
    _dev_tensor(c_kv, "c_kv", cache.dtype)
    _dev_tensor(seq_idx, "seq_idx", torch.int32)
    _dev_tensor(pos, "pos", torch.int32)
    T = seq_idx.numel()
    if pos.numel() != T or c_kv.numel() != T * cache.d_c:
        raise ValueError("c_kv, seq_idx and pos need one row / entry per appended token")
    R = cache.d_c + cache.d_r
    if out is None:
        out = torch.empty((B, H, R), dtype=cache.dtype, device=q_nope.device)
    _out_tensor(out, "out", (B, H, R), cache.dtype)
    st = cache.struct()
    paged = isinstance(cache, PagedLatentCache)
    fn, name = ((lib().mla_absorb_q_append_paged, "mla_absorb_q_append_paged") if paged
                else (lib().mla_absorb_q_append, "mla_absorb_q_append"))
    kr, qr = (k_r, q_rope) if cache.d_r > 0 else (None, None)
    _check(fn(ctypes.byref(st), _ptr(c_kv), _ptr(kr), _ptr(seq_idx), _ptr(pos), T, _ptr(q_nope), _ptr(qr),
              _ptr(q_pos), _ptr(w_uk), _ptr(out), B, H, d_k, float(rope_base), _stream(q_nope)), name)
    return out


def decode_workspace(B: int, H: int, d_c: int, dtype=torch.bfloat16, device="cuda") -> torch.Tensor:
    n = lib().mla_decode_workspace_size(B, H, d_c, _DT[dtype])
    if n == 0:
        raise MlaError(2, "mla_decode_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode_attn(q_cat: torch.Tensor, cache: LatentCache, seq_lens: torch.Tensor, scale: float,
                workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None, want_lse: bool = True):
    """o_lat [B, H, d_c] (and lse [B, H] fp32) of absorbed decode attention."""
    _dev_tensor(q_cat, "q_cat", cache.dtype)
    B, H, R = q_cat.shape
    if B != cache.B or R != cache.d_c + cache.d_r:
        raise ValueError("q_cat shape does not match the cache")
    _dev_tensor(seq_lens, "seq_lens", torch.int32)
    if seq_lens.numel() != B:
        raise ValueError("seq_lens needs one entry per sequence")
    if workspace is None:
        workspace = decode_workspace(B, H, cache.d_c, cache.dtype, q_cat.device)
    if out is None:
        out = torch.empty((B, H, cache.d_c), dtype=cache.dtype, device=q_cat.device)
    _out_tensor(out, "out", (B, H, cache.d_c), cache.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q_cat.device)
    if lse is not None:
        _out_tensor(lse, "lse", (B, H), torch.float32)
    st = cache.struct()
    _check(lib().mla_decode_attn(_ptr(q_cat), ctypes.byref(st), _ptr(seq_lens), H, float(scale), _ptr(workspace),
                                 workspace.numel(), _ptr(out), _ptr(lse), _stream(q_cat)), "mla_decode_attn")
    return out, lse


def prefill_workspace(B: int, S: int, H: int, d_c: int, dtype=torch.bfloat16, device="cuda") -> torch.Tensor:
    n = lib().mla_prefill_workspace_size(B, S, H, d_c, _DT[dtype])
    if n == 0:
        raise MlaError(2, "mla_prefill_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def prefill_attn(q_cat: torch.Tensor, cache: LatentCache, q_start: torch.Tensor, scale: float, causal: bool = True,
                 workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, want_lse: bool = True):
    """o_lat [B, S, H, d_c] (and lse [B, S, H] fp32) of absorbed prompt attention;
    query i of sequence b sits at position q_start[b] + i."""
    _dev_tensor(q_cat, "q_cat", cache.dtype)
    B, S, H, R = q_cat.shape
    if B != cache.B or R != cache.d_c + cache.d_r:
        raise ValueError("q_cat shape does not match the cache")
    _dev_tensor(q_start, "q_start", torch.int32)
    if q_start.numel() != B:
        raise ValueError("q_start needs one entry per sequence")
    if workspace is None:
        workspace = prefill_workspace(B, S, H, cache.d_c, cache.dtype, q_cat.device)
    if out is None:
        out = torch.empty((B, S, H, cache.d_c), dtype=cache.dtype, device=q_cat.device)
    _out_tensor(out, "out", (B, S, H, cache.d_c), cache.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=q_cat.device)
    if lse is not None:
        _out_tensor(lse, "lse", (B, S, H), torch.float32)
    st = cache.struct()
    _check(lib().mla_prefill_attn(_ptr(q_cat), ctypes.byref(st), _ptr(q_start), S, H, float(scale), int(causal),
                                  _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse), _stream(q_cat)),
           "mla_prefill_attn")
    return out, lse


def decode_attn_partial(q_cat: torch.Tensor, cache: LatentCache, row_begin: torch.Tensor, row_end: torch.Tensor,
                        scale: float, workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                        lse: torch.Tensor | None = None):
    """Attention of each sequence's query over its rows [row_begin[b], row_end[b])
    only, as a partial for decode_merge: (o_part [B, H, d_c], lse_part [B, H] fp32)."""
    _dev_tensor(q_cat, "q_cat", cache.dtype)
    B, H, R = q_cat.shape
    if B != cache.B or R != cache.d_c + cache.d_r:
        raise ValueError("q_cat shape does not match the cache")
    _dev_tensor(row_begin, "row_begin", torch.int32)
    _dev_tensor(row_end, "row_end", torch.int32)
    if row_begin.numel() != B or row_end.numel() != B:
        raise ValueError("row_begin and row_end need one entry per sequence")
    if workspace is None:
        workspace = decode_workspace(B, H, cache.d_c, cache.dtype, q_cat.device)
    if out is None:
        out = torch.empty((B, H, cache.d_c), dtype=cache.dtype, device=q_cat.device)
    _out_tensor(out, "out", (B, H, cache.d_c), cache.dtype)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q_cat.device)
    _out_tensor(lse, "lse", (B, H), torch.float32)
    st = cache.struct()
    _check(lib().mla_decode_attn_partial(_ptr(q_cat), ctypes.byref(st), _ptr(row_begin), _ptr(row_end), H,
                                         float(scale), _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
                                         _stream(q_cat)), "mla_decode_attn_partial")
    return out, lse


def decode_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, want_lse: bool = True):
    """Merge k partials of disjoint row ranges, o_parts [k, B, H, d_c] and lse_parts
    [k, B, H] fp32, into (o_lat [B, H, d_c], lse [B, H])."""
    _dev_tensor(o_parts, "o_parts")
    if o_parts.dim() != 4:
        raise ValueError("o_parts must be [k, B, H, d_c]")
    k, B, H, d_c = o_parts.shape
    _out_tensor(lse_parts, "lse_parts", (k, B, H), torch.float32)
    if out is None:
        out = torch.empty((B, H, d_c), dtype=o_parts.dtype, device=o_parts.device)
    _out_tensor(out, "out", (B, H, d_c), o_parts.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=o_parts.device)
    if lse is not None:
        _out_tensor(lse, "lse", (B, H), torch.float32)
    _check(lib().mla_decode_merge(_ptr(o_parts), _ptr(lse_parts), k, B, H, d_c, _DT[o_parts.dtype], _ptr(out),
                                  _ptr(lse), _stream(o_parts)), "mla_decode_merge")
    return out, lse


def decode_attn_noalloc(q_cat: torch.Tensor, cache: LatentCache, seq_lens: torch.Tensor, scale: float,
                        out: torch.Tensor, lse: torch.Tensor | None = None):
    """Same result as decode_attn, for callers that cannot allocate device memory:
    the split-KV scratch is a buffer built into the library (at most 32 sequences).
    `out` (and `lse` if wanted) must be preallocated by the caller."""
    _dev_tensor(q_cat, "q_cat", cache.dtype)
    if q_cat.dim() != 3:
        raise ValueError("q_cat must be [B, H, d_c + d_r]")
    B, H, R = q_cat.shape
    if B != cache.B or R != cache.d_c + cache.d_r:
        raise ValueError("q_cat shape does not match the cache")
    _dev_tensor(seq_lens, "seq_lens", torch.int32)
    if seq_lens.numel() != B:
        raise ValueError("seq_lens needs one entry per sequence")
    _out_tensor(out, "out", (B, H, cache.d_c), cache.dtype)
    if lse is not None:
        _out_tensor(lse, "lse", (B, H), torch.float32)
    st = cache.struct()
    _check(lib().mla_decode_attn_noalloc(_ptr(q_cat), ctypes.byref(st), _ptr(seq_lens), H, float(scale), _ptr(out),
                                         _ptr(lse), _stream(q_cat)), "mla_decode_attn_noalloc")
    return out, lse


def out_up(o_lat: torch.Tensor, w_uv: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """o [B, H, d_v] = o_lat W_UV^T per head (W_UV stored [H, d_v, d_c])."""
    _dev_tensor(o_lat, "o_lat")
    _dev_tensor(w_uv, "w_uv", o_lat.dtype)
    B, H, d_c = o_lat.shape
    d_v = w_uv.shape[1]
    if out is None:
        out = torch.empty((B, H, d_v), dtype=o_lat.dtype, device=o_lat.device)
    _check(lib().mla_out_up(_ptr(o_lat), _ptr(w_uv), _ptr(out), B, H, d_c, d_v, _DT[o_lat.dtype], _stream(o_lat)),
           "mla_out_up")
    return out


def gate(h: torch.Tensor, w_g: torch.Tensor, o: torch.Tensor) -> torch.Tensor:
    """In place: o [B, width] *= sigmoid(h W_g)."""
    _dev_tensor(h, "h")
    _dev_tensor(w_g, "w_g", h.dtype)
    _dev_tensor(o, "o", h.dtype)
    B, d_model = h.shape
    width = w_g.shape[1]
    _check(lib().mla_gate(_ptr(h), _ptr(w_g), _ptr(o), B, d_model, width, _DT[h.dtype], _stream(h)), "mla_gate")
    return o


def get_device_error() -> tuple[int, int]:
    """(status, raw word) recorded by the kernels since the last call; synchronises the device."""
    word = ctypes.c_uint32(0)
    st = lib().mla_get_device_error(ctypes.byref(word))
    return st, word.value


def debug_inject_fault(kind: int) -> None:
    """Fault injection for tests of the bounded waits: kind 1 makes later bf16
    attention launches issue no loads in their score CTAs, so their waits run out
    (MLA_ERR_DEVICE_TIMEOUT in the device error word); kind 0 switches it off."""
    _check(lib().mla_debug_inject_fault(int(kind)), "mla_debug_inject_fault")


class PagedLatentCache:
    """A paged latent cache: a pool of ``num_pages`` pages of 64 rows
    [num_pages, 64, row_stride] and a block table [B, max_blocks] int32 naming the
    page of each 64-row block of each sequence (row t of sequence b is row t % 64 of
    page block_table[b, t // 64]).  Both tensors are allocated by torch and owned by
    this object unless passed in (``data``, ``block_table``); the caller fills the
    block table."""

    def __init__(self, num_pages: int, B: int, max_blocks: int, d_c: int, d_r: int, dtype=torch.bfloat16,
                 device="cuda", row_stride: int | None = None, block_table: torch.Tensor | None = None,
                 data: torch.Tensor | None = None):
        esz = 2 if dtype == torch.bfloat16 else 4
        R = d_c + d_r
        if row_stride is None:
            row_stride = ((R * esz + 15) // 16) * 16 // esz
        self.num_pages, self.B, self.max_blocks = num_pages, B, max_blocks
        self.d_c, self.d_r, self.row_stride, self.dtype = d_c, d_r, row_stride, dtype
        if data is None:
            data = torch.zeros((num_pages, PAGE_ROWS, row_stride), dtype=dtype, device=device)
        elif tuple(data.shape) != (num_pages, PAGE_ROWS, row_stride) or data.dtype != dtype:
            raise ValueError("page pool shape/dtype mismatch")
        self.data = data
        if block_table is None:
            block_table = torch.zeros((B, max_blocks), dtype=torch.int32, device=device)
        elif tuple(block_table.shape) != (B, max_blocks) or block_table.dtype != torch.int32:
            raise ValueError("block table must be int32 [B, max_blocks]")
        self.block_table = block_table.contiguous()

    @property
    def N_max(self) -> int:
        return self.max_blocks * PAGE_ROWS

    def struct(self) -> _PagedCache:
        return _PagedCache(self.data.data_ptr(), _DT[self.dtype], self.num_pages, self.d_c, self.d_r,
                           self.row_stride, self.block_table.data_ptr(), self.B, self.max_blocks)


def cache_append_paged(cache: PagedLatentCache, c_kv: torch.Tensor, k_r: torch.Tensor | None,
                       seq_idx: torch.Tensor, pos: torch.Tensor, rope_base: float = 10000.0) -> None:
    """Write T rows into the paged cache (see cache_append)."""
    _dev_tensor(c_kv, "c_kv", cache.dtype)
    if cache.d_r > 0:
        _dev_tensor(k_r, "k_r", cache.dtype)
    _dev_tensor(seq_idx, "seq_idx", torch.int32)
    _dev_tensor(pos, "pos", torch.int32)
    st = cache.struct()
    _check(lib().mla_cache_append_paged(ctypes.byref(st), _ptr(c_kv), _ptr(k_r if cache.d_r > 0 else None),
                                        _ptr(seq_idx), _ptr(pos), seq_idx.numel(), float(rope_base),
                                        _stream(c_kv)), "mla_cache_append_paged")


def decode_attn_paged(q_cat: torch.Tensor, cache: PagedLatentCache, seq_lens: torch.Tensor, scale: float,
                      workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      lse: torch.Tensor | None = None, want_lse: bool = True):
    """o_lat [B, H, d_c] (and lse [B, H]) of absorbed decode attention over a paged cache."""
    _dev_tensor(q_cat, "q_cat", cache.dtype)
    B, H, R = q_cat.shape
    if B != cache.B or R != cache.d_c + cache.d_r:
        raise ValueError("q_cat shape does not match the cache")
    _dev_tensor(seq_lens, "seq_lens", torch.int32)
    if seq_lens.numel() != B:
        raise ValueError("seq_lens needs one entry per sequence")
    if workspace is None:
        workspace = decode_workspace(B, H, cache.d_c, cache.dtype, q_cat.device)
    if out is None:
        out = torch.empty((B, H, cache.d_c), dtype=cache.dtype, device=q_cat.device)
    _out_tensor(out, "out", (B, H, cache.d_c), cache.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q_cat.device)
    if lse is not None:
        _out_tensor(lse, "lse", (B, H), torch.float32)
    st = cache.struct()
    _check(lib().mla_decode_attn_paged(_ptr(q_cat), ctypes.byref(st), _ptr(seq_lens), H, float(scale),
                                       _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse), _stream(q_cat)),
           "mla_decode_attn_paged")
    return out, lse


def kv_down_workspace(T: int, d_model: int, d_c: int, d_r: int, dtype=torch.bfloat16,
                      device="cuda") -> torch.Tensor:
    """Device scratch for kv_down_append of T tokens."""
    n = lib().mla_kv_down_workspace_size(T, d_model, d_c, d_r, _DT[dtype])
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def kv_down_append(cache, h: torch.Tensor, w_dkvr: torch.Tensor, gamma: torch.Tensor, seq_idx: torch.Tensor,
                   pos: torch.Tensor, eps: float = 1e-6, rope_base: float = 10000.0,
                   workspace: torch.Tensor | None = None) -> None:
    """Write the rows of T new tokens from their hidden states h [T, d_model]:
    cache[seq_idx[i], pos[i]] = [RMSNorm(h[i] W_DKV) * gamma || RoPE(h[i] W_KR, pos[i])],
    with w_dkvr = [W_DKV | W_KR] of shape [d_model, d_c + d_r] (LatentCache or
    PagedLatentCache)."""
    _dev_tensor(h, "h", cache.dtype)
    _dev_tensor(w_dkvr, "w_dkvr", cache.dtype)
    _dev_tensor(gamma, "gamma", cache.dtype)
    _dev_tensor(seq_idx, "seq_idx", torch.int32)
    _dev_tensor(pos, "pos", torch.int32)
    T, d_model = h.shape
    if tuple(w_dkvr.shape) != (d_model, cache.d_c + cache.d_r) or tuple(gamma.shape) != (cache.d_c,):
        raise ValueError("w_dkvr must be [d_model, d_c + d_r] and gamma [d_c]")
    if seq_idx.numel() != T or pos.numel() != T:
        raise ValueError("seq_idx and pos need one entry per token")
    if workspace is None:
        workspace = kv_down_workspace(T, d_model, cache.d_c, cache.d_r, cache.dtype, h.device)
    st = cache.struct()
    fn, name = ((lib().mla_kv_down_append_paged, "mla_kv_down_append_paged") if isinstance(cache, PagedLatentCache)
                else (lib().mla_kv_down_append, "mla_kv_down_append"))
    _check(fn(ctypes.byref(st), _ptr(h), _ptr(w_dkvr), _ptr(gamma), float(eps), _ptr(seq_idx), _ptr(pos), T,
              d_model, float(rope_base), _ptr(workspace), workspace.numel(), _stream(h)), name)


def prefill_explicit_workspace(B: int, start: int, S: int, H: int, device="cuda") -> torch.Tensor:
    """Device scratch for prefill_explicit (the rebuilt K_nope and V)."""
    n = lib().mla_prefill_explicit_workspace_size(B, start, S, H)
    if n == 0:
        raise MlaError(1, "mla_prefill_explicit_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def prefill_explicit(q_nope: torch.Tensor, q_rope: torch.Tensor, cache: LatentCache, w_uk: torch.Tensor,
                     w_uv: torch.Tensor, start: int, scale: float, causal: bool = True, rope_base: float = 10000.0,
                     workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                     lse: torch.Tensor | None = None, want_lse: bool = True):
    """o [B, S, H, d_v] (and lse [B, S, H]) of a prompt chunk at offset `start`
    without absorption: K and V rebuilt per head from the cached latent rows."""
    _dev_tensor(q_nope, "q_nope", cache.dtype)
    _dev_tensor(q_rope, "q_rope", cache.dtype)
    _dev_tensor(w_uk, "w_uk", cache.dtype)
    _dev_tensor(w_uv, "w_uv", cache.dtype)
    B, S, H, d_k = q_nope.shape
    if B != cache.B or tuple(q_rope.shape) != (B, S, H, cache.d_r):
        raise ValueError("q_nope / q_rope shapes do not match the cache")
    d_v = w_uv.shape[1]
    if tuple(w_uk.shape) != (H, d_k, cache.d_c) or tuple(w_uv.shape) != (H, d_v, cache.d_c):
        raise ValueError("w_uk must be [H, d_k, d_c] and w_uv [H, d_v, d_c]")
    if d_k != 128 or d_v != 128:
        raise MlaError(2, "prefill_explicit (d_k = d_v = 128 only)")
    if workspace is None:
        workspace = prefill_explicit_workspace(B, start, S, H, q_nope.device)
    if out is None:
        out = torch.empty((B, S, H, d_v), dtype=cache.dtype, device=q_nope.device)
    _out_tensor(out, "out", (B, S, H, d_v), cache.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=q_nope.device)
    if lse is not None:
        _out_tensor(lse, "lse", (B, S, H), torch.float32)
    st = cache.struct()
    _check(lib().mla_prefill_explicit(_ptr(q_nope), _ptr(q_rope), ctypes.byref(st), _ptr(w_uk), _ptr(w_uv),
                                      int(start), S, 1 if causal else 0, H, float(scale), float(rope_base),
                                      _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse), _stream(q_nope)),
           "mla_prefill_explicit")
    return out, lse
