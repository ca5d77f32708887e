"""Float64 CPU oracle for Multi-head Latent Attention (MLA) decode.

TEST INFRASTRUCTURE ONLY.  This module is the independent definition that the
CUDA path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the product library never does.
It shares no code with the CUDA kernels: the only thing both sides share is the
seeded input module ``mla_workloads``.

Everything here is plain float64 numpy, written to be read against the pages:

* "MLA multi-head latent attention: low-rank compression and matrix absorption"
  (0539edu.com) -- section 2.2 (c_KV = h W_DKV, k = c_KV W_UK, v = c_KV W_UV,
  softmax attention), section 3.1 (absorption: q k^T = (q W_UK^T) c_KV^T and
  attn v = (attn c_KV) W_UV), section 3.2 and section 5.1 (the absorbed
  inference form, weights viewed as [h, d_k, d_c] / [h, d_v, d_c]),
  section 5.2 (the preallocated latent cache written by position).
* The attention-variants interview guide (hotelren.com) -- section 6.2
  (a separate RoPE key k_rope of width d_rope shared by all heads, concatenated
  to the per-head no-position key) and section 7.3 (subtract the row maximum
  before exponentiating).
* The icman.com.cn MLA article -- section 2 "decoupled RoPE" and its cache-row
  figure: each token caches 512 latent values plus a 64-wide key with RoPE
  already applied.
* "Gated MLA" (tahou.com) -- section 2.6 / 3.2 (full-rank sigmoid output gate
  multiplied channel-wise into the concatenated v-width output) and section 3.3
  (no positional encoding in the gated variant).
* The same 0539edu.com article, section 6.3: an RMSNorm placed after the
  compression projection keeps c_KV's range stable over long contexts (as in
  DeepSeek-V3), written there as an RMSNorm module of width d_c applied to
  h W_DKV; and the interview guide's section 6.2 listing, where the RoPE key is
  its own projection h W_KR of the hidden state.

Readings where the pages are silent:
RoPE rotates adjacent pairs (2i, 2i+1) with theta_i = base^(-2i/d_r); the decode
query sits at position N-1 and attends to all N cached tokens including itself;
the softmax scale is a runtime argument; the RMSNorm has a per-channel gain gamma
(all ones when untrained) and a runtime epsilon inside the square root.

Parity status: every function below is pinned by tests/test_oracle_pins.py
(closed forms, invariants, brute force on tiny shapes, and the pages' printed
cache-size values).
"""
from __future__ import annotations

import numpy as np

LOG2E = 1.4426950408889634


# --------------------------------------------------------------------------
# Rotary position embedding on the decoupled key / query part
# --------------------------------------------------------------------------
def rope_angles(pos, d_r: int, base: float) -> np.ndarray:
    """Angles pos * theta_i for i in [0, d_r/2), theta_i = base^(-2i/d_r).

    The pages only say the position key is rotated in the complex plane
    (icman.com.cn article, section 2); the pairing and frequency schedule are
    the standard RoPE reading."""
    i = np.arange(d_r // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / d_r)
    return np.asarray(pos, dtype=np.float64)[..., None] * theta


def rope(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate pairs (x[2i], x[2i+1]) of the last axis by angle pos * theta_i."""
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    if d_r == 0:
        return x.copy()
    ang = rope_angles(pos, d_r, base)
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# --------------------------------------------------------------------------
# Latent cache
# --------------------------------------------------------------------------
def cache_rows(c_kv: np.ndarray, k_r_raw: np.ndarray, positions, base: float) -> np.ndarray:
    """One sequence's cached rows [n, d_c + d_r] = [c_KV || RoPE(k_R, position)].

    The row layout is the icman.com.cn cache-row figure (latent first, then the
    rotated position key); the position-indexed write is the preallocated cache
    of the 0539edu.com page, section 5.2."""
    c_kv = np.asarray(c_kv, dtype=np.float64)
    k_rot = rope(k_r_raw, positions, base)
    return np.concatenate([c_kv, k_rot], axis=-1)


def latent_row_elements(d_c: int, d_r: int) -> int:
    """Elements cached per token per layer by MLA (icman.com.cn section 2 figure)."""
    return d_c + d_r


def mha_kv_elements(h: int, d: int) -> int:
    """Elements cached per token per layer by MHA: one K and one V per head
    (0539edu.com section 1)."""
    return 2 * h * d


def kv_cache_bytes(layers: int, heads: int, head_dim: int, seq: int, batch: int,
                   elem_bytes: int, kv_factor: int = 2) -> int:
    """Total MHA/GQA cache bytes: kv_factor * heads * head_dim * seq * batch * bytes
    per layer, times layers (nxmr.cn article, section 1.1)."""
    return layers * kv_factor * heads * head_dim * seq * batch * elem_bytes


def compression_ratio(h: int, d_k: int, d_v: int, d_c: int) -> float:
    """(h d_k + h d_v) / d_c (0539edu.com section 2.3)."""
    return (h * d_k + h * d_v) / d_c


# --------------------------------------------------------------------------
# Attention pieces
# --------------------------------------------------------------------------
def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first (hotelren.com section 7.3)."""
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def logsumexp_rows(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=-1)
    return m + np.log(np.sum(np.exp(s - m[..., None]), axis=-1))


def absorb_q(q_nope: np.ndarray, q_rope: np.ndarray, q_pos, w_uk: np.ndarray,
             base: float) -> np.ndarray:
    """Absorbed query q_cat = [q_nope_h W_UK_h || RoPE(q_R_h, pos)] per head.

    q_nope [..., H, d_k], q_rope [..., H, d_r], w_uk [H, d_k, d_c] (the
    [h, d_k, d_c] view of the up-projection weight, 0539edu.com section 5.1).
    q_lat[h, c] = sum_d q_nope[h, d] W_UK[h, d, c]: the W_UK half of the
    absorption identity (0539edu.com section 3.1).  q_pos broadcasts over the
    leading axes of q_rope without H."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    q_lat = np.einsum("...hd,hdc->...hc", q_nope, w_uk)
    pos = np.asarray(q_pos, dtype=np.float64)[..., None]  # broadcast over heads
    q_rot = rope(q_rope, pos, base)
    return np.concatenate([q_lat, q_rot], axis=-1)


def decode_absorbed(q_cat: np.ndarray, rows: np.ndarray, d_c: int, scale: float):
    """Absorbed decode attention for one sequence.

    q_cat [H, d_c + d_r], rows [n, d_c + d_r] (the cached rows).  Scores are
    scale * (q_lat . c_KV + q_R . k_R) over the whole row, softmax over the n
    tokens, o_lat = P c_KV (0539edu.com sections 3.1-3.2, icman.com.cn section 2).
    Returns (o_lat [H, d_c], lse [H]) with lse the natural log-sum-exp of the
    scaled scores."""
    q_cat = np.asarray(q_cat, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    s = scale * (q_cat @ rows.T)
    p = softmax_rows(s)
    o_lat = p @ rows[:, :d_c]
    return o_lat, logsumexp_rows(s)


def out_up(o_lat: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """o[h, d] = sum_c o_lat[h, c] W_UV[h, d, c]: W_UV applied after attention
    (0539edu.com section 3.1, second identity; weight view [h, d_v, d_c] of
    section 3.2)."""
    return np.einsum("...hc,hdc->...hd", np.asarray(o_lat, dtype=np.float64),
                     np.asarray(w_uv, dtype=np.float64))


def decode_explicit(q_nope: np.ndarray, q_rope: np.ndarray, q_pos: int,
                    c_kv: np.ndarray, k_r_raw: np.ndarray, positions,
                    w_uk: np.ndarray, w_uv: np.ndarray, scale: float, base: float):
    """Decode attention with K and V rebuilt per head (no absorption).

    k_h,t = [c_KV,t W_UK,h^T || RoPE(k_R,t, t)], v_h,t = c_KV,t W_UV,h^T,
    q_h = [q_nope,h || RoPE(q_R,h, q_pos)]; standard softmax attention
    (0539edu.com section 2.2 and its training-form listing in section 3.2;
    hotelren.com section 6.2 for the shared rotated key).
    Returns o [H, d_v]."""
    c_kv = np.asarray(c_kv, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    k_nope = np.einsum("tc,hdc->htd", c_kv, w_uk)            # [H, n, d_k]
    v = np.einsum("tc,hdc->htd", c_kv, w_uv)                 # [H, n, d_v]
    k_rot = rope(k_r_raw, positions, base)                   # [n, d_r], shared
    q_rot = rope(q_rope, q_pos, base)                        # [H, d_r]
    s = scale * (np.einsum("hd,htd->ht", np.asarray(q_nope, dtype=np.float64), k_nope)
                 + q_rot @ k_rot.T)
    p = softmax_rows(s)
    return np.einsum("ht,htd->hd", p, v)


def decode_absorbed_from_parts(q_nope, q_rope, q_pos, c_kv, k_r_raw, positions,
                               w_uk, w_uv, scale, base):
    """The absorbed form end to end for one sequence: absorb_q, cache rows,
    decode_absorbed, out_up.  Returns (o [H, d_v], o_lat [H, d_c], lse [H])."""
    d_c = np.asarray(c_kv).shape[-1]
    q_cat = absorb_q(q_nope, q_rope, q_pos, w_uk, base)
    rows = cache_rows(c_kv, k_r_raw, positions, base)
    o_lat, lse = decode_absorbed(q_cat, rows, d_c, scale)
    return out_up(o_lat, w_uv), o_lat, lse


# --------------------------------------------------------------------------
# Split-KV partials and their log-sum-exp merge
# --------------------------------------------------------------------------
def decode_partial(q_cat: np.ndarray, rows: np.ndarray, d_c: int, scale: float):
    """Unnormalised partial over a token subset: (m, l, O) with m the row max of
    the scaled scores, l = sum exp(s - m), O = sum exp(s - m) c_KV."""
    s = scale * (np.asarray(q_cat, dtype=np.float64) @ np.asarray(rows, dtype=np.float64).T)
    m = np.max(s, axis=-1)
    e = np.exp(s - m[:, None])
    return m, e.sum(axis=-1), e @ np.asarray(rows, dtype=np.float64)[:, :d_c]


def lse_merge(parts):
    """Merge partials (m_s, l_s, O_s): M = max m_s, L = sum l_s e^(m_s - M),
    o = sum e^(m_s - M) O_s / L, lse = M + ln L.  This restates the max
    subtraction of hotelren.com section 7.3 across token subsets."""
    ms = np.stack([p[0] for p in parts])
    M = ms.max(axis=0)
    w = np.exp(ms - M)
    L = sum(wi * p[1] for wi, p in zip(w, parts))
    O = sum(wi[:, None] * p[2] for wi, p in zip(w, parts))
    return O / L[:, None], M + np.log(L)


# --------------------------------------------------------------------------
# Gated variant and prefill
# --------------------------------------------------------------------------
def gate(h: np.ndarray, w_g: np.ndarray, o_flat: np.ndarray) -> np.ndarray:
    """o_flat * sigmoid(h W_g): the full-rank, input-dependent, channel-wise
    output gate over the concatenated v width (tahou.com sections 2.6, 3.2)."""
    z = np.asarray(h, dtype=np.float64) @ np.asarray(w_g, dtype=np.float64)
    return np.asarray(o_flat, dtype=np.float64) * (1.0 / (1.0 + np.exp(-z)))


def prefill_absorbed_rows(q_cat: np.ndarray, rows: np.ndarray, d_c: int, scale: float,
                          query_positions, causal: bool = True, start: int = 0):
    """Absorbed attention of selected prompt queries against the cache prefix
    (hotelren.com guide, section 2.1: prefill handles the whole prompt at once;
    0539edu.com sections 3.1-3.2: the absorbed scores keep their per-position shape).

    q_cat [S, H, R] for the S prompt queries, which sit at positions start..start+S-1;
    rows [start + S, R] the cached rows of the sequence up to the prompt's end.
    Query i reads rows 0..start+i when causal (its own row included), else all
    start + S rows.  Returns (o_lat [k, H, d_c], lse [k, H]) for the k selected i."""
    q_cat = np.asarray(q_cat, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    outs, lses = [], []
    for i in query_positions:
        n = start + i + 1 if causal else start + q_cat.shape[0]
        o, l = decode_absorbed(q_cat[i], rows[:n], d_c, scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def prefill_explicit_rows(q_nope: np.ndarray, q_rope: np.ndarray, c_kv: np.ndarray, k_r_raw: np.ndarray,
                          w_uk: np.ndarray, w_uv: np.ndarray, scale: float, base: float,
                          query_positions, causal: bool = True, start: int = 0):
    """Prefill without absorption: every head's keys and values are rebuilt from the
    latent once, k_h,t = [c_KV,t W_UK,h^T || RoPE(k_R,t, t)] and v_h,t = c_KV,t W_UV,h^T,
    and the prompt queries q_h,i = [q_nope,h,i || RoPE(q_R,h,i, start + i)] run standard
    softmax attention (0539edu.com section 2.2 and the training-form listing of
    section 3.2; the same page notes the absorbed form costs more compute in prefill
    and that the explicit form is the precision fallback; hotelren.com section 6.2
    for the rotated key shared by all heads).

    q_nope [S, H, d_k], q_rope [S, H, d_r] for the prompt queries at positions
    start..start+S-1; c_kv [n, d_c] and k_r_raw [n, d_r] for the sequence's rows
    0..n-1 (n >= start + S).  Query i reads rows 0..start+i when causal, else rows
    0..start+S-1.  Returns (o [k, H, d_v], lse [k, H]) for the k selected i."""
    c_kv = np.asarray(c_kv, dtype=np.float64)
    k_nope = np.einsum("tc,hdc->htd", c_kv, np.asarray(w_uk, dtype=np.float64))   # [H, n, d_k]
    v = np.einsum("tc,hdc->htd", c_kv, np.asarray(w_uv, dtype=np.float64))        # [H, n, d_v]
    k_rot = rope(k_r_raw, np.arange(c_kv.shape[0]), base)                           # [n, d_r]
    q_nope = np.asarray(q_nope, dtype=np.float64)
    S = q_nope.shape[0]
    outs, lses = [], []
    for i in query_positions:
        n = start + i + 1 if causal else start + S
        q_rot = rope(q_rope[i], start + i, base)                                   # [H, d_r]
        s = scale * (np.einsum("hd,htd->ht", q_nope[i], k_nope[:, :n]) + q_rot @ k_rot[:n].T)
        outs.append(np.einsum("ht,htd->hd", softmax_rows(s), v[:, :n]))
        lses.append(logsumexp_rows(s))
    return np.stack(outs), np.stack(lses)


# --------------------------------------------------------------------------
# Tiny hidden-state-driven decode (projections as input preparation)
# --------------------------------------------------------------------------
def project_from_hidden(h: np.ndarray, w_dkv, w_kr, w_uq, H: int, d_k: int, d_r: int):
    """c_KV = h W_DKV (0539edu.com section 2.2), k_R = h W_KR (hotelren.com
    section 6.2, one key shared by all heads), [q_nope || q_R]_h = h W_UQ split per
    head, the first d_k columns then the last d_r.  h [n, d_model]."""
    h = np.asarray(h, dtype=np.float64)
    c_kv = h @ np.asarray(w_dkv, dtype=np.float64)
    k_r = h @ np.asarray(w_kr, dtype=np.float64)
    q = (h @ np.asarray(w_uq, dtype=np.float64)).reshape(h.shape[0], H, d_k + d_r)
    return c_kv, k_r, q[..., :d_k], q[..., d_k:]


# --------------------------------------------------------------------------
# Cache rows straight from hidden states: normalised latent + rotated key
# --------------------------------------------------------------------------
def rms_norm(x: np.ndarray, gamma, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps), scaled channel-wise
    by gamma (0539edu.com section 6.3: applied to c_KV right after h W_DKV)."""
    x = np.asarray(x, dtype=np.float64)
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + float(eps)) * np.asarray(gamma, dtype=np.float64)


def kv_down_rows(h: np.ndarray, w_dkv, w_kr, gamma, eps: float, positions, base: float) -> np.ndarray:
    """The cache rows new tokens write, computed from their hidden states h [n, d_model]:
    [RMSNorm(h W_DKV) || RoPE(h W_KR, position)] (0539edu.com sections 2.2 and 6.3
    for the normalised latent; hotelren.com section 6.2 for the key projection
    shared by all heads; icman.com.cn section 2 for caching the key rotated)."""
    h = np.asarray(h, dtype=np.float64)
    c_kv = rms_norm(h @ np.asarray(w_dkv, dtype=np.float64), gamma, eps)
    k_r = h @ np.asarray(w_kr, dtype=np.float64)
    return cache_rows(c_kv, k_r, positions, base)
