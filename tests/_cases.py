"""Test-input builders shared by the GPU parity tests.

Inputs come from the seeded generators in ``mla_workloads``; expected values come
only from the float64 oracle.  The CUDA path receives the same materialised
(bf16 or fp32) bytes the oracle widens."""
from __future__ import annotations


import numpy as np
import torch

import mla_workloads as W
from oracle import mla_oracle as O

TOL_BF16_MAX_ABS = 2e-2
TOL_BF16_REL_L2 = 1e-2
# per output row (last axis): bf16 rounding of the stored outputs and of the MMA
# operands leaves ~0.2-0.6 % per row; a wrong row (a head, a block or a piece
# dropped or misplaced) is off by tens of percent, yet over thousands of rows it
# barely moves the global relative L2, and at long contexts the outputs are so
# small (~0.03 RMS) that the max-abs bound cannot see it either
TOL_BF16_ROW_REL_L2 = 5e-2
TOL_F32_REL_L2 = 1e-4


def to_device(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Upload a materialised array (float32, or bf16 bit patterns as uint16)."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def check_bf16(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx = float(np.max(np.abs(got - ref)))
    rl = rel_l2(got, ref)
    assert mx <= TOL_BF16_MAX_ABS and rl <= TOL_BF16_REL_L2, f"{what}: max_abs={mx:.3e} rel_l2={rl:.3e}"
    g2 = got.reshape(-1, got.shape[-1]) if got.ndim else got.reshape(1, 1)
    r2 = ref.reshape(-1, ref.shape[-1]) if ref.ndim else ref.reshape(1, 1)
    rn = np.linalg.norm(r2, axis=1)
    live = rn > 1e-6 * max(float(np.linalg.norm(r2)), 1e-300)  # rows that are exactly zero (empty sequences)
    if np.any(live):
        row = np.linalg.norm(g2 - r2, axis=1)[live] / rn[live]
        worst = int(np.argmax(row))
        assert row[worst] <= TOL_BF16_ROW_REL_L2, f"{what}: row {np.flatnonzero(live)[worst]} rel_l2={row[worst]:.3e}"
    return mx, rl


def check_f32(got: np.ndarray, ref: np.ndarray, what: str):
    rl = rel_l2(np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64))
    assert rl <= TOL_F32_REL_L2, f"{what}: rel_l2={rl:.3e}"
    return rl


class DecodeCase:
    """A decode batch: per-sequence cache inputs, queries and up-projection weights,
    drawn from a workload's distributions with optional overrides."""

    def __init__(self, workload: str, seed: int = 0, lens=None, H: int | None = None, d_r: int | None = None,
                 N_max: int | None = None):
        cfg = dict(W.WORKLOADS[workload])
        if H is not None:
            cfg["H"] = H
        if d_r is not None:
            cfg["d_r"] = d_r
        if lens is not None:
            lens = np.asarray(lens, dtype=np.int32)
            cfg["B"] = len(lens)
        else:
            lens = W.seq_lens(cfg, seed)
        self.cfg, self.seed, self.lens = cfg, seed, lens
        self.B, self.H, self.d_c, self.d_r = cfg["B"], cfg["H"], cfg["d_c"], cfg["d_r"]
        self.d_k, self.d_v = cfg["d_k"], cfg["d_v"]
        self.dtype = cfg["dtype"]
        self.base = cfg.get("rope_base", 10000.0)
        self.scale = cfg["scale"]
        self.N_max = int(N_max if N_max is not None else max(int(lens.max()), 1))
        self._rows = {}

    # -- materialised inputs --------------------------------------------------
    def seq_inputs(self, b: int):
        if b not in self._rows:
            c, k = W.latent_rows(self.cfg, self.seed, b, int(self.lens[b]))
            self._rows[b] = (W.as_dtype(c, self.dtype), W.as_dtype(k, self.dtype))
        return self._rows[b]

    def query(self):
        q_nope, q_r = W.query(self.cfg, self.seed)
        return W.as_dtype(q_nope[:, 0], self.dtype), W.as_dtype(q_r[:, 0], self.dtype)

    def weights(self):
        w_uk, w_uv = W.up_weights(self.cfg, self.seed)
        return W.as_dtype(w_uk, self.dtype), W.as_dtype(w_uv, self.dtype)

    # -- oracle -------------------------------------------------------------
    def oracle_seq(self, b: int):
        """(o [H, d_v], o_lat [H, d_c], lse [H]) of sequence b, float64."""
        n = int(self.lens[b])
        c, k = self.seq_inputs(b)
        q_nope, q_r = self.query()
        w_uk, w_uv = self.weights()
        wd = lambda x: W.widen(x, self.dtype)
        if n == 0:
            return (np.zeros((self.H, self.d_v)), np.zeros((self.H, self.d_c)), np.full(self.H, -np.inf))
        return O.decode_absorbed_from_parts(wd(q_nope[b]), wd(q_r[b]), n - 1, wd(c), wd(k), np.arange(n),
                                            wd(w_uk), wd(w_uv), self.scale, self.base)

    # -- device path ----------------------------------------------------------
    def device_cache(self, mla):
        tdt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        cache = mla.LatentCache(self.B, self.N_max, self.d_c, self.d_r, dtype=tdt)
        # fill unused rows with NaN so that any read past a sequence end shows up
        cache.data.fill_(float("nan"))
        for b in range(self.B):
            n = int(self.lens[b])
            if n == 0:
                continue
            c, k = self.seq_inputs(b)
            seq_idx = torch.full((n,), b, dtype=torch.int32, device="cuda")
            pos = torch.arange(n, dtype=torch.int32, device="cuda")
            mla.cache_append(cache, to_device(c, self.dtype), to_device(k, self.dtype) if self.d_r else None,
                             seq_idx, pos, self.base)
        return cache

    def run_device(self, mla, cache=None):
        """Append (if no cache given), absorb, decode, out-up on the GPU.  Returns
        numpy (o, o_lat, lse, q_cat)."""
        if cache is None:
            cache = self.device_cache(mla)
        q_nope, q_r = self.query()
        w_uk, w_uv = self.weights()
        q_pos = torch.from_numpy(np.maximum(self.lens - 1, 0).astype(np.int32)).cuda()
        q_cat = mla.absorb_q(to_device(q_nope, self.dtype), to_device(q_r, self.dtype) if self.d_r else None,
                             q_pos, to_device(w_uk, self.dtype), self.base)
        seq_lens = torch.from_numpy(self.lens).cuda()
        o_lat, lse = mla.decode_attn(q_cat, cache, seq_lens, self.scale)
        o = mla.out_up(o_lat, to_device(w_uv, self.dtype))
        torch.cuda.synchronize()
        f = lambda t: t.float().cpu().numpy().astype(np.float64)
        return f(o), f(o_lat), f(lse), f(q_cat)


def direct_decode_inputs(seed: int, lens, H: int, d_c: int, d_r: int, N_max: int | None = None):
    """Seeded bf16 q_cat [B, H, R] and cache rows (list of [n, R]) drawn directly,
    to test mla_decode_attn alone.  The latent part of q_cat has std 0.5 and the
    RoPE part std 1, which gives unit-variance scores at scale 1/sqrt(d_k + d_r)
    for the DeepSeek shapes."""
    R = d_c + d_r
    B = len(lens)
    q = W.normal(seed, "direct_q", (B, H, R))
    q[..., :d_c] *= 0.5
    q_bits = W.bf16_bits(q)
    rows = [W.bf16_bits(W.normal(seed, "direct_rows", (int(n), R), index=(b,))) for b, n in enumerate(lens)]
    return q_bits, rows


def oracle_direct(q_bits, rows, d_c: int, scale: float):
    out_o, out_lse = [], []
    for b, r in enumerate(rows):
        q = W.widen(q_bits[b], "bf16")
        if r.shape[0] == 0:
            out_o.append(np.zeros((q.shape[0], d_c)))
            out_lse.append(np.full(q.shape[0], -np.inf))
            continue
        o, lse = O.decode_absorbed(q, W.widen(r, "bf16"), d_c, scale)
        out_o.append(o)
        out_lse.append(lse)
    return np.stack(out_o), np.stack(out_lse)


def upload_direct(mla, q_bits, rows, d_c: int, d_r: int, N_max: int, row_stride=None):
    B = len(rows)
    cache = mla.LatentCache(B, N_max, d_c, d_r, dtype=torch.bfloat16, row_stride=row_stride)
    cache.data.fill_(float("nan"))
    for b, r in enumerate(rows):
        if r.shape[0]:
            cache.data[b, : r.shape[0], : d_c + d_r] = to_device(r, "bf16")
    return to_device(q_bits, "bf16"), cache
