"""GPU parity of mla_prefill_explicit (prefill without absorption: K and V rebuilt
per head from the cached latent rows, then standard causal attention) against the
float64 oracle, against the absorbed path on the same inputs, and at the full
B4 x S8192 x H128 prefill size on sampled query rows.

Inputs follow the prefill workload's distributions (latent rows, keys and queries
N(0,1), W_UK / W_UV N(0, 1/512), scale 1/sqrt(192): unit-variance scores).
Tolerances as for every bf16 output: max-abs <= 2e-2, relative L2 <= 1e-2."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import check_bf16, to_device

pytestmark = pytest.mark.gpu

D_C, D_R, D_K = 512, 64, 128
SCALE = 1.0 / math.sqrt(192.0)
BASE = 10000.0


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _inputs(seed, B, start, S, H, N_max):
    n = start + S
    c = [W.as_dtype(W.normal(seed, "px_c", (n, D_C), index=(b,)), "bf16") for b in range(B)]
    k = [W.as_dtype(W.normal(seed, "px_k", (n, D_R), index=(b,)), "bf16") for b in range(B)]
    q_nope = W.as_dtype(W.normal(seed, "px_qn", (B, S, H, D_K)), "bf16")
    q_r = W.as_dtype(W.normal(seed, "px_qr", (B, S, H, D_R)), "bf16")
    w_uk = W.as_dtype(W.normal(seed, "px_wuk", (H, D_K, D_C), std=1 / math.sqrt(D_C)), "bf16")
    w_uv = W.as_dtype(W.normal(seed, "px_wuv", (H, D_K, D_C), std=1 / math.sqrt(D_C)), "bf16")
    return c, k, q_nope, q_r, w_uk, w_uv


def _upload(mla, c, k, N_max):
    B, n = len(c), c[0].shape[0]
    cache = mla.LatentCache(B, N_max, D_C, D_R, dtype=torch.bfloat16)
    cache.data.fill_(float("nan"))  # rows past the prefix must never be read
    pos = torch.arange(n, dtype=torch.int32, device="cuda")
    for b in range(B):
        mla.cache_append(cache, to_device(c[b], "bf16"), to_device(k[b], "bf16"),
                         torch.full((n,), b, dtype=torch.int32, device="cuda"), pos, BASE)
    return cache


def _run(mla, cache, q_nope, q_r, w_uk, w_uv, start, causal):
    o, lse = mla.prefill_explicit(to_device(q_nope, "bf16"), to_device(q_r, "bf16"), cache, to_device(w_uk, "bf16"),
                                  to_device(w_uv, "bf16"), start, SCALE, causal=causal, rope_base=BASE)
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"
    return o, lse


# several 128-query tiles with a ragged last tile, a prefix that is not a multiple
# of the key tile, causal and not, and a cache longer than the prefix
@pytest.mark.parametrize("B,start,S,H,causal,extra", [(1, 0, 300, 4, True, 0), (2, 37, 200, 2, True, 64),
                                                      (1, 5, 130, 2, False, 0), (2, 130, 257, 2, True, 0)])
def test_prefill_explicit_matches_oracle(mla, B, start, S, H, causal, extra):
    c, k, q_nope, q_r, w_uk, w_uv = _inputs(B * 100 + start, B, start, S, H, start + S + extra)
    cache = _upload(mla, c, k, start + S + extra)
    o, lse = _run(mla, cache, q_nope, q_r, w_uk, w_uv, start, causal)
    wd = lambda x: W.widen(x, "bf16")
    for b in range(B):
        ro, rl = O.prefill_explicit_rows(wd(q_nope[b]), wd(q_r[b]), wd(c[b]), wd(k[b]), wd(w_uk), wd(w_uv), SCALE,
                                         BASE, range(S), causal, start)
        check_bf16(o[b].float().cpu().numpy(), ro, f"explicit prefill b={b} start={start} causal={causal}")
        np.testing.assert_allclose(lse[b].cpu().numpy(), rl, rtol=1e-3, atol=2e-2)


def test_prefill_explicit_equals_absorbed_path(mla):
    # the absorbed prompt path (absorb_q, prefill_attn, out_up) on the same rows
    B, start, S, H = 2, 64, 384, 16
    c, k, q_nope, q_r, w_uk, w_uv = _inputs(3, B, start, S, H, start + S)
    cache = _upload(mla, c, k, start + S)
    o_ex, lse_ex = _run(mla, cache, q_nope, q_r, w_uk, w_uv, start, True)
    pos = torch.arange(start, start + S, dtype=torch.int32, device="cuda")
    q_cat = torch.empty((B, S, H, D_C + D_R), dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        mla.absorb_q(to_device(q_nope[b], "bf16"), to_device(q_r[b], "bf16"), pos, to_device(w_uk, "bf16"), BASE,
                     out=q_cat[b])
    o_lat, lse_ab = mla.prefill_attn(q_cat, cache, torch.full((B,), start, dtype=torch.int32, device="cuda"), SCALE)
    o_ab = mla.out_up(o_lat.view(B * S, H, D_C), to_device(w_uv, "bf16")).view(B, S, H, D_K)
    torch.cuda.synchronize()
    check_bf16(o_ex.float().cpu().numpy(), o_ab.float().cpu().numpy(), "explicit vs absorbed")
    np.testing.assert_allclose(lse_ex.cpu().numpy(), lse_ab.cpu().numpy(), rtol=1e-3, atol=2e-2)


def test_prefill_explicit_full_size_sampled(mla):
    # B4 x S8192 x H128 prompt (prefill workload shapes): every 61st query row plus
    # the first and the last 64 of each prompt (260 rows each), all heads, against
    # the oracle's absorbed form, which its pins tie to the explicit form
    cfg = W.WORKLOADS["prefill_h128_b4_s8192"]
    B, S, H = cfg["B"], cfg["S"], cfg["H"]
    seed = 13
    w_uk, w_uv = (W.as_dtype(w, "bf16") for w in W.up_weights(cfg, seed))
    cache = mla.LatentCache(B, S, D_C, D_R, dtype=torch.bfloat16)
    pos = torch.arange(S, dtype=torch.int32, device="cuda")
    q_nope = torch.empty((B, S, H, D_K), dtype=torch.bfloat16, device="cuda")
    q_r = torch.empty((B, S, H, D_R), dtype=torch.bfloat16, device="cuda")
    host = {}
    for b in range(B):
        c, k = (W.as_dtype(x, "bf16") for x in W.latent_rows(cfg, seed, b, S))
        mla.cache_append(cache, to_device(c, "bf16"), to_device(k, "bf16"),
                         torch.full((S,), b, dtype=torch.int32, device="cuda"), pos, BASE)
        qn = W.as_dtype(W.normal(seed, "prefill_q_nope", (S, H, D_K), index=(b,)), "bf16")
        qr = W.as_dtype(W.normal(seed, "prefill_q_r", (S, H, D_R), index=(b,)), "bf16")
        q_nope[b] = to_device(qn, "bf16")
        q_r[b] = to_device(qr, "bf16")
        host[b] = (c, k, qn, qr)
    o, lse = mla.prefill_explicit(q_nope, q_r, cache, to_device(w_uk, "bf16"), to_device(w_uv, "bf16"), 0,
                                  cfg["scale"], causal=True, rope_base=BASE)
    torch.cuda.synchronize()
    assert mla.get_device_error()[0] == 0
    wd = lambda x: W.widen(x, "bf16")
    rows_checked = sorted(set(range(0, S, 61)) | set(range(64)) | set(range(S - 64, S)))
    idx = torch.tensor(rows_checked, device="cuda")
    for b in range(B):
        c, k, qn, qr = host[b]
        got_o = o[b].index_select(0, idx).float().cpu().numpy()
        got_lse = lse[b].index_select(0, idx).cpu().numpy()
        rows = O.cache_rows(wd(c), wd(k), np.arange(S), BASE)
        q_ref = O.absorb_q(wd(qn[rows_checked]), wd(qr[rows_checked]), np.asarray(rows_checked), wd(w_uk), BASE)
        for j, i in enumerate(rows_checked):
            ref_lat, ref_lse = O.decode_absorbed(q_ref[j], rows[: i + 1], D_C, cfg["scale"])
            check_bf16(got_o[j], O.out_up(ref_lat, wd(w_uv)), f"explicit prefill b={b} i={i}")
            np.testing.assert_allclose(got_lse[j], ref_lse, rtol=1e-3, atol=2e-2)
