"""GPU parity of mla_prefill_attn (absorbed prompt attention, causal and not)
against the float64 oracle, plus the whole prefill step at the full
B4 x S8192 x H128 size on sampled query rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import check_bf16, check_f32, to_device

pytestmark = pytest.mark.gpu

D_C, D_R = 512, 64


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import head_latent_attention_29_b300 as m
    return m


def prefill_inputs(seed: int, starts, S: int, H: int, d_c: int, d_r: int, dtype: str = "bf16"):
    """Seeded q_cat [B, S, H, R] (latent part std 0.5, RoPE part std 1: unit-variance
    scores at scale 1/sqrt(d_k + d_r)) and per-sequence cache rows [start + S, R]."""
    R = d_c + d_r
    B = len(starts)
    q = W.normal(seed, "prefill_q", (B, S, H, R))
    q[..., :d_c] *= 0.5
    rows = [W.as_dtype(W.normal(seed, "prefill_rows", (int(st) + S, R), index=(b,)), dtype)
            for b, st in enumerate(starts)]
    return W.as_dtype(q, dtype), rows


def upload(mla, q, rows, d_c, d_r, N_max, dtype="bf16"):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    cache = mla.LatentCache(len(rows), N_max, d_c, d_r, dtype=tdt)
    cache.data.fill_(float("nan"))  # rows past a query's limit must never be read
    for b, r in enumerate(rows):
        cache.data[b, : r.shape[0], : d_c + d_r] = to_device(r, dtype)
    return to_device(q, dtype), cache


def oracle_all(q, rows, starts, d_c, scale, causal, dtype="bf16", which=None):
    outs, lses = [], []
    for b, st in enumerate(starts):
        sel = range(q.shape[1]) if which is None else which
        o, l = O.prefill_absorbed_rows(W.widen(q[b], dtype), W.widen(rows[b], dtype), d_c, scale, sel,
                                       causal=causal, start=int(st))
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def run(mla, q_dev, cache, starts, scale, causal):
    q_start = torch.tensor(starts, dtype=torch.int32, device="cuda")
    o, lse = mla.prefill_attn(q_dev, cache, q_start, scale, causal=causal)
    torch.cuda.synchronize()
    st, detail = mla.get_device_error()
    assert st == 0, f"device error {st} ({detail:#x})"
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_two_sequences_all_rows(mla, causal):
    # 200 queries (several 64-row blocks and a ragged tail), the second sequence's
    # prompt after a 37-row prefix
    starts, S, H = [0, 37], 200, 128
    scale = 1.0 / np.sqrt(192.0)
    q, rows = prefill_inputs(1, starts, S, H, D_C, D_R)
    q_dev, cache = upload(mla, q, rows, D_C, D_R, max(starts) + S)
    o, lse = run(mla, q_dev, cache, starts, scale, causal)
    o_ref, lse_ref = oracle_all(q, rows, starts, D_C, scale, causal)
    check_bf16(o, o_ref, f"prefill o_lat causal={causal}")
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=2e-3)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_few_heads_no_rope(mla, causal):
    starts, S, H = [5, 0, 64], 130, 16
    scale = 1.0 / np.sqrt(128.0)
    q, rows = prefill_inputs(2, starts, S, H, D_C, 0)
    q_dev, cache = upload(mla, q, rows, D_C, 0, max(starts) + S + 3)
    o, lse = run(mla, q_dev, cache, starts, scale, causal)
    o_ref, lse_ref = oracle_all(q, rows, starts, D_C, scale, causal)
    check_bf16(o, o_ref, f"prefill H=16 d_r=0 causal={causal}")
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=2e-3)


def test_prefill_long_prefix_spans_many_runs(mla):
    # three queries after a 20000-row prefix: every query's rows are cut into pieces
    # by run boundaries and merged by the combine kernel
    starts, S, H = [20000], 3, 128
    scale = 1.0 / np.sqrt(192.0)
    q, rows = prefill_inputs(3, starts, S, H, D_C, D_R)
    q_dev, cache = upload(mla, q, rows, D_C, D_R, starts[0] + S)
    o, lse = run(mla, q_dev, cache, starts, scale, True)
    o_ref, lse_ref = oracle_all(q, rows, starts, D_C, scale, True)
    check_bf16(o, o_ref, "prefill long prefix")
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=2e-3)


def test_prefill_single_query_matches_decode(mla):
    # S = 1 at position start is the decode problem with start + 1 rows
    starts, S, H = [100, 4095, 0], 1, 128
    scale = 1.0 / np.sqrt(192.0)
    q, rows = prefill_inputs(4, starts, S, H, D_C, D_R)
    q_dev, cache = upload(mla, q, rows, D_C, D_R, max(starts) + 1)
    o, lse = run(mla, q_dev, cache, starts, scale, True)
    lens = torch.tensor([s + 1 for s in starts], dtype=torch.int32, device="cuda")
    o_d, lse_d = mla.decode_attn(q_dev[:, 0].contiguous(), cache, lens, scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o[:, 0], o_d.float().cpu().numpy())
    np.testing.assert_array_equal(lse[:, 0], lse_d.cpu().numpy())
    o_ref, lse_ref = oracle_all(q, rows, starts, D_C, scale, True)
    check_bf16(o, o_ref, "prefill S=1")


def test_prefill_block_aligned_lengths(mla):
    # causal lengths that end exactly on 64-row block boundaries (queries 63, 127)
    starts, S, H = [0, 64], 128, 64
    scale = 1.0 / np.sqrt(192.0)
    q, rows = prefill_inputs(5, starts, S, H, D_C, D_R)
    q_dev, cache = upload(mla, q, rows, D_C, D_R, max(starts) + S)
    o, lse = run(mla, q_dev, cache, starts, scale, True)
    o_ref, lse_ref = oracle_all(q, rows, starts, D_C, scale, True)
    check_bf16(o, o_ref, "prefill block-aligned")
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=2e-3)


def test_prefill_f32_tiny(mla):
    starts, S, H, d_c, d_r = [0, 9], 40, 4, 32, 8
    scale = 1.0 / np.sqrt(24.0)
    q, rows = prefill_inputs(6, starts, S, H, d_c, d_r, dtype="f32")
    q_dev, cache = upload(mla, q, rows, d_c, d_r, max(starts) + S, dtype="f32")
    for causal in (True, False):
        o, lse = run(mla, q_dev, cache, starts, scale, causal)
        o_ref, lse_ref = oracle_all(q, rows, starts, d_c, scale, causal, dtype="f32")
        check_f32(o, o_ref, f"prefill f32 causal={causal}")
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-5)


def test_prefill_start_out_of_range_is_recorded(mla):
    # q_start + S > N_max: lengths are clamped to the cache and the device error word
    # records MLA_ERR_DEVICE_INDEX (6)
    starts, S, H = [10], 8, 128
    q, rows = prefill_inputs(7, [0], S, H, D_C, D_R)
    q_dev, cache = upload(mla, q, rows, D_C, D_R, S)
    q_start = torch.tensor(starts, dtype=torch.int32, device="cuda")
    mla.prefill_attn(q_dev, cache, q_start, 0.07, causal=True)
    torch.cuda.synchronize()
    st, detail = mla.get_device_error()
    assert st == 6, (st, detail)


def test_prefill_full_size_step_sampled(mla):
    # B4 x S8192 x H128: append the prompt rows (RoPE at 0..8191), absorb every
    # query at its own position, prefill attention, W_UV.  Checked against the
    # oracle: every 61st query row plus the first and the last 64, all heads, of
    # every sequence (260 rows each)
    cfg = W.WORKLOADS["prefill_h128_b4_s8192"]
    B, S, H, d_k, d_v = cfg["B"], cfg["S"], cfg["H"], cfg["d_k"], cfg["d_v"]
    seed, base, scale = 11, cfg["rope_base"], cfg["scale"]
    w_uk, w_uv = (W.as_dtype(w, "bf16") for w in W.up_weights(cfg, seed))
    cache = mla.LatentCache(B, S, D_C, D_R, dtype=torch.bfloat16)
    q_cat = torch.empty((B, S, H, D_C + D_R), dtype=torch.bfloat16, device="cuda")
    w_uk_d = to_device(w_uk, "bf16")
    pos = torch.arange(S, dtype=torch.int32, device="cuda")
    host = {}
    for b in range(B):
        c, k = W.latent_rows(cfg, seed, b, S)
        c, k = W.as_dtype(c, "bf16"), W.as_dtype(k, "bf16")
        mla.cache_append(cache, to_device(c, "bf16"), to_device(k, "bf16"),
                         torch.full((S,), b, dtype=torch.int32, device="cuda"), pos, base)
        q_nope = W.as_dtype(W.normal(seed, "prefill_q_nope", (S, H, d_k), index=(b,)), "bf16")
        q_r = W.as_dtype(W.normal(seed, "prefill_q_r", (S, H, D_R), index=(b,)), "bf16")
        mla.absorb_q(to_device(q_nope, "bf16"), to_device(q_r, "bf16"), pos, w_uk_d, base, out=q_cat[b])
        host[b] = (c, k, q_nope, q_r)
    q_start = torch.zeros(B, dtype=torch.int32, device="cuda")
    o_lat, lse = mla.prefill_attn(q_cat, cache, q_start, scale, causal=True)
    o = mla.out_up(o_lat.view(B * S, H, D_C), to_device(w_uv, "bf16"))
    torch.cuda.synchronize()
    st, detail = mla.get_device_error()
    assert st == 0, (st, detail)
    o = o.view(B, S, H, d_v)
    wd = lambda x: W.widen(x, "bf16")
    rows_checked = sorted(set(range(0, S, 61)) | set(range(64)) | set(range(S - 64, S)))
    idx = torch.tensor(rows_checked, device="cuda")
    for b in range(B):
        c, k, q_nope, q_r = host[b]
        got_lat = o_lat[b].index_select(0, idx).float().cpu().numpy()
        got_o = o[b].index_select(0, idx).float().cpu().numpy()
        got_lse = lse[b].index_select(0, idx).cpu().numpy()
        rows = O.cache_rows(wd(c), wd(k), np.arange(S), base)
        q_ref = O.absorb_q(wd(q_nope[rows_checked]), wd(q_r[rows_checked]), np.asarray(rows_checked), wd(w_uk), base)
        for j, i in enumerate(rows_checked):
            ref_lat, ref_lse = O.decode_absorbed(q_ref[j], rows[: i + 1], D_C, scale)
            ref_o = O.out_up(ref_lat, wd(w_uv))
            check_bf16(got_lat[j], ref_lat, f"prefill o_lat b={b} i={i}")
            check_bf16(got_o[j], ref_o, f"prefill o b={b} i={i}")
            # q_lat is rounded to bf16 before the scores (as in the decode step): about
            # 2^-9 relative per term, a few 1e-3 on a unit-variance score
            np.testing.assert_allclose(got_lse[j], ref_lse, rtol=1e-3, atol=2e-2)
