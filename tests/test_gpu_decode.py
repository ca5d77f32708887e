"""GPU parity of the decode path against the float64 oracle (bf16 and fp32).

Tolerances: bf16 inputs -- max-abs <= 2e-2 and relative L2 <= 1e-2; fp32 inputs --
relative L2 <= 1e-4 (both against the float64 oracle on the same seeded inputs)."""
import math

import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import (DecodeCase, check_bf16, check_f32, direct_decode_inputs, oracle_direct, to_device,
                          upload_direct)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _decode_direct(mla, lens, H, d_r, seed=0, N_max=None, row_stride=None):
    d_c = 512
    lens = np.asarray(lens, dtype=np.int32)
    N_max = N_max or max(int(lens.max()), 1)
    scale = 1.0 / math.sqrt(128 + d_r)
    q_bits, rows = direct_decode_inputs(seed, lens, H, d_c, d_r)
    q, cache = upload_direct(mla, q_bits, rows, d_c, d_r, N_max, row_stride)
    o_lat, lse = mla.decode_attn(q, cache, torch.from_numpy(lens).cuda(), scale)
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"
    ref_o, ref_lse = oracle_direct(q_bits, rows, d_c, scale)
    return o_lat.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse


# ---------------------------------------------------------------------------
# mla_decode_attn alone, seeded q_cat and cache rows
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [200, 1, 64, 129], [4097, 300], [1000] * 5])
def test_decode_ragged_lengths_rope(mla, lens):
    o, lse, ro, rlse = _decode_direct(mla, lens, H=128, d_r=64)
    check_bf16(o, ro, f"o_lat lens={lens}")
    np.testing.assert_allclose(lse, rlse, atol=2e-2, rtol=1e-3)


@pytest.mark.parametrize("H", [128, 64, 100, 16])
def test_decode_head_counts(mla, H):
    o, lse, ro, rlse = _decode_direct(mla, [777, 64, 1500], H=H, d_r=64, seed=1)
    check_bf16(o, ro, f"o_lat H={H}")
    np.testing.assert_allclose(lse, rlse, atol=2e-2, rtol=1e-3)


def test_decode_without_rope_key(mla):
    o, lse, ro, rlse = _decode_direct(mla, [900, 65, 3000], H=64, d_r=0, seed=2)
    check_bf16(o, ro, "o_lat no-rope")
    np.testing.assert_allclose(lse, rlse, atol=2e-2, rtol=1e-3)


def test_decode_zero_length_and_padded_rows(mla):
    # a zero-length sequence gives zeros / -inf; N_max larger than every length;
    # rows padded to a 640-element stride
    o, lse, ro, rlse = _decode_direct(mla, [0, 70, 1], H=128, d_r=64, seed=3, N_max=300, row_stride=640)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    check_bf16(o[1:], ro[1:], "o_lat padded")
    np.testing.assert_allclose(lse[1:], rlse[1:], atol=2e-2, rtol=1e-3)


def test_decode_many_runs_span_sequences(mla):
    # enough blocks that runs of the token stream cross sequence boundaries
    rng = np.random.default_rng(4)
    lens = rng.integers(1, 2500, size=40)
    o, lse, ro, rlse = _decode_direct(mla, lens, H=128, d_r=64, seed=4)
    check_bf16(o, ro, "o_lat spanning runs")
    np.testing.assert_allclose(lse, rlse, atol=2e-2, rtol=1e-3)


def test_decode_large_scores_trigger_rescale(mla):
    # a peaked query: later blocks exceed the running maximum by far more than the
    # 2^8 threshold, which exercises the in-place rescaling of the accumulator
    lens = np.array([3000, 2000], dtype=np.int32)
    d_c, d_r, H = 512, 64, 128
    q_bits, rows = direct_decode_inputs(5, lens, H, d_c, d_r)
    # make scores grow along the sequence through the RoPE key columns (which do
    # not enter o_lat, so the output keeps unit magnitude): the score of token t
    # rises by ~20 (natural units) from the first block to the last
    for b, r in enumerate(rows):
        f = W.bf16_to_f32(r)
        f[:, d_c] = np.linspace(-3, 3, f.shape[0]).astype(np.float32) * 4
        rows[b] = W.bf16_bits(f)
    qf = W.bf16_to_f32(q_bits)
    qf[..., d_c] = 6.0
    q_bits = W.bf16_bits(qf)
    scale = 1.0 / math.sqrt(192)
    q, cache = upload_direct(mla, q_bits, rows, d_c, d_r, int(lens.max()))
    o_lat, lse = mla.decode_attn(q, cache, torch.from_numpy(lens).cuda(), scale)
    ref_o, ref_lse = oracle_direct(q_bits, rows, d_c, scale)
    check_bf16(o_lat.float().cpu().numpy(), ref_o, "o_lat rescale")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, atol=2e-2, rtol=1e-3)


def test_decode_out_of_range_length_is_recorded(mla):
    lens = np.array([50, 70], dtype=np.int32)
    q_bits, rows = direct_decode_inputs(6, lens, 128, 512, 64)
    q, cache = upload_direct(mla, q_bits, rows, 512, 64, 70)
    bad = torch.tensor([50, 71], dtype=torch.int32, device="cuda")  # 71 > N_max
    mla.decode_attn(q, cache, bad, 0.07)
    st, word = mla.get_device_error()
    assert st == 6 and (word >> 8) == 2
    assert mla.get_device_error()[0] == 0  # cleared


# ---------------------------------------------------------------------------
# The full decode step through the C ABI: append (RoPE), absorb, attention, out-up
# ---------------------------------------------------------------------------
def test_step_tiny_fp32_from_hidden_states(mla):
    cfg = W.WORKLOADS["tiny_fp32"]
    m = W.hidden_model(cfg, seed=0)
    H, d_k, d_r, d_c, N = cfg["H"], cfg["d_k"], cfg["d_r"], cfg["d_c"], cfg["N"]
    h = m["h"][0]
    # input preparation: the projections (not part of the decode path), taken from
    # the oracle's pinned projection function and rounded to fp32
    hd = W.widen(h, "f32")
    c64, k64, qn64, qr64 = O.project_from_hidden(hd, m["w_dkv"], m["w_kr"], m["w_uq"], H, d_k, d_r)
    c_kv, k_r = c64.astype(np.float32), k64.astype(np.float32)
    q = np.concatenate([qn64[N - 1], qr64[N - 1]], axis=-1).astype(np.float32)
    cache = mla.LatentCache(1, N, d_c, d_r, dtype=torch.float32)
    mla.cache_append(cache, to_device(c_kv, "f32"), to_device(k_r, "f32"),
                     torch.zeros(N, dtype=torch.int32, device="cuda"),
                     torch.arange(N, dtype=torch.int32, device="cuda"), cfg["rope_base"])
    q_cat = mla.absorb_q(to_device(q[None, :, :d_k], "f32"), to_device(q[None, :, d_k:], "f32"),
                         torch.tensor([N - 1], dtype=torch.int32, device="cuda"), to_device(m["w_uk"], "f32"),
                         cfg["rope_base"])
    o_lat, lse = mla.decode_attn(q_cat, cache, torch.tensor([N], dtype=torch.int32, device="cuda"), cfg["scale"])
    o = mla.out_up(o_lat, to_device(m["w_uv"], "f32"))
    torch.cuda.synchronize()
    # oracle from the same hidden states, both forms
    pos = np.arange(N)
    ref_o, ref_lat, ref_lse = O.decode_absorbed_from_parts(qn64[N - 1], qr64[N - 1], N - 1, c64, k64, pos,
                                                           m["w_uk"], m["w_uv"], cfg["scale"], cfg["rope_base"])
    ref_exp = O.decode_explicit(qn64[N - 1], qr64[N - 1], N - 1, c64, k64, pos, m["w_uk"], m["w_uv"],
                                cfg["scale"], cfg["rope_base"])
    check_f32(o.cpu().numpy()[0], ref_o, "o (absorbed oracle)")
    check_f32(o.cpu().numpy()[0], ref_exp, "o (explicit oracle)")
    check_f32(o_lat.cpu().numpy()[0], ref_lat, "o_lat")
    check_f32(lse.cpu().numpy()[0], ref_lse, "lse")


def test_cache_append_rotates_the_key(mla):
    case = DecodeCase("decode_h128_b32_n4096", seed=7, lens=[300, 5000])
    cache = case.device_cache(mla)
    torch.cuda.synchronize()
    for b in range(2):
        n = int(case.lens[b])
        c, k = case.seq_inputs(b)
        ref = O.cache_rows(W.widen(c, "bf16"), W.widen(k, "bf16"), np.arange(n), case.base)
        got = cache.rows[b, :n].float().cpu().numpy()
        np.testing.assert_array_equal(got[:, :512], W.widen(c, "bf16"))   # latent copied bit-exactly
        # rotated key: one bf16 rounding of the exact rotation
        np.testing.assert_allclose(got[:, 512:], ref[:, 512:], rtol=2 ** -8, atol=1e-6)


def test_absorb_q_matches_oracle(mla):
    case = DecodeCase("decode_h128_b32_n4096", seed=8, lens=[4096] * 32)
    q_nope, q_r = case.query()
    w_uk, _ = case.weights()
    q_pos = torch.full((32,), 4095, dtype=torch.int32, device="cuda")
    q_cat = mla.absorb_q(to_device(q_nope, "bf16"), to_device(q_r, "bf16"), q_pos, to_device(w_uk, "bf16"))
    ref = O.absorb_q(W.widen(q_nope, "bf16"), W.widen(q_r, "bf16"), np.full(32, 4095), W.widen(w_uk, "bf16"), 1e4)
    check_bf16(q_cat.float().cpu().numpy(), ref, "q_cat")


def test_out_up_matches_oracle(mla):
    rng_o = W.bf16_bits(W.normal(9, "o_lat_direct", (32, 128, 512)))
    _, w_uv = DecodeCase("decode_h128_b32_n4096", seed=9, lens=[1] * 32).weights()
    o = mla.out_up(to_device(rng_o, "bf16"), to_device(w_uv, "bf16"))
    ref = O.out_up(W.widen(rng_o, "bf16"), W.widen(w_uv, "bf16"))
    check_bf16(o.float().cpu().numpy(), ref, "o")


def test_step_headline_workload_full_size(mla):
    """B=32, H=128, d_c=512, d_r=64, N=4096 bf16: every sequence checked."""
    case = DecodeCase("decode_h128_b32_n4096", seed=0)
    o, o_lat, lse, _ = case.run_device(mla)
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"
    ref = [case.oracle_seq(b) for b in range(case.B)]
    check_bf16(o_lat, np.stack([r[1] for r in ref]), "o_lat headline")
    check_bf16(o, np.stack([r[0] for r in ref]), "o headline")
    np.testing.assert_allclose(lse, np.stack([r[2] for r in ref]), atol=2e-2, rtol=1e-3)


def test_step_ragged_long_context_full_size(mla):
    """B=64, lengths uniform in [1024, 32768]: the whole batch runs and every
    sequence is checked against the oracle (most of them are cut by run
    boundaries, so their pieces go through the log-sum-exp combine)."""
    case = DecodeCase("ragged_h128_b64_n1k_32k", seed=0)
    o, o_lat, lse, _ = case.run_device(mla)
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"
    for b in range(case.B):
        r_o, r_lat, r_lse = case.oracle_seq(b)
        check_bf16(o_lat[b], r_lat, f"o_lat ragged b={b} n={case.lens[b]}")
        check_bf16(o[b], r_o, f"o ragged b={b}")
        np.testing.assert_allclose(lse[b], r_lse, atol=2e-2, rtol=1e-3)


# ---------------------------------------------------------------------------
# Tensor-core per-head GEMMs: batch sizes that are not multiples of the tile and
# batches spanning several N tiles
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B", [1, 5, 40, 300])
def test_absorb_q_batch_shapes(mla, B):
    H, d_k, d_c, d_r = 16, 128, 512, 64
    q_nope = W.bf16_bits(W.normal(21, "abs_q", (B, H, d_k)))
    q_r = W.bf16_bits(W.normal(21, "abs_qr", (B, H, d_r)))
    w_uk = W.bf16_bits(W.normal(21, "abs_w", (H, d_k, d_c), std=1 / math.sqrt(512)))
    pos = (np.arange(B, dtype=np.int32) * 97) % 32768
    q_cat = mla.absorb_q(to_device(q_nope, "bf16"), to_device(q_r, "bf16"), torch.from_numpy(pos).cuda(),
                         to_device(w_uk, "bf16"))
    ref = O.absorb_q(W.widen(q_nope, "bf16"), W.widen(q_r, "bf16"), pos, W.widen(w_uk, "bf16"), 1e4)
    check_bf16(q_cat.float().cpu().numpy(), ref, f"q_cat B={B}")


@pytest.mark.parametrize("d_r", [0, 8, 128])
def test_absorb_q_rope_widths_and_far_positions(mla, d_r):
    # the query rotation for every pair count the tensor-core path takes, at positions
    # up to 2^20 (large angles: the fp32 turn reduction against the float64 oracle)
    B, H, d_k, d_c = 33, 8, 128, 512
    q_nope = W.bf16_bits(W.normal(23, "abs_q", (B, H, d_k)))
    q_r = W.bf16_bits(W.normal(23, "abs_qr", (B, H, d_r)))
    w_uk = W.bf16_bits(W.normal(23, "abs_w", (H, d_k, d_c), std=1 / math.sqrt(512)))
    pos = np.concatenate([[0, 1, 2 ** 20 - 1, 2 ** 20], (np.arange(B - 4, dtype=np.int64) * 65537) % (2 ** 20)])
    pos = pos.astype(np.int32)
    q_cat = mla.absorb_q(to_device(q_nope, "bf16"), to_device(q_r, "bf16") if d_r else None,
                         torch.from_numpy(pos).cuda(), to_device(w_uk, "bf16"))
    ref = O.absorb_q(W.widen(q_nope, "bf16"), W.widen(q_r, "bf16"), pos, W.widen(w_uk, "bf16"), 1e4)
    got = q_cat.float().cpu().numpy()
    check_bf16(got, ref, f"q_cat d_r={d_r}")
    if d_r:
        # the rotated part alone: one bf16 rounding of the exact rotation
        np.testing.assert_allclose(got[..., d_c:], ref[..., d_c:], rtol=2 ** -8, atol=2e-3)


@pytest.mark.parametrize("B", [1, 5, 40, 300])
def test_out_up_batch_shapes(mla, B):
    H, d_c, d_v = 16, 512, 128
    o_lat = W.bf16_bits(W.normal(22, "oup_o", (B, H, d_c)))
    w_uv = W.bf16_bits(W.normal(22, "oup_w", (H, d_v, d_c), std=1 / math.sqrt(512)))
    o = mla.out_up(to_device(o_lat, "bf16"), to_device(w_uv, "bf16"))
    ref = O.out_up(W.widen(o_lat, "bf16"), W.widen(w_uv, "bf16"))
    check_bf16(o.float().cpu().numpy(), ref, f"o B={B}")


# ---------------------------------------------------------------------------
# A few long sequences: each is cut into many pieces (as many as there are runs
# for a single sequence), which the combine merges in groups and a second kernel
# merges across groups; every sequence against the oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("lens", [[20000], [30000, 100], [9000, 12000, 64, 7000], [16384] * 5, [65536]])
def test_decode_few_long_sequences_grouped_merge(mla, lens):
    o, lse, ro, rlse = _decode_direct(mla, lens, H=128, d_r=64, seed=50 + len(lens))
    for b in range(len(lens)):
        check_bf16(o[b], ro[b], f"few long sequences b={b} n={lens[b]}")
    np.testing.assert_allclose(lse, rlse, atol=2e-2, rtol=1e-3)
