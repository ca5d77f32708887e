"""Pins for the float64 oracle: checks against facts fixed by the pages and by
mathematics, never against the oracle's own formulas retyped.

Each test targets a mistake the oracle could plausibly contain (a dropped RoPE
term, a transposed up-projection, a wrong sign in the rotation, a missing max
subtraction, a wrong LSE merge, an off-by-one in the causal mask)."""
import json
import math
import os

import numpy as np
import pytest

import mla_workloads as W
from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------
def test_rope_position_zero_is_identity():
    x = _rand((5, 8), 1)
    np.testing.assert_array_equal(O.rope(x, np.zeros(5), 10000.0), x)


def test_rope_closed_form_values():
    # d_r = 2: theta_0 = 1, so position p rotates by exactly p radians
    np.testing.assert_allclose(O.rope(np.array([1.0, 0.0]), 1, 10000.0), [math.cos(1), math.sin(1)], atol=1e-15)
    np.testing.assert_allclose(O.rope(np.array([0.0, 1.0]), 1, 10000.0), [-math.sin(1), math.cos(1)], atol=1e-15)
    # d_r = 4, base 100: theta_1 = 100^(-1/2) = 0.1, so position 10 rotates pair 1 by 1 rad
    got = O.rope(np.array([0.0, 0.0, 1.0, 0.0]), 10, 100.0)
    np.testing.assert_allclose(got, [0.0, 0.0, math.cos(1), math.sin(1)], atol=1e-15)
    # pair 0 of the same vector at position 10 rotates by 10 rad
    got = O.rope(np.array([1.0, 0.0, 0.0, 0.0]), 10, 100.0)
    np.testing.assert_allclose(got, [math.cos(10), math.sin(10), 0.0, 0.0], atol=1e-14)


def test_rope_preserves_norm_and_depends_on_relative_position():
    d_r = 64
    q, k = _rand(d_r, 2), _rand(d_r, 3)
    for m, n in [(0, 5), (17, 4000), (32767, 3), (1234, 1234)]:
        lhs = O.rope(q, m, 10000.0) @ O.rope(k, n, 10000.0)
        rhs = q @ O.rope(k, n - m, 10000.0)
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(lhs))
        assert abs(np.linalg.norm(O.rope(q, m, 10000.0)) - np.linalg.norm(q)) < 1e-12


# ---------------------------------------------------------------------------
# Softmax
# ---------------------------------------------------------------------------
def test_softmax_rows_sum_to_one_and_match_naive():
    s = _rand((7, 300), 4, 3.0)
    p = O.softmax_rows(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    naive = np.exp(s) / np.exp(s).sum(-1, keepdims=True)
    np.testing.assert_allclose(p, naive, rtol=1e-12)
    # shift invariance: the max subtraction keeps huge scores finite
    p_big = O.softmax_rows(s + 1000.0)
    assert np.all(np.isfinite(p_big))
    np.testing.assert_allclose(p_big, p, rtol=1e-10)
    np.testing.assert_allclose(O.logsumexp_rows(s + 1000.0), O.logsumexp_rows(s) + 1000.0, rtol=1e-14)


# ---------------------------------------------------------------------------
# Absorbed vs explicit (the identity of 0539edu.com section 3.1)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,d_c,d_r,d_k,d_v,N", [(4, 32, 8, 16, 16, 64), (3, 24, 0, 8, 12, 9), (2, 16, 4, 8, 8, 1)])
def test_absorbed_equals_explicit(H, d_c, d_r, d_k, d_v, N):
    rng = np.random.default_rng(H * 100 + N)
    q_nope, q_r = rng.standard_normal((H, d_k)), rng.standard_normal((H, d_r))
    c_kv, k_r = rng.standard_normal((N, d_c)), rng.standard_normal((N, d_r))
    w_uk = rng.standard_normal((H, d_k, d_c)) / math.sqrt(d_c)
    w_uv = rng.standard_normal((H, d_v, d_c)) / math.sqrt(d_c)
    scale = 1.0 / math.sqrt(d_k + d_r)
    pos = np.arange(N)
    o_abs, _, _ = O.decode_absorbed_from_parts(q_nope, q_r, N - 1, c_kv, k_r, pos, w_uk, w_uv, scale, 10000.0)
    o_exp = O.decode_explicit(q_nope, q_r, N - 1, c_kv, k_r, pos, w_uk, w_uv, scale, 10000.0)
    rel = np.linalg.norm(o_abs - o_exp) / np.linalg.norm(o_exp)
    assert rel < 1e-12


def test_tiny_workload_from_hidden_states_absorbed_equals_explicit():
    cfg = W.WORKLOADS["tiny_fp32"]
    m = W.hidden_model(cfg, seed=0)
    H, d_k, d_r = cfg["H"], cfg["d_k"], cfg["d_r"]
    h = W.widen(m["h"], "f32")[0]                                      # [N, d_model]
    c_kv, k_r, q_nope_all, q_r_all = O.project_from_hidden(h, m["w_dkv"], m["w_kr"], m["w_uq"], H, d_k, d_r)
    N = cfg["N"]
    pos = np.arange(N)
    o_abs, _, _ = O.decode_absorbed_from_parts(q_nope_all[N - 1], q_r_all[N - 1], N - 1, c_kv, k_r, pos,
                                               m["w_uk"], m["w_uv"], cfg["scale"], cfg["rope_base"])
    o_exp = O.decode_explicit(q_nope_all[N - 1], q_r_all[N - 1], N - 1, c_kv, k_r, pos,
                              m["w_uk"], m["w_uv"], cfg["scale"], cfg["rope_base"])
    assert np.linalg.norm(o_abs - o_exp) / np.linalg.norm(o_exp) < 1e-12
    # the projection split: q per head is d_k no-position columns then d_r rotated columns
    q_full = (h[N - 1] @ m["w_uq"].astype(np.float64)).reshape(H, d_k + d_r)
    np.testing.assert_allclose(q_nope_all[N - 1], q_full[:, :d_k], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(q_r_all[N - 1], q_full[:, d_k:], rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# The projections from hidden states, pinned without their own formula
# (0539edu.com section 2.2: c_KV = h W_DKV; hotelren.com section 6.2: one RoPE
# key k_R = h W_KR for all heads; per head d_k no-position query columns, then d_r)
# ---------------------------------------------------------------------------
def test_project_from_hidden_one_hot_rows_select_weight_rows():
    rng = np.random.default_rng(7)
    d_model, d_c, H, d_k, d_r = 6, 5, 3, 4, 2
    w_dkv = rng.standard_normal((d_model, d_c))
    w_kr = rng.standard_normal((d_model, d_r))
    w_uq = rng.standard_normal((d_model, H * (d_k + d_r)))
    # row i of h is the unit vector e_i: every projection returns row i of its weight
    c_kv, k_r, q_nope, q_r = O.project_from_hidden(np.eye(d_model), w_dkv, w_kr, w_uq, H, d_k, d_r)
    assert np.array_equal(c_kv, w_dkv) and np.array_equal(k_r, w_kr)
    for i in range(d_model):
        for hh in range(H):
            base_col = hh * (d_k + d_r)
            assert np.array_equal(q_nope[i, hh], w_uq[i, base_col:base_col + d_k])
            assert np.array_equal(q_r[i, hh], w_uq[i, base_col + d_k:base_col + d_k + d_r])


def test_project_from_hidden_head_major_split_order():
    # W_UQ built so that head hh's block holds (hh + 1) in its d_k no-position
    # columns and -(hh + 1) in its d_r position columns: a component-major layout
    # or swapped q_nope / q_R columns gives different constants.
    d_model, H, d_k, d_r = 3, 4, 5, 2
    w_uq = np.zeros((d_model, H * (d_k + d_r)))
    for hh in range(H):
        w_uq[0, hh * (d_k + d_r):hh * (d_k + d_r) + d_k] = hh + 1
        w_uq[0, hh * (d_k + d_r) + d_k:(hh + 1) * (d_k + d_r)] = -(hh + 1)
    h = np.array([[1.0, 0.0, 0.0], [2.0, 5.0, -1.0]])  # only column 0 of h reaches W_UQ's row 0
    _, _, q_nope, q_r = O.project_from_hidden(h, np.zeros((d_model, 1)), np.zeros((d_model, d_r)), w_uq,
                                              H, d_k, d_r)
    for n, scale in ((0, 1.0), (1, 2.0)):
        for hh in range(H):
            assert np.all(q_nope[n, hh] == scale * (hh + 1))
            assert np.all(q_r[n, hh] == -scale * (hh + 1))


def test_project_from_hidden_matches_scalar_loops_two_heads():
    rng = np.random.default_rng(11)
    n, d_model, d_c, H, d_k, d_r = 3, 4, 3, 2, 3, 2
    h = rng.standard_normal((n, d_model))
    w_dkv = rng.standard_normal((d_model, d_c))
    w_kr = rng.standard_normal((d_model, d_r))
    w_uq = rng.standard_normal((d_model, H * (d_k + d_r)))
    c_kv, k_r, q_nope, q_r = O.project_from_hidden(h, w_dkv, w_kr, w_uq, H, d_k, d_r)
    for t in range(n):
        for j in range(d_c):
            assert abs(c_kv[t, j] - sum(h[t, m] * w_dkv[m, j] for m in range(d_model))) < 1e-12
        for j in range(d_r):
            assert abs(k_r[t, j] - sum(h[t, m] * w_kr[m, j] for m in range(d_model))) < 1e-12
        for hh in range(H):
            for j in range(d_k + d_r):
                col = hh * (d_k + d_r) + j
                want = sum(h[t, m] * w_uq[m, col] for m in range(d_model))
                got = q_nope[t, hh, j] if j < d_k else q_r[t, hh, j - d_k]
                assert abs(got - want) < 1e-12


# ---------------------------------------------------------------------------
# Brute force with scalar loops on tiny shapes
# ---------------------------------------------------------------------------
def _brute_force(q_nope, q_r, q_pos, c_kv, k_r, w_uk, w_uv, scale, base):
    H, d_k = len(q_nope), len(q_nope[0])
    d_r = len(q_r[0])
    N, d_c = len(c_kv), len(c_kv[0])
    d_v = len(w_uv[0])

    def rot(x, p):
        out = list(x)
        for i in range(len(x) // 2):
            ang = p * base ** (-2.0 * i / len(x))
            a, b = x[2 * i], x[2 * i + 1]
            out[2 * i] = a * math.cos(ang) - b * math.sin(ang)
            out[2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
        return out

    o = []
    for h in range(H):
        qr = rot(q_r[h], q_pos)
        scores = []
        for t in range(N):
            kr = rot(k_r[t], t)
            s = 0.0
            for d in range(d_k):
                k_d = sum(c_kv[t][c] * w_uk[h][d][c] for c in range(d_c))
                s += q_nope[h][d] * k_d
            for d in range(d_r):
                s += qr[d] * kr[d]
            scores.append(s * scale)
        mx = max(scores)
        e = [math.exp(s - mx) for s in scores]
        z = sum(e)
        row = []
        for d in range(d_v):
            acc = 0.0
            for t in range(N):
                v_td = sum(c_kv[t][c] * w_uv[h][d][c] for c in range(d_c))
                acc += e[t] / z * v_td
            row.append(acc)
        o.append(row)
    return np.array(o)


@pytest.mark.parametrize("H,d_c,d_r,d_k,d_v,N", [(2, 6, 4, 3, 2, 5), (3, 4, 2, 2, 3, 7), (1, 5, 0, 4, 4, 3)])
def test_brute_force_agrees_with_both_forms(H, d_c, d_r, d_k, d_v, N):
    rng = np.random.default_rng(7 + N)
    q_nope, q_r = rng.standard_normal((H, d_k)), rng.standard_normal((H, d_r))
    c_kv, k_r = rng.standard_normal((N, d_c)), rng.standard_normal((N, d_r))
    w_uk, w_uv = rng.standard_normal((H, d_k, d_c)), rng.standard_normal((H, d_v, d_c))
    scale = 0.37
    ref = _brute_force(q_nope.tolist(), q_r.tolist(), N - 1, c_kv.tolist(), k_r.tolist(),
                       w_uk.tolist(), w_uv.tolist(), scale, 50.0)
    pos = np.arange(N)
    o_abs, _, _ = O.decode_absorbed_from_parts(q_nope, q_r, N - 1, c_kv, k_r, pos, w_uk, w_uv, scale, 50.0)
    o_exp = O.decode_explicit(q_nope, q_r, N - 1, c_kv, k_r, pos, w_uk, w_uv, scale, 50.0)
    np.testing.assert_allclose(o_abs, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(o_exp, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Special cases with closed forms
# ---------------------------------------------------------------------------
def test_single_token_returns_its_latent():
    rng = np.random.default_rng(11)
    q_cat = rng.standard_normal((4, 40))
    rows = rng.standard_normal((1, 40))
    o_lat, lse = O.decode_absorbed(q_cat, rows, 32, 0.3)
    np.testing.assert_array_equal(o_lat, np.broadcast_to(rows[0, :32], (4, 32)))
    np.testing.assert_allclose(lse, 0.3 * q_cat @ rows[0], rtol=1e-15)


def test_zero_query_gives_uniform_weights():
    rows = _rand((50, 40), 12)
    o_lat, lse = O.decode_absorbed(np.zeros((3, 40)), rows, 32, 0.5)
    np.testing.assert_allclose(o_lat, np.broadcast_to(rows[:, :32].mean(0), (3, 32)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(50.0), rtol=1e-15)


def test_identical_rows_return_that_row():
    row = _rand(40, 13)
    rows = np.tile(row, (33, 1))
    o_lat, _ = O.decode_absorbed(_rand((5, 40), 14, 4.0), rows, 32, 1.0)
    np.testing.assert_allclose(o_lat, np.broadcast_to(row[:32], (5, 32)), rtol=1e-13)


def test_one_hot_scores_select_the_peaked_token():
    # a query aligned with one cached row and a large scale puts all weight there
    rows = np.eye(40)[:20] * 1.0
    q = np.zeros((1, 40))
    q[0, 7] = 1.0
    o_lat, _ = O.decode_absorbed(q, rows, 32, 200.0)
    expect = np.zeros(32)
    expect[7] = 1.0
    np.testing.assert_allclose(o_lat[0], expect, atol=1e-80)


def test_rope_key_term_contributes():
    # two tokens whose latents are equal differ only through the rotated key;
    # dropping the RoPE term would give equal weights 0.5 / 0.5
    rng = np.random.default_rng(15)
    c_kv = np.tile(rng.standard_normal((1, 8)), (2, 1))
    k_r = rng.standard_normal((2, 4))
    rows = O.cache_rows(c_kv, k_r, np.arange(2), 10000.0)
    q_cat = np.concatenate([np.zeros((1, 8)), rng.standard_normal((1, 4))], axis=1)
    s = q_cat @ rows.T
    assert abs(s[0, 0] - s[0, 1]) > 1e-3
    np.testing.assert_array_equal(rows[:, :8], c_kv)


# ---------------------------------------------------------------------------
# Split-KV partials: the merge over any partition equals the unsplit result
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cuts", [[10], [1, 2, 3], [0, 99], [33, 34, 35, 70]])
def test_lse_merge_is_partition_invariant(cuts):
    rng = np.random.default_rng(16)
    q_cat, rows = rng.standard_normal((6, 40)), rng.standard_normal((100, 40))
    ref_o, ref_lse = O.decode_absorbed(q_cat, rows, 32, 0.2)
    edges = [0] + [c for c in cuts if 0 < c < 100] + [100]
    parts = [O.decode_partial(q_cat, rows[a:b], 32, 0.2) for a, b in zip(edges[:-1], edges[1:])]
    o, lse = O.lse_merge(parts)
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)


# ---------------------------------------------------------------------------
# Gate
# ---------------------------------------------------------------------------
def test_gate_with_zero_weights_halves_output():
    o = _rand((3, 10), 17)
    np.testing.assert_array_equal(O.gate(_rand((3, 6), 18), np.zeros((6, 10)), o), 0.5 * o)


def test_gate_closed_form_channels():
    # h = [1], W_g = [[0, ln 3, -ln 3, 100]] gives gates 1/2, 3/4, 1/4, ~1
    g = O.gate(np.array([[1.0]]), np.array([[0.0, math.log(3.0), -math.log(3.0), 100.0]]), np.ones((1, 4)))
    np.testing.assert_allclose(g[0], [0.5, 0.75, 0.25, 1.0], rtol=1e-15)


# ---------------------------------------------------------------------------
# Causal prefill: the per-row prefix form equals a masked full-matrix softmax
# ---------------------------------------------------------------------------
def test_prefill_rows_match_masked_full_softmax():
    rng = np.random.default_rng(19)
    S, H, R, d_c = 12, 3, 20, 16
    q_cat, rows = rng.standard_normal((S, H, R)), rng.standard_normal((S, R))
    scale = 0.4
    o_rows, lse_rows = O.prefill_absorbed_rows(q_cat, rows, d_c, scale, range(S))
    for h in range(H):
        s = scale * q_cat[:, h, :] @ rows.T
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        np.testing.assert_allclose(o_rows[:, h, :], p @ rows[:, :d_c], rtol=1e-12, atol=1e-14)
    # the first query sees only itself
    np.testing.assert_allclose(o_rows[0], np.broadcast_to(rows[0, :d_c], (H, d_c)), rtol=1e-15)


def test_prefill_in_chunks_equals_one_pass():
    # A prompt processed as two chunks (the second starting at position S1 over the
    # rows of both) gives the rows of one pass: the chunk offset is only a shift of
    # the causal limit.  The non-causal chunk reads every row up to its own end.
    rng = np.random.default_rng(23)
    S1, S2, H, R, d_c = 7, 9, 2, 24, 16
    q_cat, rows = rng.standard_normal((S1 + S2, H, R)), rng.standard_normal((S1 + S2, R))
    scale = 0.3
    whole_o, whole_l = O.prefill_absorbed_rows(q_cat, rows, d_c, scale, range(S1 + S2))
    o1, l1 = O.prefill_absorbed_rows(q_cat[:S1], rows[:S1], d_c, scale, range(S1))
    o2, l2 = O.prefill_absorbed_rows(q_cat[S1:], rows, d_c, scale, range(S2), start=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), whole_o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(np.concatenate([l1, l2]), whole_l, rtol=1e-13)
    # non-causal second chunk: every query reads all S1 + S2 rows (as the last query does)
    o_nc, l_nc = O.prefill_absorbed_rows(q_cat[S1:], rows, d_c, scale, range(S2), causal=False, start=S1)
    for i in range(S2):
        o_ref, l_ref = O.decode_absorbed(q_cat[S1 + i], rows, d_c, scale)
        np.testing.assert_allclose(o_nc[i], o_ref, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(l_nc[i], l_ref, rtol=1e-13)
    # a wrong offset would be visible: the first query of the chunk must see S1 + 1 rows
    o_wrong, _ = O.decode_absorbed(q_cat[S1], rows[:1], d_c, scale)
    assert np.max(np.abs(o2[0] - o_wrong)) > 1e-3


# ---------------------------------------------------------------------------
# Magnitudes of the headline workload: unit-variance scores
# ---------------------------------------------------------------------------
def test_headline_scores_have_unit_variance():
    cfg = W.WORKLOADS["decode_h128_b32_n4096"]
    rng = np.random.default_rng(20)
    H, d_k, d_c, d_r = cfg["H"], cfg["d_k"], cfg["d_c"], cfg["d_r"]
    w_uk = rng.standard_normal((H, d_k, d_c)) * cfg["w_std"]
    q_cat = O.absorb_q(rng.standard_normal((H, d_k)), rng.standard_normal((H, d_r)), 300, w_uk, 10000.0)
    rows = O.cache_rows(rng.standard_normal((256, d_c)), rng.standard_normal((256, d_r)), np.arange(256), 10000.0)
    s = cfg["scale"] * q_cat @ rows.T
    assert abs(s.var() - 1.0) < 0.05


# ---------------------------------------------------------------------------
# Cache-size values printed on the pages
# ---------------------------------------------------------------------------
def _golden():
    with open(os.path.join(GOLDEN, "cache_bytes.json")) as f:
        return {e["id"]: e for e in json.load(f)["entries"]}


def test_cache_size_values_printed_on_the_pages():
    g = _golden()
    KiB, MiB, GiB = 1024, 1024 ** 2, 1024 ** 3
    e = g["mha_elements_per_token_layer"]
    assert O.mha_kv_elements(e["inputs"]["h"], e["inputs"]["d"]) == e["printed"]
    e = g["mha_bytes_per_token_layer_fp16"]
    assert O.mha_kv_elements(128, 128) * 2 / KiB == e["printed"]
    e = g["mha_bytes_per_token_60_layers"]
    assert O.kv_cache_bytes(60, 128, 128, 1, 1, 2) / MiB == e["printed"]
    e = g["mha_total_32k_ctx_32_seqs"]
    assert round(3.75e6 * 32768 * 32 / 1e12, 1) == e["printed"]
    e = g["mla_ratio_deepseek_v2"]
    assert O.compression_ratio(128, 128, 128, 512) == e["printed"]
    e = g["mla_ratio_dc_1024"]
    assert O.compression_ratio(128, 128, 128, 1024) == e["printed"]
    e = g["mla_latent_bytes_per_token_layer"]
    assert O.latent_row_elements(512, 0) * 2 / KiB == e["printed"]
    e = g["mla_latent_total_60L_32k_b16"]
    assert O.latent_row_elements(512, 0) * 2 * 60 * 32768 * 16 / GiB == e["printed"]
    e = g["mha_layer_bytes_8h_4096_b32"]
    assert O.kv_cache_bytes(1, 8, 128, 4096, 32, 2) == e["printed"]
    e = g["mha_layer_gb_8h_4096_b32"]
    assert O.kv_cache_bytes(1, 8, 128, 4096, 32, 2) / GiB == e["printed"]
    e = g["mha_50_layers_gb"]
    assert O.kv_cache_bytes(50, 8, 128, 4096, 32, 2) / GiB == e["printed"]
    e = g["latent_256_fraction"]
    assert 256 / O.mha_kv_elements(8, 128) == e["printed"]
    e = g["latent_256_total_gb"]
    assert round(O.kv_cache_bytes(50, 8, 128, 4096, 32, 2) / GiB * 256 / O.mha_kv_elements(8, 128), 1) == e["printed"]
    e = g["mla_row_elements"]
    assert O.latent_row_elements(512, 64) == e["printed"]
    e = g["compression_28_to_32"]
    lo, hi = e["printed"]
    assert int(128 * 128 / O.latent_row_elements(512, 64)) == lo
    assert 128 * 128 / O.latent_row_elements(512, 0) == hi
    e = g["mla_per_token_table"]
    assert round(O.latent_row_elements(512, 64) * 2 * 60 / MiB, 2) == e["printed"]


# ---------------------------------------------------------------------------
# The seeded inputs are reproducible and shaped as the workloads state
# ---------------------------------------------------------------------------
def test_workload_draws_are_reproducible():
    cfg = W.WORKLOADS["ragged_h128_b64_n1k_32k"]
    a = W.seq_lens(cfg, 0)
    assert a.shape == (64,) and a.min() >= 1024 and a.max() <= 32768
    np.testing.assert_array_equal(a, W.seq_lens(cfg, 0))
    c1, k1 = W.latent_rows(cfg, 0, 5, 10)
    c2, k2 = W.latent_rows(cfg, 0, 5, 10)
    np.testing.assert_array_equal(c1, c2)
    assert c1.shape == (10, 512) and k1.shape == (10, 64)
    # a prefix draw is the prefix of a longer draw of the same sequence
    c3, _ = W.latent_rows(cfg, 0, 5, 20)
    np.testing.assert_array_equal(c3[:10], c1)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], dtype=np.float32)
    y = W.bf16_to_f32(W.bf16_bits(x))
    np.testing.assert_array_equal(y[:4], np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5], dtype=np.float32))
    assert abs(y[4] - 3.0e38) / 3.0e38 < 2 ** -8


# ---------------------------------------------------------------------------
# RMSNorm on the compressed latent and cache rows from hidden states
# ---------------------------------------------------------------------------
def test_rms_norm_matches_the_library_routine():
    # torch's own RMSNorm (CPU, float64) with a non-unit gain: a dropped gain, a
    # sum in place of the mean or eps outside the square root each fail here
    import torch
    x = _rand((7, 48), 31)
    g = 1.0 + _rand(48, 32, 0.3)
    for eps in (0.0, 1e-6, 0.5):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (48,), weight=torch.from_numpy(g), eps=eps).numpy()
        np.testing.assert_allclose(O.rms_norm(x, g, eps), ref, rtol=1e-13, atol=1e-14)


def test_rms_norm_closed_forms():
    # a constant vector c (any width) has mean square c^2: RMSNorm gives
    # gamma * c / sqrt(c^2 + eps), so gamma * sign(c) at eps = 0
    g = np.array([1.0, 2.0, -0.5, 3.0])
    np.testing.assert_allclose(O.rms_norm(np.full(4, -3.0), g, 0.0), -g, rtol=1e-15)
    np.testing.assert_allclose(O.rms_norm(np.full(4, 2.0), g, 5.0), g * 2.0 / 3.0, rtol=1e-15)
    # x = (3, 4): mean square 12.5
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), np.ones(2), 0.0),
                               np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    # unit gain, eps = 0: the output's mean square is exactly 1 and the map is
    # invariant to a positive rescale of its input
    x = _rand((3, 512), 33)
    y = O.rms_norm(x, np.ones(512), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.rms_norm(17.0 * x, np.ones(512), 0.0), y, rtol=1e-13)


def test_kv_down_rows_brute_force():
    # tiny shapes, every sum written out as a loop, the rotation as a 2 x 2 matrix
    rng = np.random.default_rng(34)
    n, dm, d_c, d_r, base, eps = 3, 6, 4, 4, 100.0, 1e-3
    h = rng.standard_normal((n, dm))
    w_dkv = rng.standard_normal((dm, d_c))
    w_kr = rng.standard_normal((dm, d_r))
    g = 1.0 + 0.2 * rng.standard_normal(d_c)
    pos = np.array([0, 5, 1234])
    got = O.kv_down_rows(h, w_dkv, w_kr, g, eps, pos, base)
    assert got.shape == (n, d_c + d_r)
    for t in range(n):
        c = [sum(h[t, i] * w_dkv[i, j] for i in range(dm)) for j in range(d_c)]
        ms = sum(v * v for v in c) / d_c
        for j in range(d_c):
            assert got[t, j] == pytest.approx(c[j] / math.sqrt(ms + eps) * g[j], rel=1e-12)
        k = [sum(h[t, i] * w_kr[i, j] for i in range(dm)) for j in range(d_r)]
        for p in range(d_r // 2):
            ang = pos[t] * base ** (-2.0 * p / d_r)
            rot = np.array([[math.cos(ang), -math.sin(ang)], [math.sin(ang), math.cos(ang)]])
            want = rot @ np.array([k[2 * p], k[2 * p + 1]])
            np.testing.assert_allclose(got[t, d_c + 2 * p:d_c + 2 * p + 2], want, rtol=1e-11, atol=1e-12)


def test_kv_down_rows_invariants():
    # at position 0 the key is the plain projection; at any position every rotated
    # pair keeps its length; with a unit gain the latent part has unit mean square
    cfg = W.WORKLOADS["kvdown_b32_d7168"]
    h, w_dkv, w_kr, _ = W.kv_down_inputs(dict(cfg, d_model=256), seed=3, T=5)
    rows0 = O.kv_down_rows(h, w_dkv, w_kr, np.ones(512), 0.0, np.zeros(5), 1e4)
    np.testing.assert_allclose(rows0[:, 512:], h.astype(np.float64) @ w_kr.astype(np.float64), rtol=1e-12)
    np.testing.assert_allclose(np.mean(rows0[:, :512] ** 2, axis=-1), 1.0, rtol=1e-13)
    rows = O.kv_down_rows(h, w_dkv, w_kr, np.ones(512), 0.0, np.arange(5) * 1000 + 7, 1e4)
    pair = lambda r: np.hypot(r[:, 512::2], r[:, 513::2])
    np.testing.assert_allclose(pair(rows), pair(rows0), rtol=1e-12)
    assert not np.allclose(rows[:, 512:], rows0[:, 512:])
    # no positional key (d_r = 0): the row is the normalised latent alone
    r = O.kv_down_rows(h, w_dkv, np.zeros((256, 0)), np.ones(512), 0.0, np.zeros(5), 1e4)
    assert r.shape == (5, 512)


# ---------------------------------------------------------------------------
# Explicit (non-absorbed) prefill
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal,start", [(True, 0), (True, 5), (False, 3)])
def test_explicit_prefill_equals_absorbed(causal, start):
    # the absorption identities (0539edu.com section 3.1) make the two forms equal:
    # a transposed W_UK / W_UV, a RoPE at the wrong position or a wrong causal
    # limit in either would break it
    rng = np.random.default_rng(41 + start)
    S, H, d_c, d_r, d_k, d_v, base, scale = 6, 3, 16, 4, 8, 5, 100.0, 0.3
    n = start + S
    c_kv, k_r = rng.standard_normal((n, d_c)), rng.standard_normal((n, d_r))
    q_nope, q_r = rng.standard_normal((S, H, d_k)), rng.standard_normal((S, H, d_r))
    w_uk, w_uv = rng.standard_normal((H, d_k, d_c)) * 0.3, rng.standard_normal((H, d_v, d_c)) * 0.3
    o_ex, lse_ex = O.prefill_explicit_rows(q_nope, q_r, c_kv, k_r, w_uk, w_uv, scale, base, range(S), causal, start)
    rows = O.cache_rows(c_kv, k_r, np.arange(n), base)
    q_cat = np.stack([O.absorb_q(q_nope[i], q_r[i], start + i, w_uk, base) for i in range(S)])
    o_lat, lse_ab = O.prefill_absorbed_rows(q_cat, rows, d_c, scale, range(S), causal, start)
    np.testing.assert_allclose(o_ex, O.out_up(o_lat, w_uv), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse_ex, lse_ab, rtol=1e-12)


def test_explicit_prefill_brute_force():
    # one head, every score and weight written out as loops
    rng = np.random.default_rng(47)
    S, d_c, d_r, d_k, d_v, base, scale = 4, 3, 2, 2, 2, 10.0, 0.7
    c_kv, k_r = rng.standard_normal((S, d_c)), rng.standard_normal((S, d_r))
    q_nope, q_r = rng.standard_normal((S, 1, d_k)), rng.standard_normal((S, 1, d_r))
    w_uk, w_uv = rng.standard_normal((1, d_k, d_c)), rng.standard_normal((1, d_v, d_c))
    o, lse = O.prefill_explicit_rows(q_nope, q_r, c_kv, k_r, w_uk, w_uv, scale, base, range(S))

    def rot(x, p):  # d_r = 2: one pair, angle p * base^0 = p
        return [x[0] * math.cos(p) - x[1] * math.sin(p), x[0] * math.sin(p) + x[1] * math.cos(p)]

    for i in range(S):
        qr = rot(q_r[i, 0], i)
        scores = []
        for t in range(i + 1):
            k = [sum(c_kv[t, c] * w_uk[0, d, c] for c in range(d_c)) for d in range(d_k)]
            kr = rot(k_r[t], t)
            scores.append(scale * (sum(q_nope[i, 0, d] * k[d] for d in range(d_k)) + qr[0] * kr[0] + qr[1] * kr[1]))
        z = sum(math.exp(x) for x in scores)
        for d in range(d_v):
            want = sum(math.exp(scores[t]) / z * sum(c_kv[t, c] * w_uv[0, d, c] for c in range(d_c))
                       for t in range(i + 1))
            assert o[i, 0, d] == pytest.approx(want, rel=1e-11, abs=1e-13)
        assert lse[i, 0] == pytest.approx(math.log(z), rel=1e-12)
    # the first query attends only to token 0: its value row exactly
    np.testing.assert_allclose(o[0, 0], w_uv[0] @ c_kv[0], rtol=1e-13)


def test_hidden_state_workload_recipe():
    # the kv_down inputs follow the recipe the design states: h ~ N(0,1), W_DKV and
    # W_KR ~ N(0, 1/d_model), a gain 1 + N(0, 0.1^2); seeded and reproducible
    cfg = W.WORKLOADS["kvdown_b32_d7168"]
    h, w_dkv, w_kr, g = W.kv_down_inputs(cfg, 0)
    assert h.shape == (32, 7168) and w_dkv.shape == (7168, 512) and w_kr.shape == (7168, 64) and g.shape == (512,)
    assert abs(h.std() - 1.0) < 0.01 and abs(h.mean()) < 0.01
    assert abs(w_dkv.std() * math.sqrt(7168) - 1.0) < 0.01 and abs(w_kr.std() * math.sqrt(7168) - 1.0) < 0.01
    assert abs(g.mean() - 1.0) < 0.02 and abs(g.std() - 0.1) < 0.01
    for a, b in zip((h, w_dkv, w_kr, g), W.kv_down_inputs(cfg, 0)):
        np.testing.assert_array_equal(a, b)
    assert not np.array_equal(h, W.kv_down_inputs(cfg, 1)[0])
    # the projection keeps unit scale: x = h W_DKV has unit variance per channel
    x = h.astype(np.float64) @ w_dkv.astype(np.float64)
    assert abs(x.std() - 1.0) < 0.05
