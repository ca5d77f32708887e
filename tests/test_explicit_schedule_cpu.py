"""A CPU model of the explicit-prefill attention kernel's schedule: the same work
mapping (heavy query tiles first), key-tile counts, causal limits, lazy maximum
(raised only past 2^8), bf16 rounding of the rebuilt K / V, the rotated query, P
and the output.  It must reproduce the float64 oracle within the bf16 tolerances,
and every tile the kernel loads must stay inside its tensor: a mistake in the
schedule shows here without a GPU.  It shares no code with the kernel."""
import math

import numpy as np
import pytest

from oracle import mla_oracle as O


def bf16(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def model(B, S, H, start, causal, seed=0, scale=1/math.sqrt(192), base=1e4, N_max=None):
    rng = np.random.default_rng(seed)
    P = start + S
    N_max = N_max or P
    d_c, d_r, dk = 512, 64, 128
    c_kv = bf16(rng.standard_normal((B, N_max, d_c)))
    k_r = bf16(rng.standard_normal((B, N_max, d_r)))
    q_nope = bf16(rng.standard_normal((B, S, H, dk)))
    q_r = bf16(rng.standard_normal((B, S, H, d_r)))
    w_uk = bf16(rng.standard_normal((H, dk, d_c)) / math.sqrt(512))
    w_uv = bf16(rng.standard_normal((H, dk, d_c)) / math.sqrt(512))
    # cache rows as the append kernel writes them (rotated key, bf16)
    k_rot = np.stack([bf16(O.rope(k_r[b], np.arange(N_max), base)) for b in range(B)])
    # (1) rebuilt K / V, bf16, [B][P][H][128]
    K = bf16(np.einsum("btc,hdc->bthd", c_kv[:, :P], w_uk))
    V = bf16(np.einsum("btc,hdc->bthd", c_kv[:, :P], w_uv))
    q_tiles = -(-S // 128)
    o = np.full((B, S, H, dk), np.nan)
    lse = np.full((B, S, H), np.nan)
    seen = set()
    for blk in range(B * H * q_tiles):
        qt = q_tiles - 1 - blk // (B * H)
        rem = blk % (B * H)
        b, h = rem // H, rem % H
        seen.add((b, h, qt))
        q0 = qt * 128
        q_last = start + min(q0 + 128, S) - 1
        n_keys = q_last + 1 if causal else P
        nkt = -(-n_keys // 128)
        # TMA coordinates: queries rows b*S+q0 .. +127 of [B*S]; keys rows b*P + j*128 of [B*P];
        # k_R rows j*128 .. of [N_max] for sequence b
        assert 0 <= b * S + q0 < B * S
        for j in range(nkt):
            assert 0 <= b * P + j * 128 < B * P and 0 <= j * 128 < N_max
        rows = np.arange(128)
        qi = q0 + rows
        qpos = start + np.minimum(qi, S - 1)
        limit = qpos if causal else np.full(128, P - 1)
        # query rows: rows past B*S read zeros, others the next rows of [B*S]
        flat = b * S + q0 + rows
        Qn = np.zeros((128, dk)); Qr = np.zeros((128, d_r))
        ok = flat < B * S
        fb, fi = flat[ok] // S, flat[ok] % S
        Qn[ok] = q_nope[fb, fi, h]
        Qr[ok] = q_r[fb, fi, h]
        Qr = np.stack([bf16(O.rope(Qr[i], start + qi[i], base)) for i in range(128)])
        Q = np.concatenate([Qn, Qr], 1)
        m_ref = np.zeros(128); l = np.zeros(128); Oacc = np.zeros((128, dk))
        for j in range(nkt):
            t = j * 128 + np.arange(128)
            kflat = b * P + t
            Kt = np.zeros((128, dk)); Vt = np.zeros((128, dk)); Kr = np.zeros((128, d_r))
            okk = kflat < B * P
            Kt[okk] = K[kflat[okk] // P, kflat[okk] % P, h]
            Vt[okk] = V[kflat[okk] // P, kflat[okk] % P, h]
            okr = t < N_max
            Kr[okr] = k_rot[b, t[okr]]
            s = Q @ np.concatenate([Kt, Kr], 1).T  # [128 q, 128 keys]
            mask = t[None, :] <= limit[:, None]
            mloc = np.where(mask, s, -np.inf).max(1) * scale * math.log2(math.e)
            alpha = np.ones(128)
            if j == 0:
                assert np.all(np.isfinite(mloc))
                m_ref = mloc.copy()
            else:
                up = mloc > m_ref + 8.0
                alpha[up] = np.exp2(m_ref[up] - mloc[up]); m_ref[up] = mloc[up]
            p = np.where(mask, np.exp2(s * scale * math.log2(math.e) - m_ref[:, None]), 0.0)
            p = bf16(p)
            Oacc = Oacc * alpha[:, None] + p @ Vt
            l = l * alpha + p.sum(1)
        for r in range(128):
            if qi[r] < S:
                o[b, qi[r], h] = bf16(Oacc[r] / l[r])
                lse[b, qi[r], h] = (m_ref[r] + math.log2(l[r])) * math.log(2)
    assert len(seen) == B * H * q_tiles
    assert not np.isnan(o).any()
    # oracle
    ref_all, got_all = [], []
    for b in range(B):
        ro, rl = O.prefill_explicit_rows(q_nope[b], q_r[b], c_kv[b, :P], k_r[b, :P], w_uk, w_uv, scale, base,
                                         range(S), causal, start)
        ref_all.append(ro); got_all.append(o[b])
        np.testing.assert_allclose(lse[b], rl, atol=2e-2, rtol=1e-3)
    ref = np.stack(ref_all); got = np.stack(got_all)
    mx = np.abs(got - ref).max(); rl2 = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert mx <= 2e-2 and rl2 <= 1e-2



@pytest.mark.parametrize("B,S,H,start,causal,extra", [(1, 300, 2, 0, True, 0), (2, 200, 1, 37, True, 0),
                                                      (1, 130, 1, 5, False, 0), (1, 257, 1, 130, True, 0),
                                                      (1, 100, 1, 20, True, 300)])
def test_explicit_prefill_schedule_reproduces_oracle(B, S, H, start, causal, extra):
    model(B, S, H, start, causal, N_max=start + S + extra if extra else None)


@pytest.mark.parametrize("B,start,S,H", [(1, 0, 300, 2), (2, 37, 200, 4), (4, 0, 8192, 128), (1, 130, 257, 6)])
def test_kv_rebuild_grid_writes_every_output_once(B, start, S, H):
    # kvup grid (H feature tiles: H / 2 for K, H / 2 for V; ceil(P / 128) token
    # tiles; B sequences): every (sequence, token < P, feature) of both buffers is
    # written by exactly one CTA, and every weight tile lies inside W_UK / W_UV
    P = start + S
    feats = H * 128
    count = np.zeros((2, B, -(-P // 128) * 128, feats // 256), dtype=np.int64)
    for ft in range(H):
        is_v = ft >= H // 2
        f0 = (ft - H // 2 if is_v else ft) * 256
        assert f0 % 256 == 0 and f0 + 256 <= feats          # the 256-row weight box stays inside
        for ty in range(-(-P // 128)):
            t0 = ty * 128
            count[int(is_v), :, t0:t0 + 128, f0 // 256] += 1  # all B sequences (grid z)
    assert np.all(count[:, :, :P] == 1)
