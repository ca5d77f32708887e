"""GPU parity of the partial over a row range (mla_decode_attn_partial) and of the
log-sum-exp merge of partials (mla_decode_merge): the pieces of decode sharded by
sequence position (0539edu.com section 8), checked against the float64 oracle's
partials and its unsplit attention.  Tolerances as for every bf16 output:
max-abs <= 2e-2 and relative L2 <= 1e-2 (per row <= 5e-2)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import check_bf16, direct_decode_inputs, oracle_direct, upload_direct

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _ok(mla):
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"


def test_partials_of_three_ranges_merge_to_the_full_attention(mla):
    lens = np.array([4096, 300, 1, 777, 2000, 65], dtype=np.int32)
    q_bits, rows = direct_decode_inputs(41, lens, 128, 512, 64)
    q, cache = upload_direct(mla, q_bits, rows, 512, 64, int(lens.max()))
    rng = np.random.default_rng(3)
    # cut points at arbitrary (not block-aligned) rows; some ranges are empty
    c1 = np.array([rng.integers(0, n + 1) for n in lens], dtype=np.int32)
    c2 = np.array([rng.integers(a, n + 1) for a, n in zip(c1, lens)], dtype=np.int32)
    c1[2], c2[2] = 0, 1   # the one-row sequence: empty, the row, empty
    bounds = [(np.zeros_like(lens), c1), (c1, c2), (c2, lens)]
    o_parts = torch.empty((3, len(lens), 128, 512), dtype=torch.bfloat16, device="cuda")
    lse_parts = torch.empty((3, len(lens), 128), dtype=torch.float32, device="cuda")
    for s, (b0, b1) in enumerate(bounds):
        mla.decode_attn_partial(q, cache, torch.from_numpy(b0).cuda(), torch.from_numpy(b1).cuda(), SCALE,
                                out=o_parts[s], lse=lse_parts[s])
    _ok(mla)
    # each partial against the oracle's partial of its rows (log-sum-exp form)
    for s, (b0, b1) in enumerate(bounds):
        got_o = o_parts[s].float().cpu().numpy()
        got_l = lse_parts[s].cpu().numpy()
        for b in range(len(lens)):
            if b1[b] == b0[b]:
                assert np.all(got_o[b] == 0) and np.all(np.isneginf(got_l[b]))
                continue
            m, l, o_un = O.decode_partial(W.widen(q_bits[b], "bf16"), W.widen(rows[b][b0[b]:b1[b]], "bf16"), 512,
                                          SCALE)
            check_bf16(got_o[b], o_un / l[:, None], f"partial {s} of b={b} rows [{b0[b]}, {b1[b]})")
            np.testing.assert_allclose(got_l[b], m + np.log(l), atol=2e-2, rtol=1e-3)
    # the merge equals the attention over all rows
    o, lse = mla.decode_merge(o_parts, lse_parts)
    _ok(mla)
    ref_o, ref_lse = oracle_direct(q_bits, rows, 512, SCALE)
    check_bf16(o.float().cpu().numpy(), ref_o, "merged partials")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, atol=2e-2, rtol=1e-3)


def test_full_range_partial_is_the_decode_and_merging_it_alone_changes_nothing(mla):
    lens = np.array([4097, 128, 900], dtype=np.int32)
    q_bits, rows = direct_decode_inputs(42, lens, 128, 512, 64)
    q, cache = upload_direct(mla, q_bits, rows, 512, 64, int(lens.max()))
    seq_lens = torch.from_numpy(lens).cuda()
    o_ref, lse_ref = mla.decode_attn(q, cache, seq_lens, SCALE)
    o_p, lse_p = mla.decode_attn_partial(q, cache, torch.zeros_like(seq_lens), seq_lens, SCALE)
    o_m, lse_m = mla.decode_merge(o_p[None], lse_p[None])
    _ok(mla)
    # rows [0, n) are exactly the decode problem; a single partial merges with weight 1
    assert torch.equal(o_p.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse_p, lse_ref)
    assert torch.equal(o_m.view(torch.int16), o_ref.view(torch.int16))
    torch.testing.assert_close(lse_m, lse_ref, rtol=0, atol=2e-6)


def test_shards_of_four_ranks_on_one_gpu(mla):
    # the row shares four sequence-parallel ranks would hold, run one after another
    # on this GPU, gathered and merged by the host path's merge
    from head_latent_attention_29_b300.seqpar import SeqShardedDecode, library_attend, library_merge, shard_rows
    lens = np.array([4096, 1000, 64, 3333], dtype=np.int32)
    q_bits, rows = direct_decode_inputs(43, lens, 128, 512, 64)
    q, cache = upload_direct(mla, q_bits, rows, 512, 64, int(lens.max()))
    world = 4
    o_all = torch.empty((world, len(lens), 128, 512), dtype=torch.bfloat16, device="cuda")
    lse_all = torch.empty((world, len(lens), 128), dtype=torch.float32, device="cuda")
    for r in range(world):
        b0, b1 = shard_rows(lens, world, r)
        sd = SeqShardedDecode(len(lens), 128, 512, 1, 0,
                              attend=library_attend(cache, SCALE, torch.from_numpy(b0).cuda(),
                                                    torch.from_numpy(b1).cuda()),
                              merge=lambda o, l: (o[0], l[0]))
        o_all[r], lse_all[r] = sd.step(q, None)
    o, lse = library_merge()(o_all, lse_all)
    _ok(mla)
    ref_o, ref_lse = oracle_direct(q_bits, rows, 512, SCALE)
    check_bf16(o.float().cpu().numpy(), ref_o, "four shards merged")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, atol=2e-2, rtol=1e-3)


def test_merge_of_empty_partials_and_fp32_parts(mla):
    o_parts = torch.randn((2, 3, 4, 64), device="cuda")
    lse_parts = torch.full((2, 3, 4), -math.inf, device="cuda")
    lse_parts[1, 0] = 0.5   # row (0, h) has one non-empty partial
    o, lse = mla.decode_merge(o_parts, lse_parts)
    _ok(mla)
    assert torch.equal(o[0], o_parts[1, 0]) and torch.all(lse[0] == 0.5)
    assert torch.all(o[1:] == 0) and torch.all(torch.isneginf(lse[1:]))


def test_partial_range_outside_the_cache_is_recorded(mla):
    lens = np.array([100, 70], dtype=np.int32)
    q_bits, rows = direct_decode_inputs(44, lens, 128, 512, 64)
    q, cache = upload_direct(mla, q_bits, rows, 512, 64, 100)
    begin = torch.tensor([10, 50], dtype=torch.int32, device="cuda")
    end = torch.tensor([101, 40], dtype=torch.int32, device="cuda")   # past N_max; end before begin
    mla.decode_attn_partial(q, cache, begin, end, SCALE)
    st, word = mla.get_device_error()
    assert st == 6 and (word >> 8) == 2
