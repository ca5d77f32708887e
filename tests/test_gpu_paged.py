"""GPU parity of the paged latent cache: rows written through a block table land
where the table says, and decode attention over pages gives, bit for bit, what it
gives over a contiguous cache holding the same rows (and so matches the float64
oracle within the bf16 tolerances of the contiguous path).

The pages' caches are position-indexed buffers per sequence; the paged layout
splits each into 64-row pages of one pool so sequences grow without a
per-sequence preallocation.  Rows past a sequence's length in its last page, and
pages no sequence owns, hold NaN here, so any read of them would show."""
import math

import numpy as np
import pytest
import torch

import mla_workloads as W
from tests._cases import check_bf16, direct_decode_inputs, oracle_direct, to_device

pytestmark = pytest.mark.gpu

PR = 64  # rows per page
ERR_DEVICE_INDEX = 6


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _page_assignment(seed: int, lens, max_blocks: int, spare: int):
    """A shuffled page for every block each sequence uses (pool = used + spare pages);
    unused table entries point at pages that hold NaN."""
    rng = np.random.default_rng(seed)
    need = [-(-int(n) // PR) for n in lens]
    num_pages = sum(need) + spare
    perm = rng.permutation(num_pages)
    table = np.empty((len(lens), max_blocks), dtype=np.int32)
    k = 0
    for b, nb in enumerate(need):
        table[b, :nb] = perm[k:k + nb]
        k += nb
        table[b, nb:] = perm[-1] if spare else 0
    return table, num_pages


def _paged_and_contiguous(mla, lens, H, d_r, seed, spare=3, max_blocks=None):
    d_c = 512
    lens = np.asarray(lens, dtype=np.int32)
    max_blocks = max_blocks or max(1, -(-int(lens.max()) // PR))
    q_bits, rows = direct_decode_inputs(seed, lens, H, d_c, d_r)
    table, num_pages = _page_assignment(seed, lens, max_blocks, spare)
    paged = mla.PagedLatentCache(num_pages, len(lens), max_blocks, d_c, d_r,
                                 block_table=torch.from_numpy(table).cuda())
    paged.data.fill_(float("nan"))
    flat = mla.LatentCache(len(lens), max_blocks * PR, d_c, d_r, dtype=torch.bfloat16)
    flat.data.fill_(float("nan"))
    for b, r in enumerate(rows):
        n = r.shape[0]
        if n == 0:
            continue
        dev = to_device(r, "bf16")
        flat.data[b, :n, :d_c + d_r] = dev
        for j in range(-(-n // PR)):
            m = min(PR, n - j * PR)
            paged.data[table[b, j], :m, :d_c + d_r] = dev[j * PR:j * PR + m]
    return q_bits, rows, paged, flat, lens


@pytest.mark.parametrize("lens,H,d_r", [
    ([1, 63, 64, 65, 777, 4097], 128, 64),
    ([200, 0, 1, 129], 128, 64),
    ([1000] * 7, 64, 64),
    ([3000, 65, 900], 64, 0),
    ([513, 2], 16, 64),
    ([24000], 128, 64),           # one long sequence: the grouped merge
    ([12000, 9000, 70], 128, 64),
])
def test_paged_decode_bit_equal_to_contiguous(mla, lens, H, d_r):
    q_bits, rows, paged, flat, lens = _paged_and_contiguous(mla, lens, H, d_r, seed=len(lens) + H)
    q = to_device(q_bits, "bf16")
    seq_lens = torch.from_numpy(lens).cuda()
    scale = 1.0 / math.sqrt(128 + d_r)
    o_p, lse_p = mla.decode_attn_paged(q, paged, seq_lens, scale)
    o_f, lse_f = mla.decode_attn(q, flat, seq_lens, scale)
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"
    assert torch.equal(o_p.view(torch.int16), o_f.view(torch.int16))
    assert torch.equal(lse_p.view(torch.int32), lse_f.view(torch.int32))
    ref_o, ref_lse = oracle_direct(q_bits, rows, 512, scale)
    check_bf16(o_p.float().cpu().numpy(), ref_o, f"paged o_lat lens={list(lens)}")
    live = lens > 0
    np.testing.assert_allclose(lse_p.cpu().numpy()[live], ref_lse[live], atol=2e-2, rtol=1e-3)


def test_paged_decode_headline_shape_sampled(mla):
    # B = 32 sequences of 4096 tokens (the headline decode shape) over a shuffled
    # pool with spare pages; bit-equal to the contiguous cache, and a sample of
    # sequences against the oracle
    B, n, H, d_r = 32, 4096, 128, 64
    q_bits, rows, paged, flat, lens = _paged_and_contiguous(mla, [n] * B, H, d_r, seed=11, spare=8)
    q = to_device(q_bits, "bf16")
    seq_lens = torch.from_numpy(lens).cuda()
    scale = 1.0 / math.sqrt(128 + d_r)
    o_p, lse_p = mla.decode_attn_paged(q, paged, seq_lens, scale)
    o_f, lse_f = mla.decode_attn(q, flat, seq_lens, scale)
    torch.cuda.synchronize()
    assert mla.get_device_error()[0] == 0
    assert torch.equal(o_p.view(torch.int16), o_f.view(torch.int16))
    assert torch.equal(lse_p.view(torch.int32), lse_f.view(torch.int32))
    for b in (0, 17, 31):
        ref_o, _ = oracle_direct(q_bits[b:b + 1], rows[b:b + 1], 512, scale)
        check_bf16(o_p[b:b + 1].float().cpu().numpy(), ref_o, f"paged headline b={b}")


def test_paged_append_lands_where_the_table_says(mla):
    # appending through a block table writes the same bits a contiguous append
    # writes, at row pos % 64 of page table[b][pos // 64]
    d_c, d_r, B, max_blocks = 512, 64, 3, 4
    lens = [200, 64, 1]
    table, num_pages = _page_assignment(5, lens, max_blocks, spare=2)
    paged = mla.PagedLatentCache(num_pages, B, max_blocks, d_c, d_r, block_table=torch.from_numpy(table).cuda())
    paged.data.fill_(float("nan"))
    flat = mla.LatentCache(B, max_blocks * PR, d_c, d_r, dtype=torch.bfloat16)
    flat.data.fill_(float("nan"))
    seq = np.concatenate([np.full(n, b, dtype=np.int32) for b, n in enumerate(lens)])
    pos = np.concatenate([np.random.default_rng(b).permutation(n).astype(np.int32) for b, n in enumerate(lens)])
    T = len(seq)
    c_kv = to_device(W.bf16_bits(W.normal(5, "paged_ckv", (T, d_c))), "bf16")
    k_r = to_device(W.bf16_bits(W.normal(5, "paged_kr", (T, d_r))), "bf16")
    s_dev, p_dev = torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda()
    mla.cache_append(flat, c_kv, k_r, s_dev, p_dev)
    mla.cache_append_paged(paged, c_kv, k_r, s_dev, p_dev)
    torch.cuda.synchronize()
    assert mla.get_device_error()[0] == 0
    R = d_c + d_r
    for b, n in enumerate(lens):
        got = torch.cat([paged.data[table[b, j]] for j in range(max_blocks)])[:n, :R]
        assert torch.equal(got.view(torch.int16), flat.data[b, :n, :R].view(torch.int16)), b
    # the spare pages stay untouched
    used = {int(table[b, j]) for b, n in enumerate(lens) for j in range(-(-n // PR))}
    for pg in set(range(num_pages)) - used:
        assert torch.isnan(paged.data[pg].float()).all()


def test_paged_out_of_range_page_is_recorded(mla):
    # a block-table entry outside the pool is recorded as a device index error; the
    # kernels read page 0 instead (decode) or skip the row (append), both in bounds
    d_c, d_r, B, max_blocks = 512, 64, 2, 2
    table = np.array([[0, 1], [2, 7]], dtype=np.int32)  # pool of 4 pages: 7 is outside
    paged = mla.PagedLatentCache(4, B, max_blocks, d_c, d_r, block_table=torch.from_numpy(table).cuda())
    q = torch.zeros((B, 128, d_c + d_r), dtype=torch.bfloat16, device="cuda")
    mla.get_device_error()  # clear
    mla.decode_attn_paged(q, paged, torch.tensor([100, 100], dtype=torch.int32, device="cuda"), 0.1)
    st, word = mla.get_device_error()
    assert st == ERR_DEVICE_INDEX, f"{word:#x}"
    c_kv = torch.zeros((1, d_c), dtype=torch.bfloat16, device="cuda")
    k_r = torch.zeros((1, d_r), dtype=torch.bfloat16, device="cuda")
    mla.cache_append_paged(paged, c_kv, k_r, torch.tensor([1], dtype=torch.int32, device="cuda"),
                           torch.tensor([70], dtype=torch.int32, device="cuda"))
    st, word = mla.get_device_error()
    assert st == ERR_DEVICE_INDEX, f"{word:#x}"
    # in range again: no error left behind
    mla.decode_attn_paged(q, paged, torch.tensor([100, 64], dtype=torch.int32, device="cuda"), 0.1)
    assert mla.get_device_error()[0] == 0
