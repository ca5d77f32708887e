"""GPU checks of mla_absorb_q_append (the decode step's new cache rows written by
the absorb launch): its q_cat and cache rows are bit-identical to mla_absorb_q plus
mla_cache_append on the same inputs (contiguous and paged caches), and both match
the float64 oracle (0539edu.com sections 3.1 and 5.2; icman.com.cn section 2).
Tolerances as for every bf16 output: max-abs <= 2e-2, relative L2 <= 1e-2."""
import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import check_bf16, to_device

pytestmark = pytest.mark.gpu
ERR_DEVICE_INDEX = 6


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _inputs(seed, B, H, N_max, d_c=512, d_r=64, d_k=128):
    rng = np.random.default_rng(seed)
    bf = lambda a: to_device(W.as_dtype(a.astype(np.float32), "bf16"), "bf16")
    c_kv = rng.standard_normal((B, d_c))
    k_r = rng.standard_normal((B, d_r))
    q_nope = rng.standard_normal((B, H, d_k))
    q_rope = rng.standard_normal((B, H, d_r))
    w_uk = rng.standard_normal((H, d_k, d_c)) / np.sqrt(d_c)
    pos = rng.integers(0, N_max, size=B).astype(np.int32)
    host = dict(c_kv=c_kv, k_r=k_r, q_nope=q_nope, q_rope=q_rope, w_uk=w_uk)
    dev = {k: bf(v) for k, v in host.items()}
    dev["seq"] = torch.arange(B, dtype=torch.int32, device="cuda")
    dev["pos"] = torch.from_numpy(pos).cuda()
    return host, dev, pos


def _separate(mla, cache, d):
    append = mla.cache_append_paged if isinstance(cache, mla.PagedLatentCache) else mla.cache_append
    append(cache, d["c_kv"], d["k_r"], d["seq"], d["pos"])
    return mla.absorb_q(d["q_nope"], d["q_rope"], d["pos"], d["w_uk"])


def _fused(mla, cache, d):
    return mla.absorb_q_append(cache, d["c_kv"], d["k_r"], d["seq"], d["pos"], d["q_nope"], d["q_rope"], d["pos"],
                               d["w_uk"])


def _ok(mla):
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"


@pytest.mark.parametrize("B,H", [(32, 128), (1, 128), (40, 64), (300, 16)])
def test_fused_equals_separate_calls_and_the_oracle(mla, B, H):
    N_max = 700
    host, d, pos = _inputs(B * 7 + H, B, H, N_max)
    a = mla.LatentCache(B, N_max, 512, 64)
    a.data.fill_(float("nan"))
    b = mla.LatentCache(B, N_max, 512, 64)
    b.data.fill_(float("nan"))
    q_ref = _separate(mla, a, d)
    q_got = _fused(mla, b, d)
    _ok(mla)
    assert torch.equal(q_got.view(torch.int16), q_ref.view(torch.int16))
    assert torch.equal(a.data.view(torch.int16), b.data.view(torch.int16))  # NaN rows stay NaN in both
    # against the oracle: the absorbed query and the rows
    wid = lambda k: W.widen(W.as_dtype(host[k].astype(np.float32), "bf16"), "bf16")
    q_or = O.absorb_q(wid("q_nope"), wid("q_rope"), pos, wid("w_uk"), 1e4)
    check_bf16(q_got.float().cpu().numpy(), q_or, f"q_cat B={B} H={H}")
    rows = b.data[torch.arange(B).cuda(), d["pos"].long()].float().cpu().numpy()
    ref_rows = O.cache_rows(wid("c_kv"), wid("k_r"), pos, 1e4)
    check_bf16(rows, ref_rows, f"appended rows B={B}")


def test_fused_paged_equals_separate(mla):
    B, H, max_blocks = 8, 128, 6
    host, d, pos = _inputs(5, B, H, 64 * max_blocks)
    table = torch.from_numpy(np.random.default_rng(5).permutation(B * max_blocks).astype(np.int32)
                             .reshape(B, max_blocks)).cuda()
    a = mla.PagedLatentCache(B * max_blocks, B, max_blocks, 512, 64, block_table=table)
    b = mla.PagedLatentCache(B * max_blocks, B, max_blocks, 512, 64, block_table=table)
    a.data.fill_(float("nan"))
    b.data.fill_(float("nan"))
    q_ref = _separate(mla, a, d)
    q_got = _fused(mla, b, d)
    _ok(mla)
    assert torch.equal(q_got.view(torch.int16), q_ref.view(torch.int16))
    assert torch.equal(a.data.view(torch.int16), b.data.view(torch.int16))


def test_fused_bad_row_is_skipped_and_recorded(mla):
    B, H, N_max = 4, 128, 100
    host, d, pos = _inputs(6, B, H, N_max)
    d["pos"][2] = N_max  # out of range: skipped
    cache = mla.LatentCache(B, N_max, 512, 64)
    cache.data.fill_(float("nan"))
    mla.get_device_error()
    _fused(mla, cache, d)
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == ERR_DEVICE_INDEX, f"{word:#x}"
    assert bool(torch.isnan(cache.data[2].float()).all())  # nothing of sequence 2 was written
    assert not bool(torch.isnan(cache.data[0, int(d["pos"][0])].float()).any())
