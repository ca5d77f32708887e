"""The allocation-free decode entry point gives the same attention as the
workspace entry point.

mla_decode_attn_noalloc is for callers that cannot hand the library device
memory when they run attention: code under an allocator that must not be
re-entered from that point, runtimes whose device memory is fixed at start-up,
or embedders that only own the input and output buffers.  It runs the same
kernels as mla_decode_attn with their scratch taken from a buffer built into the
library, so on the same inputs its outputs must be bit-identical.  This file is
collected last on purpose: a run that stops at the first failure has then run
every other test."""
import math

import numpy as np
import pytest
import torch

from tests._cases import check_bf16, direct_decode_inputs, oracle_direct, upload_direct

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(mla):
    scale = 1.0 / math.sqrt(192)
    # calls in a row on different batches: none may see another's scratch (the
    # lengths differ, so the run plans and the cut problems differ); the last two are
    # a few long sequences, whose pieces go through the grouped merge's partials
    cases = [(31, [4096, 100, 65, 2000, 1]), (32, [777, 3000, 64, 5000] * 8), (33, [30000]),
             (34, [20000, 16000, 9000])]
    for k, (seed, lens) in enumerate(cases):
        lens = np.asarray(lens, dtype=np.int32)
        q_bits, rows = direct_decode_inputs(seed, lens, 128, 512, 64)
        q, cache = upload_direct(mla, q_bits, rows, 512, 64, int(lens.max()))
        seq_lens = torch.from_numpy(lens).cuda()
        out = torch.empty((len(lens), 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((len(lens), 128), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        mla.decode_attn_noalloc(q, cache, seq_lens, scale, out, lse)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before  # the binding allocates nothing either
        st, word = mla.get_device_error()
        assert st == 0, f"device error word {word:#x}"
        ref_o, ref_lse = mla.decode_attn(q, cache, seq_lens, scale)
        torch.cuda.synchronize()
        # same kernels, same inputs: the same bits
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)), f"call {k}: o_lat bits differ"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), f"call {k}: lse bits differ"
        if k == 0:
            o_ref, lse_ref = oracle_direct(q_bits, rows, 512, scale)
            check_bf16(out.float().cpu().numpy(), o_ref, "no-alloc o_lat vs oracle")
            np.testing.assert_allclose(lse.cpu().numpy(), lse_ref, atol=2e-2, rtol=1e-3)


def test_noalloc_rejects_batches_beyond_its_scratch(mla):
    cache = mla.LatentCache(33, 8, 512, 64)
    q = torch.zeros((33, 128, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((33, 128, 512), dtype=torch.bfloat16, device="cuda")
    seq_lens = torch.ones(33, dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.decode_attn_noalloc(q, cache, seq_lens, 0.07, out)
    assert e.value.status == 5  # MLA_ERR_WORKSPACE


def test_noalloc_checks_caller_buffers_before_launch(mla):
    cache = mla.LatentCache(4, 64, 512, 64)
    q = torch.zeros((4, 128, 576), dtype=torch.bfloat16, device="cuda")
    seq_lens = torch.ones(4, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):   # output one sequence short
        mla.decode_attn_noalloc(q, cache, seq_lens, 0.07, torch.empty((3, 128, 512), dtype=torch.bfloat16,
                                                                      device="cuda"))
    out = torch.empty((4, 128, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):   # lse of the wrong shape
        mla.decode_attn_noalloc(q, cache, seq_lens, 0.07, out, torch.empty((4, 64), device="cuda"))
    with pytest.raises(ValueError):   # q_cat of another batch
        mla.decode_attn_noalloc(q[:2], cache, seq_lens, 0.07, out)
