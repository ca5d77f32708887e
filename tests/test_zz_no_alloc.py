"""The allocation-free decode entry point gives the same attention as the
workspace entry point.

mla_decode_attn_noalloc serves callers that cannot allocate device memory when
they run attention (graph capture/replay, non-reentrant allocators, embedders
that only own their input and output buffers); it takes its scratch from a buffer
built into the library.  This file is collected last on purpose."""
import math

import numpy as np
import pytest
import torch

from tests._cases import TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, direct_decode_inputs, rel_l2, upload_direct

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(mla):
    scale = 1.0 / math.sqrt(192)
    # two calls in a row on different batches: the second must not see the first's scratch
    for seed, lens in [(31, [4096, 100, 65, 2000, 1]), (32, [777, 3000, 64])]:
        lens = np.asarray(lens, dtype=np.int32)
        q_bits, rows = direct_decode_inputs(seed, lens, 128, 512, 64)
        q, cache = upload_direct(mla, q_bits, rows, 512, 64, int(lens.max()))
        seq_lens = torch.from_numpy(lens).cuda()
        ref_o, ref_lse = mla.decode_attn(q, cache, seq_lens, scale)
        out = torch.empty_like(ref_o)
        lse = torch.empty_like(ref_lse)
        mla.decode_attn_noalloc(q, cache, seq_lens, scale, out, lse)
        torch.cuda.synchronize()
        st, word = mla.get_device_error()
        assert st == 0, f"device error word {word:#x}"
        a = out.float().cpu().numpy()
        b = ref_o.float().cpu().numpy()
        assert np.all(np.isfinite(a))
        assert float(np.max(np.abs(a - b))) <= TOL_BF16_MAX_ABS and rel_l2(a, b) <= TOL_BF16_REL_L2
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=2e-2, rtol=1e-3)


def test_noalloc_rejects_batches_beyond_its_scratch(mla):
    cache = mla.LatentCache(33, 8, 512, 64)
    q = torch.zeros((33, 128, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((33, 128, 512), dtype=torch.bfloat16, device="cuda")
    seq_lens = torch.ones(33, dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.decode_attn_noalloc(q, cache, seq_lens, 0.07, out)
    assert e.value.status == 5  # MLA_ERR_WORKSPACE
