"""Failure detection on the GPU without a fault: every wait of the tensor-core
attention kernel is bounded.  With the test-only fault injection the score CTAs
issue no loads, so the waits on them run out after their bound (about one
second); the call must record MLA_ERR_DEVICE_TIMEOUT in the device error word,
nothing may fault or hang, and the next call on the same context must give the
normal result."""
import math

import numpy as np
import pytest
import torch

from tests._cases import direct_decode_inputs, upload_direct

pytestmark = pytest.mark.gpu

MLA_ERR_DEVICE_TIMEOUT = 4
SITE_DECODE_WAIT = 3


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def test_bounded_waits_expire_and_the_context_survives(mla):
    lens = np.asarray([300, 64], dtype=np.int32)
    q_bits, rows = direct_decode_inputs(41, lens, 128, 512, 64)
    q, cache = upload_direct(mla, q_bits, rows, 512, 64, int(lens.max()))
    seq_lens = torch.from_numpy(lens).cuda()
    scale = 1.0 / math.sqrt(192)
    ref, ref_lse = mla.decode_attn(q, cache, seq_lens, scale)
    assert mla.get_device_error()[0] == 0

    mla.debug_inject_fault(1)
    try:
        mla.decode_attn(q, cache, seq_lens, scale)
        st, word = mla.get_device_error()
    finally:
        mla.debug_inject_fault(0)
    assert st == MLA_ERR_DEVICE_TIMEOUT, f"status {st}, word {word:#x}"
    assert (word & 0xFF) == MLA_ERR_DEVICE_TIMEOUT and (word >> 8) == SITE_DECODE_WAIT
    assert mla.get_device_error()[0] == 0  # read and cleared

    out, lse = mla.decode_attn(q, cache, seq_lens, scale)
    assert mla.get_device_error()[0] == 0
    np.testing.assert_array_equal(out.float().cpu().numpy(), ref.float().cpu().numpy())
    np.testing.assert_array_equal(lse.cpu().numpy(), ref_lse.cpu().numpy())


def test_fault_injection_rejects_unknown_kinds(mla):
    with pytest.raises(mla.MlaError):
        mla.debug_inject_fault(7)
