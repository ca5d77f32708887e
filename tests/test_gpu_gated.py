"""GPU parity of the output gate (tensor-core and CUDA-core paths) and of the gated,
RoPE-free decode step at its full size (B16 x H64 x N131072, d_model 4096)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import DecodeCase, check_bf16, check_f32, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import head_latent_attention_29_b300 as m
    return m


def _gate_case(mla, seed, B, d_model, width, dtype):
    h = W.as_dtype(W.normal(seed, "t_gate_h", (B, d_model)), dtype)
    w_g = W.as_dtype(W.normal(seed, "t_gate_w", (d_model, width), std=1.0 / np.sqrt(d_model)), dtype)
    o = W.as_dtype(W.normal(seed, "t_gate_o", (B, width)), dtype)
    o_dev = to_device(o, dtype)
    mla.gate(to_device(h, dtype), to_device(w_g, dtype), o_dev)
    torch.cuda.synchronize()
    ref = O.gate(W.widen(h, dtype), W.widen(w_g, dtype), W.widen(o, dtype))
    return o_dev.float().cpu().numpy(), ref


@pytest.mark.parametrize("B,d_model,width", [(16, 4096, 8192), (5, 128, 256), (1, 64, 128), (40, 192, 384),
                                             (300, 256, 256)])
def test_gate_tensor_core(mla, B, d_model, width):
    got, ref = _gate_case(mla, 1, B, d_model, width, "bf16")
    check_bf16(got, ref, f"gate B{B} d{d_model} w{width}")


@pytest.mark.parametrize("B,d_model,width", [(4, 64, 96), (17, 33, 40), (3, 4096, 256)])
def test_gate_fp32_cuda_cores(mla, B, d_model, width):
    # fp32 runs on the CUDA cores, any shape
    got, ref = _gate_case(mla, 2, B, d_model, width, "f32")
    check_f32(got, ref, "gate fp32")


def test_gate_bf16_shape_outside_the_tensor_cores_is_refused(mla):
    # bf16 has no CUDA-core gate to fall back to: a width that is not a multiple of
    # 128 is refused and the output is left as it was
    o = torch.ones(3, 200, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.gate(torch.ones(3, 100, dtype=torch.bfloat16, device="cuda"),
                 torch.ones(100, 200, dtype=torch.bfloat16, device="cuda"), o)
    assert e.value.status == 2  # MLA_ERR_UNSUPPORTED
    assert bool(torch.all(o == 1))


def test_gate_zero_weights_halves(mla):
    # W_g = 0 gives sigmoid(0) = 1/2 on every channel (exact in bf16 for these o)
    B, d_model, width = 4, 128, 256
    o = W.as_dtype(W.normal(3, "t_gate_o", (B, width)), "bf16")
    o_dev = to_device(o, "bf16")
    mla.gate(torch.ones(B, d_model, dtype=torch.bfloat16, device="cuda"),
             torch.zeros(d_model, width, dtype=torch.bfloat16, device="cuda"), o_dev)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o_dev.float().cpu().numpy(), W.widen(o, "bf16") * 0.5)


def test_gated_step_full_size(mla):
    # the whole gated step at B16 x H64 x N131072 (no RoPE, scale 1/sqrt(128)):
    # append, absorb, split attention + combine, W_UV, gate; every sequence checked
    # against the oracle one by one
    case = DecodeCase("gated_h64_b16_n131072", seed=5)
    cfg = case.cfg
    cache = case.device_cache(mla)
    q_nope, _ = case.query()
    w_uk, w_uv = case.weights()
    B, H = case.B, case.H
    q_pos = torch.from_numpy((case.lens - 1).astype(np.int32)).cuda()
    q_cat = mla.absorb_q(to_device(q_nope, "bf16"), None, q_pos, to_device(w_uk, "bf16"))
    o_lat, lse = mla.decode_attn(q_cat, cache, torch.from_numpy(case.lens).cuda(), case.scale)
    o = mla.out_up(o_lat, to_device(w_uv, "bf16"))
    h, w_g = W.gate_inputs(cfg, case.seed)
    h, w_g = W.as_dtype(h, "bf16"), W.as_dtype(w_g, "bf16")
    o_flat = o.view(B, -1)
    o_before = o_flat.float().cpu().numpy()
    mla.gate(to_device(h, "bf16"), to_device(w_g, "bf16"), o_flat)
    torch.cuda.synchronize()
    st, detail = mla.get_device_error()
    assert st == 0, (st, detail)
    got = o_flat.float().cpu().numpy()
    wg64 = W.widen(w_g, "bf16")
    for b in range(B):
        ref_o, ref_lat, ref_lse = case.oracle_seq(b)
        check_bf16(o_lat[b].float().cpu().numpy(), ref_lat, f"gated o_lat b={b}")
        np.testing.assert_allclose(lse[b].cpu().numpy(), ref_lse, rtol=1e-3, atol=2e-2)
        check_bf16(o_before[b], ref_o.reshape(-1), f"gated o (before gate) b={b}")
        ref_g = O.gate(W.widen(h[b : b + 1], "bf16"), wg64, ref_o.reshape(1, -1))[0]
        check_bf16(got[b], ref_g, f"gated output b={b}")
