"""GPU checks of the captured decode step (head_latent_attention_29_b300.step.
DecodeStep, the runner the benchmark times): the new token's row appended by the
absorb launch, absorbed attention, W_UV -- replayed from a CUDA graph.  Its output
is bit-identical to the same step run eagerly through the separate calls
(mla_cache_append, mla_absorb_q, mla_decode_attn, mla_out_up) and matches the
float64 oracle (0539edu.com sections 3.1 and 5.2).  Tolerances as for every bf16
output: max-abs <= 2e-2, relative L2 <= 1e-2; fp32 relative L2 <= 1e-4."""
import numpy as np
import pytest
import torch

from head_latent_attention_29_b300.step import DecodeStep
from tests._cases import DecodeCase, check_bf16, check_f32, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _prefix_cache(mla, case, paged):
    """The cache with every row but each sequence's last (the step appends that one)."""
    tdt = torch.bfloat16 if case.dtype == "bf16" else torch.float32
    if paged:
        max_blocks = (case.N_max + 63) // 64
        table = np.random.default_rng(case.seed).permutation(case.B * max_blocks).astype(np.int32)
        cache = mla.PagedLatentCache(case.B * max_blocks, case.B, max_blocks, case.d_c, case.d_r, dtype=tdt,
                                     block_table=torch.from_numpy(table.reshape(case.B, max_blocks)).cuda())
    else:
        cache = mla.LatentCache(case.B, case.N_max, case.d_c, case.d_r, dtype=tdt)
    cache.data.fill_(float("nan"))
    append = mla.cache_append_paged if paged else mla.cache_append
    for b in range(case.B):
        n = int(case.lens[b]) - 1
        if n <= 0:
            continue
        c, k = case.seq_inputs(b)
        append(cache, to_device(c[:n], case.dtype), to_device(k[:n], case.dtype) if case.d_r else None,
               torch.full((n,), b, dtype=torch.int32, device="cuda"),
               torch.arange(n, dtype=torch.int32, device="cuda"), case.base)
    return cache


def _step_inputs(case):
    q_nope, q_r = case.query()
    new_c = np.stack([case.seq_inputs(b)[0][-1] for b in range(case.B)])
    new_k = np.stack([case.seq_inputs(b)[1][-1] for b in range(case.B)]) if case.d_r else None
    return new_c, new_k, q_nope, q_r


def _run_step(mla, case, paged):
    cache = _prefix_cache(mla, case, paged)
    w_uk, w_uv = case.weights()
    seq_lens = torch.from_numpy(case.lens).cuda()
    st = DecodeStep(cache, to_device(w_uk, case.dtype), to_device(w_uv, case.dtype), seq_lens, case.scale,
                    case.base)
    new_c, new_k, q_nope, q_r = _step_inputs(case)
    st.inputs["c_kv"].copy_(to_device(new_c, case.dtype))
    st.inputs["q_nope"].copy_(to_device(q_nope, case.dtype))
    if case.d_r:
        st.inputs["k_r"].copy_(to_device(new_k, case.dtype))
        st.inputs["q_rope"].copy_(to_device(q_r, case.dtype))
    st.launch()  # one eager run: one-time host set-up outside the capture
    torch.cuda.synchronize()
    st.capture()
    # the captured step re-appends the same rows and recomputes: same bits
    st.replay()
    torch.cuda.synchronize()
    stt, word = mla.get_device_error()
    assert stt == 0, f"device error word {word:#x}"
    return st


def _separate_calls(mla, case, paged):
    cache = _prefix_cache(mla, case, paged)
    w_uk, w_uv = case.weights()
    new_c, new_k, q_nope, q_r = _step_inputs(case)
    seq_idx = torch.arange(case.B, dtype=torch.int32, device="cuda")
    pos = torch.from_numpy(np.maximum(case.lens - 1, 0).astype(np.int32)).cuda()
    append = mla.cache_append_paged if paged else mla.cache_append
    append(cache, to_device(new_c, case.dtype), to_device(new_k, case.dtype) if case.d_r else None, seq_idx, pos,
           case.base)
    q_cat = mla.absorb_q(to_device(q_nope, case.dtype), to_device(q_r, case.dtype) if case.d_r else None, pos,
                         to_device(w_uk, case.dtype), case.base)
    attend = mla.decode_attn_paged if paged else mla.decode_attn
    o_lat, lse = attend(q_cat, cache, torch.from_numpy(case.lens).cuda(), case.scale)
    o = mla.out_up(o_lat, to_device(w_uv, case.dtype))
    torch.cuda.synchronize()
    return o, o_lat, lse


@pytest.mark.parametrize("paged", [False, True])
def test_captured_step_matches_separate_calls_and_the_oracle(mla, paged):
    lens = [300, 1, 64, 1000, 4096, 65, 129, 2048, 777, 3000, 17, 4095]
    case = DecodeCase("decode_h128_b32_n4096", seed=3, lens=lens)
    st = _run_step(mla, case, paged)
    o_ref, o_lat_ref, lse_ref = _separate_calls(mla, case, paged)
    assert torch.equal(st.o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(st.o_lat.view(torch.int16), o_lat_ref.view(torch.int16))
    assert torch.equal(st.lse, lse_ref)
    o = st.o.float().cpu().numpy()
    for b in range(case.B):
        r_o, r_lat, r_lse = case.oracle_seq(b)
        check_bf16(o[b], r_o, f"step o b={b} n={lens[b]} paged={paged}")
        np.testing.assert_allclose(st.lse[b].cpu().numpy(), r_lse, atol=2e-2, rtol=1e-3)


def test_captured_step_fp32_tiny(mla):
    # the tiny fp32 shapes: the CUDA-core kernels behind the same calls
    case = DecodeCase("tiny_fp32", seed=4, lens=[64, 1, 33])
    st = _run_step(mla, case, False)
    o_ref, _, _ = _separate_calls(mla, case, False)
    assert torch.equal(st.o, o_ref)
    o = st.o.cpu().numpy()
    for b in range(case.B):
        check_f32(o[b], case.oracle_seq(b)[0], f"fp32 step o b={b}")
