"""GPU parity of mla_kv_down_append -- new tokens' cache rows from their hidden
states, [RMSNorm(h W_DKV) * gamma || RoPE(h W_KR, pos)] -- against the float64
oracle on the same materialised inputs.

Tolerances as for every bf16 output (max-abs <= 2e-2, relative L2 <= 1e-2) and
relative L2 <= 1e-4 for fp32.  Rows the call must not touch hold NaN and are
checked to still hold it."""
import numpy as np
import pytest
import torch

import mla_workloads as W
from oracle import mla_oracle as O
from tests._cases import check_bf16, check_f32, to_device

pytestmark = pytest.mark.gpu
ERR_DEVICE_INDEX = 6


@pytest.fixture(scope="module")
def mla():
    import head_latent_attention_29_b300 as m
    m.lib()
    return m


def _inputs(T, d_model, d_c, d_r, dtype, seed, B=4, N_max=300):
    cfg = dict(W.WORKLOADS["kvdown_b32_d7168"], d_model=d_model, d_c=d_c, d_r=d_r)
    h, w_dkv, w_kr, gamma = W.kv_down_inputs(cfg, seed, T=T)
    w = np.concatenate([w_dkv, w_kr], axis=1)
    rng = np.random.default_rng(seed)
    # distinct (sequence, position) slots: rows must not alias
    slots = rng.choice(B * N_max, size=T, replace=False)
    seq, pos = (slots // N_max).astype(np.int32), (slots % N_max).astype(np.int32)
    mat = {k: W.as_dtype(v, dtype) for k, v in dict(h=h, w=w, gamma=gamma).items()}
    return mat, seq, pos


def _oracle(mat, dtype, d_c, pos, eps, base=1e4):
    h, w, g = (W.widen(mat[k], dtype) for k in ("h", "w", "gamma"))
    return O.kv_down_rows(h, w[:, :d_c], w[:, d_c:], g, eps, pos, base)


def _run(mla, mat, seq, pos, dtype, d_c, d_r, B, N_max, eps, cache=None):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    if cache is None:
        cache = mla.LatentCache(B, N_max, d_c, d_r, dtype=tdt)
        cache.data.fill_(float("nan"))
    mla.kv_down_append(cache, to_device(mat["h"], dtype), to_device(mat["w"], dtype),
                       to_device(mat["gamma"], dtype), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                       eps=eps)
    torch.cuda.synchronize()
    st, word = mla.get_device_error()
    assert st == 0, f"device error word {word:#x}"
    return cache


def _written(cache, seq, pos, R):
    return cache.data[torch.from_numpy(seq).long(), torch.from_numpy(pos).long(), :R].float().cpu().numpy()


def _untouched_nan(cache, seq, pos, R):
    mask = torch.ones(cache.data.shape[:2], dtype=torch.bool)
    mask[torch.from_numpy(seq).long(), torch.from_numpy(pos).long()] = False
    rest = cache.data[..., :R][mask.cuda()]
    return bool(torch.isnan(rest.float()).all())


# tensor-core projection: one and several 128-column tiles with a 64-wide last tile,
# token tiles of 16..256 and a ragged second token tile, K split over the SMs
# (K ranges: 30 at d_model 7168, 16 at 1024, 32 at 2048, 2 at 128, 1 at 64)
@pytest.mark.parametrize("T,d_model,d_r", [(1, 7168, 64), (5, 1024, 64), (32, 7168, 64), (300, 512, 64),
                                           (17, 2048, 0), (64, 64, 64), (64, 7168, 64), (65, 7168, 64),
                                           (33, 128, 64)])
def test_kv_down_tensor_core_path(mla, T, d_model, d_r):
    d_c, B, N_max, eps = 512, 4, 300, 1e-6
    mat, seq, pos = _inputs(T, d_model, d_c, d_r, "bf16", seed=T + d_model)
    cache = _run(mla, mat, seq, pos, "bf16", d_c, d_r, B, N_max, eps)
    got = _written(cache, seq, pos, d_c + d_r)
    check_bf16(got, _oracle(mat, "bf16", d_c, pos, eps), f"kv_down T={T} d_model={d_model} d_r={d_r}")
    assert _untouched_nan(cache, seq, pos, d_c + d_r)


def test_kv_down_fp32_tiny_shapes(mla):
    # the tiny fp32 model's widths (d_model 64, d_c 32, d_r 8): the CUDA-core path
    cfg = W.WORKLOADS["tiny_fp32"]
    d_c, d_r, B, N_max, eps = cfg["d_c"], cfg["d_r"], 2, 64, 1e-5
    mat, seq, pos = _inputs(40, cfg["d_model"], d_c, d_r, "f32", seed=7, B=B, N_max=N_max)
    cache = _run(mla, mat, seq, pos, "f32", d_c, d_r, B, N_max, eps)
    check_f32(_written(cache, seq, pos, d_c + d_r), _oracle(mat, "f32", d_c, pos, eps), "kv_down fp32")
    assert _untouched_nan(cache, seq, pos, d_c + d_r)


def test_kv_down_bf16_shape_outside_the_tensor_cores_is_refused(mla):
    # d_model = 200 is not a multiple of 64: bf16 has no CUDA-core projection to
    # fall back to, so the call is refused and the cache stays untouched
    d_c, d_r, eps = 512, 64, 0.0
    mat, seq, pos = _inputs(9, 200, d_c, d_r, "bf16", seed=8)
    with pytest.raises(mla.MlaError) as e:
        _run(mla, mat, seq, pos, "bf16", d_c, d_r, 4, 300, eps)
    assert e.value.status == 2  # MLA_ERR_UNSUPPORTED


def test_kv_down_deterministic_and_paged_equal(mla):
    # the same call twice gives the same bits; through a shuffled page table it
    # writes exactly the rows the contiguous cache gets
    d_c, d_r, B, N_max, T = 512, 64, 4, 256, 48
    mat, seq, pos = _inputs(T, 7168, d_c, d_r, "bf16", seed=9, B=B, N_max=N_max)
    a = _run(mla, mat, seq, pos, "bf16", d_c, d_r, B, N_max, 1e-6)
    b = _run(mla, mat, seq, pos, "bf16", d_c, d_r, B, N_max, 1e-6)
    assert torch.equal(a.data.view(torch.int16), b.data.view(torch.int16))
    max_blocks = N_max // 64
    table = np.random.default_rng(9).permutation(B * max_blocks).astype(np.int32).reshape(B, max_blocks)
    paged = mla.PagedLatentCache(B * max_blocks, B, max_blocks, d_c, d_r, block_table=torch.from_numpy(table).cuda())
    paged.data.fill_(float("nan"))
    _run(mla, mat, seq, pos, "bf16", d_c, d_r, B, N_max, 1e-6, cache=paged)
    for s, p in zip(seq, pos):
        got = paged.data[table[s, p // 64], p % 64]
        assert torch.equal(got.view(torch.int16), a.data[s, p].view(torch.int16))


def test_kv_down_out_of_range_rows_recorded(mla):
    d_c, d_r = 512, 64
    mat, seq, pos = _inputs(4, 1024, d_c, d_r, "bf16", seed=10)
    pos = pos.copy()
    pos[2] = 300  # == N_max: out of range, skipped
    tdt = torch.bfloat16
    cache = mla.LatentCache(4, 300, d_c, d_r, dtype=tdt)
    cache.data.fill_(float("nan"))
    mla.get_device_error()
    mla.kv_down_append(cache, to_device(mat["h"], "bf16"), to_device(mat["w"], "bf16"),
                       to_device(mat["gamma"], "bf16"), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda())
    st, word = mla.get_device_error()
    assert st == ERR_DEVICE_INDEX, f"{word:#x}"
    keep = np.array([0, 1, 3])
    ref = _oracle({k: v[keep] if k == "h" else v for k, v in mat.items()}, "bf16", d_c, pos[keep], 1e-6)
    check_bf16(_written(cache, seq[keep], pos[keep], d_c + d_r), ref, "kv_down rows kept")
    assert _untouched_nan(cache, seq[keep], pos[keep], d_c + d_r)


@pytest.mark.parametrize("workload,sample", [("kvdown_b32_d7168", None), ("kvdown_t32768_d7168", 48)])
def test_kv_down_workload_sizes(mla, workload, sample):
    # the two measured workloads at full size, in the launch configuration the
    # benchmark times; the prompt-sized one is checked on sampled tokens
    cfg = W.WORKLOADS[workload]
    T, d_c, d_r, eps = cfg["T"], cfg["d_c"], cfg["d_r"], cfg["eps"]
    h, w_dkv, w_kr, gamma = W.kv_down_inputs(cfg, seed=0)
    mat = {k: W.as_dtype(v, "bf16") for k, v in
           dict(h=h, w=np.concatenate([w_dkv, w_kr], axis=1), gamma=gamma).items()}
    if "prompt" in cfg:
        B, N_max = cfg["B"], cfg["prompt"]
        seq = np.repeat(np.arange(B, dtype=np.int32), N_max)
        pos = np.tile(np.arange(N_max, dtype=np.int32), B)
    else:
        B, N_max = cfg["B"], cfg["N"]
        seq = np.arange(T, dtype=np.int32) % B
        pos = np.full(T, N_max - 1, dtype=np.int32)
    cache = _run(mla, mat, seq, pos, "bf16", d_c, d_r, B, N_max, eps)
    idx = np.arange(T) if sample is None else np.sort(np.random.default_rng(0).choice(T, sample, replace=False))
    ref = _oracle({"h": mat["h"][idx], "w": mat["w"], "gamma": mat["gamma"]}, "bf16", d_c, pos[idx], eps)
    check_bf16(_written(cache, seq[idx], pos[idx], d_c + d_r), ref, workload)
