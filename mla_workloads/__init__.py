"""Seeded synthetic inputs for the MLA decode workloads.

This module is shared by the float64 oracle, the tests and ``bench.py``.  It holds
shapes, distributions and random draws only -- none of the attention arithmetic
(no projection, rotation, softmax or contraction lives here).  The only numeric
transform is the round-to-nearest-even narrowing of float32 draws to bfloat16,
which is how every bf16 workload is materialised before either side sees it.

Every tensor is drawn from its own PCG64 stream keyed by (seed, tensor name,
optional index), so a test can regenerate one sequence of a large ragged batch
without drawing the rest.
"""
from __future__ import annotations

import math
import zlib

import numpy as np

# ---------------------------------------------------------------------------
# Workload table.  Shapes and distributions follow the DeepSeek-V2/V3-shaped
# MLA decode described in "MLA multi-head latent attention: low-rank
# compression and matrix absorption" (0539edu.com, sections 2.2 and 4.1:
# h=128, d_k=d_v=128, d_c=512) with the 512+64 cache row of the icman.com.cn
# MLA article (section 2, decoupled RoPE), and the gated no-RoPE variant of the
# "Gated MLA" write-up (tahou.com, sections 2.6 and 3.3).
# ---------------------------------------------------------------------------
WORKLOADS: dict[str, dict] = {
    # tiny fp32 decode driven from hidden states; both absorbed and explicit
    # forms are checked on it
    "tiny_fp32": dict(
        B=1, H=4, d_model=64, d_c=32, d_r=8, d_k=16, d_v=16, N=64,
        dtype="f32", rope_base=10000.0, scale=1.0 / math.sqrt(24.0),
    ),
    # the headline decode: 32 sequences of 4096 cached tokens, 128 heads
    "decode_h128_b32_n4096": dict(
        B=32, H=128, d_c=512, d_r=64, d_k=128, d_v=128, N=4096,
        dtype="bf16", rope_base=10000.0, w_std=1.0 / math.sqrt(512.0),
        scale=1.0 / math.sqrt(192.0),
    ),
    # long-context ragged decode: per-sequence lengths uniform in [1024, 32768]
    "ragged_h128_b64_n1k_32k": dict(
        B=64, H=128, d_c=512, d_r=64, d_k=128, d_v=128, N_lo=1024, N_hi=32768,
        dtype="bf16", rope_base=10000.0, w_std=1.0 / math.sqrt(512.0),
        scale=1.0 / math.sqrt(192.0),
    ),
    # chunked causal prefill over the latent cache (absorbed form)
    "prefill_h128_b4_s8192": dict(
        B=4, H=128, d_c=512, d_r=64, d_k=128, d_v=128, S=8192,
        dtype="bf16", rope_base=10000.0, w_std=1.0 / math.sqrt(512.0),
        scale=1.0 / math.sqrt(192.0),
    ),
    # a small causal prefill of the same shape per token (profiling-sized case)
    "prefill_h128_b1_s2048": dict(
        B=1, H=128, d_c=512, d_r=64, d_k=128, d_v=128, S=2048,
        dtype="bf16", rope_base=10000.0, w_std=1.0 / math.sqrt(512.0),
        scale=1.0 / math.sqrt(192.0),
    ),
    # the new tokens' cache rows straight from their hidden states: c_KV =
    # RMSNorm(h W_DKV), k_R = RoPE(h W_KR), written at position N - 1 of each of
    # the 32 decode sequences (DeepSeek-V3 hidden size)
    "kvdown_b32_d7168": dict(
        T=32, B=32, N=4096, d_model=7168, d_c=512, d_r=64,
        dtype="bf16", rope_base=10000.0, eps=1e-6,
    ),
    # the same for a 8192-token prompt chunk of 4 sequences (prefill shape)
    "kvdown_t32768_d7168": dict(
        T=32768, B=4, prompt=8192, d_model=7168, d_c=512, d_r=64,
        dtype="bf16", rope_base=10000.0, eps=1e-6,
    ),
    # gated MLA without RoPE: 64 heads, 131072 cached tokens, full-rank gate
    "gated_h64_b16_n131072": dict(
        B=16, H=64, d_c=512, d_r=0, d_k=128, d_v=128, N=131072, d_model=4096,
        dtype="bf16", w_std=1.0 / math.sqrt(512.0), wg_std=1.0 / math.sqrt(4096.0),
        scale=1.0 / math.sqrt(128.0),
    ),
}


def _rng(seed: int, name: str, *index: int) -> np.random.Generator:
    key = zlib.crc32(name.encode("utf-8"))
    return np.random.Generator(np.random.PCG64([int(seed), key, *[int(i) for i in index]]))


def normal(seed: int, name: str, shape, std: float = 1.0, index: tuple = ()) -> np.ndarray:
    """float32 draws from N(0, std^2) on the stream (seed, name, *index)."""
    x = _rng(seed, name, *index).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def uniform_int(seed: int, name: str, lo: int, hi: int, size: int) -> np.ndarray:
    """int32 draws uniform on the inclusive range [lo, hi]."""
    return _rng(seed, name).integers(lo, hi + 1, size=size, dtype=np.int64).astype(np.int32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Materialise a float32 draw in the workload dtype.

    Returns float32 for "f32" and the bf16 bit patterns (uint16) for "bf16"."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits(x)
    raise ValueError(dtype)


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 view of a materialised tensor (exact for both dtypes)."""
    if dtype == "bf16":
        return bf16_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Per-workload draws.  Names are stable so that any subset can be redrawn.
# ---------------------------------------------------------------------------
def seq_lens(cfg: dict, seed: int) -> np.ndarray:
    """Context length of every sequence (int32 [B])."""
    if "N" in cfg:
        return np.full(cfg["B"], cfg["N"], dtype=np.int32)
    return uniform_int(seed, "seq_lens", cfg["N_lo"], cfg["N_hi"], cfg["B"])


def latent_rows(cfg: dict, seed: int, b: int, n: int):
    """Cached inputs of sequence b: c_KV [n, d_c] and the pre-rotation k_R [n, d_r]
    (float32 draws, N(0,1))."""
    c_kv = normal(seed, "c_kv", (n, cfg["d_c"]), index=(b,))
    k_r = normal(seed, "k_r", (n, cfg["d_r"]), index=(b,))
    return c_kv, k_r


def query(cfg: dict, seed: int, B: int | None = None, S: int = 1):
    """Per-head query parts q_nope [B, S, H, d_k] and q_R [B, S, H, d_r], N(0,1)."""
    B = cfg["B"] if B is None else B
    q_nope = normal(seed, "q_nope", (B, S, cfg["H"], cfg["d_k"]))
    q_r = normal(seed, "q_r", (B, S, cfg["H"], cfg["d_r"]))
    return q_nope, q_r


def up_weights(cfg: dict, seed: int):
    """W_UK [H, d_k, d_c] and W_UV [H, d_v, d_c], N(0, w_std^2)."""
    std = cfg.get("w_std", 1.0 / math.sqrt(cfg["d_c"]))
    w_uk = normal(seed, "w_uk", (cfg["H"], cfg["d_k"], cfg["d_c"]), std=std)
    w_uv = normal(seed, "w_uv", (cfg["H"], cfg["d_v"], cfg["d_c"]), std=std)
    return w_uk, w_uv


def gate_inputs(cfg: dict, seed: int):
    """Gate input hidden state h [B, d_model] ~ N(0,1) and W_g [d_model, H*d_v]."""
    h = normal(seed, "gate_h", (cfg["B"], cfg["d_model"]))
    w_g = normal(seed, "w_g", (cfg["d_model"], cfg["H"] * cfg["d_v"]), std=cfg["wg_std"])
    return h, w_g


def hidden_model(cfg: dict, seed: int):
    """Hidden states and projection weights for the tiny hidden-state-driven decode.

    Returns h [B, N, d_model] ~ N(0,1) and W_DKV [d_model, d_c], W_KR [d_model, d_r],
    W_UQ [d_model, H*(d_k+d_r)] ~ N(0, 1/d_model), W_UK [H, d_k, d_c] and
    W_UV [H, d_v, d_c] ~ N(0, 1/d_c)."""
    B, N, dm = cfg["B"], cfg["N"], cfg["d_model"]
    H, d_c, d_r, d_k, d_v = cfg["H"], cfg["d_c"], cfg["d_r"], cfg["d_k"], cfg["d_v"]
    h = normal(seed, "h", (B, N, dm))
    s_in = 1.0 / math.sqrt(dm)
    w_dkv = normal(seed, "w_dkv", (dm, d_c), std=s_in)
    w_kr = normal(seed, "w_kr", (dm, d_r), std=s_in)
    w_uq = normal(seed, "w_uq", (dm, H * (d_k + d_r)), std=s_in)
    s_c = 1.0 / math.sqrt(d_c)
    w_uk = normal(seed, "w_uk", (H, d_k, d_c), std=s_c)
    w_uv = normal(seed, "w_uv", (H, d_v, d_c), std=s_c)
    return dict(h=h, w_dkv=w_dkv, w_kr=w_kr, w_uq=w_uq, w_uk=w_uk, w_uv=w_uv)


def kv_down_inputs(cfg: dict, seed: int, T: int | None = None):
    """Hidden states h [T, d_model] ~ N(0,1), W_DKV [d_model, d_c] and W_KR
    [d_model, d_r] ~ N(0, 1/d_model), and the RMSNorm gain gamma [d_c] ~ 1 + N(0, 0.1^2)
    (a trained gain is not all ones; a unit gain would hide a dropped gain)."""
    T = cfg["T"] if T is None else T
    dm, d_c, d_r = cfg["d_model"], cfg["d_c"], cfg["d_r"]
    s_in = 1.0 / math.sqrt(dm)
    h = normal(seed, "kvd_h", (T, dm))
    w_dkv = normal(seed, "kvd_w_dkv", (dm, d_c), std=s_in)
    w_kr = normal(seed, "kvd_w_kr", (dm, d_r), std=s_in)
    gamma = 1.0 + normal(seed, "kvd_gamma", (d_c,), std=0.1)
    return h, w_dkv, w_kr, gamma.astype(np.float32)
