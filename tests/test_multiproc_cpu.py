"""The N > 1 host path on CPU: two gloo ranks (replicas) agree on the slowest
replica's time, the job rate counts every replica's units, and the oracle arm runs
on rank 0 only."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms per step: every rank must see the slowest, 2 ms
        t = bench.max_over_ranks(float(rank + 1), world, torch.device("cpu"))
        rate = bench.job_throughput(32, world, t * 1e-3)

        class Args:
            workload = "decode_h128_b32_n4096"
            seed = 0
            steps = 1
            warmup = 3

        ref = bench.run_reference(Args(), rank, world) if rank != 0 else "skipped"
        q.put((rank, t, rate, ref))
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, rate, ref in results:
        assert t == pytest.approx(2.0)
        assert rate == pytest.approx(32 * 2 / 2e-3)  # both replicas' tokens over the slowest step
        if rank != 0:
            assert ref is None  # the oracle arm runs (and prints) on rank 0 only


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_throughput(32, 1, 1e-4) == pytest.approx(320000.0)


def test_clock_window_brackets_a_short_region():
    # samples inside the timed region are used as they are; a region shorter than
    # the sampling period takes the samples on either side of it
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.samples = [(1.0, 1900.0, []), (2.0, 1950.0, ["sw_power_cap"]), (3.0, 2000.0, [])]
    c.max_mhz, c._mode, c.error = 2032.0, "smi", None
    c._t0, c._t1 = 1.5, 2.5
    s = c.summary()
    assert (s["sm_mhz"], s["samples"], s["window"], s["reasons"]) == (1950.0, 1, "inside", ["sw_power_cap"])
    c._t0, c._t1 = 2.1, 2.2
    s = c.summary()
    assert (s["sm_mhz"], s["samples"], s["window"]) == (1975.0, 2, "adjacent")


def test_decode_metric_names_its_shape():
    sys.path.insert(0, ROOT)
    import bench
    import mla_workloads as W
    assert bench.decode_metric("decode_h128_b32_n4096", W.WORKLOADS["decode_h128_b32_n4096"]).startswith(
        "MLA decode tokens/s at H=128,d_c=512,B=32,N=4K bf16")
    m = bench.decode_metric("gated_h64_b16_n131072", W.WORKLOADS["gated_h64_b16_n131072"])
    assert "H=64" in m and "N=131072" in m and "no RoPE" in m and "gate" in m
    assert "ragged" in bench.decode_metric("ragged_h128_b64_n1k_32k", W.WORKLOADS["ragged_h128_b64_n1k_32k"])


def test_stored_traffic_follows_kernel_code_not_comments(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(ROOT, "head_latent_attention_29_b300", "csrc", "k_decode_tc.cu")
    with open(src) as f:
        text = f.read()
    d = tmp_path / "head_latent_attention_29_b300" / "csrc"
    d.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (d / "k_decode_tc.cu").write_text(text)
    h0 = bench._kernel_hash()
    (d / "k_decode_tc.cu").write_text("// a new leading comment\n/* and a block\n comment */\n" + text + "\n\n")
    assert bench._kernel_hash() == h0
    (d / "k_decode_tc.cu").write_text(text.replace("constexpr int kBN = 64;", "constexpr int kBN = 32;"))
    assert bench._kernel_hash() != h0


def test_paged_block_table_is_a_permutation_of_the_needed_pages():
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    lens = np.array([4096, 1, 64, 65, 0, 130])
    table, num_pages = bench.paged_block_table(lens, seed=3)
    need = [-(-int(n) // 64) for n in lens]
    assert num_pages == sum(need) and table.shape == (len(lens), max(need))
    used = np.concatenate([table[b, :k] for b, k in enumerate(need)])
    assert sorted(used.tolist()) == list(range(num_pages))   # every page once, no sharing
    assert not np.array_equal(used, np.arange(num_pages))    # shuffled, not the contiguous order
    t2, _ = bench.paged_block_table(lens, seed=3)
    assert np.array_equal(table, t2)                          # seeded


def test_kv_down_bench_accounting():
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import mla_workloads as W
    cfg = W.WORKLOADS["kvdown_b32_d7168"]
    seq, pos, B, N = bench.kvdown_rows_slots(cfg)
    assert (B, N) == (32, 4096) and np.array_equal(seq, np.arange(32)) and np.all(pos == 4095)
    nbytes, flops = bench.kvdown_bytes_flops(cfg)
    # W once (7168 x 576 bf16) + h (32 x 7168) + gamma (512) + 32 rows of 576
    assert nbytes == 2 * (7168 * 576 + 32 * 7168 + 512 + 32 * 576)
    assert flops == 2 * 32 * 7168 * 576
    cfg = W.WORKLOADS["kvdown_t32768_d7168"]
    seq, pos, B, N = bench.kvdown_rows_slots(cfg)
    assert len(seq) == cfg["T"] == B * N and len(set(zip(seq.tolist(), pos.tolist()))) == cfg["T"]


def test_decode_step_roofline_accounting():
    # the whole step adds W_UK and W_UV (2 x 128 x 128 x 512 bf16 = 33.6 MB) to the
    # cache read, and the absorb and up-projection contractions (2 B H (d_k + d_v) d_c
    # = 1.07 GFLOP) to the attention's FLOPs; the gated step adds W_g and its GEMM
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import mla_workloads as W
    cfg = W.WORKLOADS["decode_h128_b32_n4096"]
    lens = W.seq_lens(cfg, 0)
    b_att, f_att = bench.workload_bytes_flops(cfg, lens)
    b_step, f_step = bench.step_bytes_flops(cfg, lens)
    assert b_att == 150_994_944 and b_step - b_att == 33_554_432
    assert f_step - f_att == 1_073_741_824
    g = W.WORKLOADS["gated_h64_b16_n131072"]
    lens = W.seq_lens(g, 0)
    b_att, f_att = bench.workload_bytes_flops(g, lens)
    b_step, f_step = bench.step_bytes_flops(g, lens)
    assert b_step - b_att == 64 * 256 * 512 * 2 + 4096 * 8192 * 2
    assert f_step - f_att == 2 * 16 * 64 * 256 * 512 + 2 * 16 * 4096 * 8192
    assert np.isclose(b_att, 16 * 131072 * 512 * 2)
