"""Sequence-sharded decode, host side on CPU: the row shares of the ranks cover
every sequence exactly once, and two gloo ranks that each attend over their own
rows, all-gather the partials and merge them reproduce the unsharded attention.
The per-rank compute is the float64 oracle's partial (0539edu.com section 8:
sequence-parallel decode; hotelren.com section 7.3: the max-subtracted softmax
across row subsets)."""
from __future__ import annotations

import math
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_rows_cover_each_sequence_once(world):
    from head_latent_attention_29_b300.seqpar import shard_rows
    lens = np.array([0, 1, 63, 64, 65, 4096, 5000, 130], dtype=np.int32)
    seen = np.zeros((len(lens), int(lens.max())), dtype=np.int32)
    for r in range(world):
        b, e = shard_rows(lens, world, r)
        assert np.all(b <= e) and np.all(e <= lens)
        assert np.all((b % 64 == 0) | (b == lens))  # shares start on whole 64-row blocks
        for i in range(len(lens)):
            seen[i, b[i]:e[i]] += 1
    for i, n in enumerate(lens):
        assert np.all(seen[i, :n] == 1) and np.all(seen[i, n:] == 0)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(B=3, H=4, d_c=32, d_r=8, seed=5):
    rng = np.random.default_rng(seed)
    lens = np.array([300, 65, 1000][:B], dtype=np.int32)
    q = rng.standard_normal((B, H, d_c + d_r))
    rows = [rng.standard_normal((int(n), d_c + d_r)) for n in lens]
    return lens, q, rows, 1.0 / math.sqrt(16 + d_r)


def _rank_main(rank, world, port, q_out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from head_latent_attention_29_b300.seqpar import SeqShardedDecode, shard_rows
    from oracle import mla_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lens, q, rows, scale = _inputs()
        B, H, R = q.shape
        d_c = 32
        begin, end = shard_rows(lens, world, rank)

        def attend(q_cat, _rows, out, lse):
            # this rank's partial over its rows, in log-sum-exp form
            for b in range(B):
                if end[b] > begin[b]:
                    m, l, o_un = O.decode_partial(q_cat[b], rows[b][begin[b]:end[b]], d_c, scale)
                    out[b] = torch.from_numpy(o_un / l[:, None])
                    lse[b] = torch.from_numpy(m + np.log(l))
                else:
                    out[b] = 0.0
                    lse[b] = -math.inf
            return out, lse

        def merge(o_all, lse_all):
            parts = [(lse_all[s].double().numpy(), np.ones((B, H)), o_all[s].double().numpy()) for s in range(world)]
            outs, lses = [], []
            for b in range(B):
                o_b, l_b = O.lse_merge([(p[0][b], p[1][b], p[2][b]) for p in parts
                                        if np.isfinite(p[0][b]).all()])
                outs.append(o_b)
                lses.append(l_b)
            return np.stack(outs), np.stack(lses)

        sd = SeqShardedDecode(B, H, d_c, world, rank, dtype=torch.float64, device="cpu", attend=attend, merge=merge,
                              lse_dtype=torch.float64)
        o, lse = sd.step(q, None)
        q_out.put((rank, o, lse, [int(x) for x in begin], [int(x) for x in end]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_merge_to_the_unsharded_attention():
    from oracle import mla_oracle as O
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q_out)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted([q_out.get(timeout=180) for _ in range(world)], key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    lens, q, rows, scale = _inputs()
    # the ranks held different rows ...
    assert results[0][3] != results[1][3]
    for rank, o, lse, _, _ in results:
        for b in range(len(lens)):
            ref_o, ref_lse = O.decode_absorbed(q[b], rows[b], 32, scale)
            # ... and every rank ends with the attention over all rows of every sequence
            np.testing.assert_allclose(o[b], ref_o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-12, atol=1e-12)
