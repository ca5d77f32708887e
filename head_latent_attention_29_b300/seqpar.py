"""Decode sharded by sequence position across processes, one GPU each.

Every rank holds a contiguous share of the rows of every sequence (rank r: rows
[begin_r[b], end_r[b]) of sequence b).  For a decode step each rank computes the
attention of the (replicated) absorbed queries over its own rows only -- a partial
in log-sum-exp form, (o_r, lse_r) -- gathers every rank's partial into local
buffers with one all-gather per tensor, and merges them with the library's
log-sum-exp merge, which gives exactly the attention over all rows.  This is the
exchange step of sequence-parallel decode (the sequence-parallel remark of the
0539edu.com MLA page, section 8): the cache never moves, only B x H x (d_c + 1)
values per rank and step do.

The host path is written against torch.distributed (NCCL between GPUs; gloo on
CPU for its tests).  The per-rank compute is injectable so that the orchestration
can be exercised without a GPU; by default it is the library's
decode_attn_partial / decode_merge (or decode_attn over a rank-local cache that
holds only the rank's rows).
"""
from __future__ import annotations

from typing import Callable

import numpy as np
import torch


def shard_rows(lens, world: int, rank: int, align: int = 64) -> tuple[np.ndarray, np.ndarray]:
    """Rank `rank`'s rows of each sequence: [begin, end) with the n rows of a sequence
    cut into `world` contiguous shares of whole `align`-row blocks (the last shares
    may be shorter or empty).  The shares of all ranks cover [0, n) exactly once."""
    lens = np.asarray(lens, dtype=np.int64)
    if world < 1 or not (0 <= rank < world):
        raise ValueError("rank must lie in [0, world)")
    blocks = (lens + align - 1) // align
    per = (blocks + world - 1) // world            # blocks per share, rounded up
    begin = np.minimum(rank * per * align, lens)
    end = np.minimum((rank + 1) * per * align, lens)
    return begin.astype(np.int32), end.astype(np.int32)


class SeqShardedDecode:
    """One rank's side of a sequence-sharded decode step.

    attend(q_cat, rows, out, lse) -> (o_part, lse_part): this rank's partial over its
        rows (writes into `out` [B, H, d_c] and `lse` [B, H] fp32 when given).
    merge(o_parts, lse_parts) -> (o_lat, lse): the log-sum-exp merge of the gathered
        partials [world, B, H, d_c] / [world, B, H].
    The gather buffers are allocated once; the partial is written straight into this
    rank's slot, so the all-gather moves only the other ranks' data into place."""

    def __init__(self, B: int, H: int, d_c: int, world: int, rank: int, dtype=torch.bfloat16,
                 device="cuda", group=None, attend: Callable | None = None, merge: Callable | None = None,
                 lse_dtype=torch.float32):
        self.B, self.H, self.d_c, self.world, self.rank, self.group = B, H, d_c, world, rank, group
        self.o_all = torch.empty((world, B, H, d_c), dtype=dtype, device=device)
        self.lse_all = torch.empty((world, B, H), dtype=lse_dtype, device=device)
        self.attend, self.merge = attend, merge

    def step(self, q_cat, rows):
        """Partial on this rank's rows, all-gather, merge: returns (o_lat, lse)."""
        mine_o, mine_lse = self.o_all[self.rank], self.lse_all[self.rank]
        o_part, lse_part = self.attend(q_cat, rows, mine_o, mine_lse)
        if o_part.data_ptr() != mine_o.data_ptr():
            mine_o.copy_(o_part)
        if lse_part.data_ptr() != mine_lse.data_ptr():
            mine_lse.copy_(lse_part)
        if self.world > 1:
            import torch.distributed as dist
            # every rank contributes its own slot; the output is the whole buffer
            dist.all_gather_into_tensor(self.o_all.view(self.world * self.B, self.H, self.d_c), mine_o.clone(),
                                        group=self.group)
            dist.all_gather_into_tensor(self.lse_all.view(self.world * self.B, self.H), mine_lse.clone(),
                                        group=self.group)
        return self.merge(self.o_all, self.lse_all)


def library_attend(cache, scale: float, row_begin: torch.Tensor | None = None, row_end: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None):
    """attend() for SeqShardedDecode on the GPU: with row_begin/row_end, this rank's
    rows of a cache that holds whole sequences (decode_attn_partial); without them, a
    rank-local cache that holds only this rank's rows (decode_attn over its lengths,
    passed as `rows`)."""
    from . import decode_attn, decode_attn_partial

    def attend(q_cat, rows, out, lse):
        if row_begin is not None:
            return decode_attn_partial(q_cat, cache, row_begin, row_end, scale, workspace, out, lse)
        return decode_attn(q_cat, cache, rows, scale, workspace, out, lse)
    return attend


def library_merge(out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """merge() for SeqShardedDecode on the GPU: the library's log-sum-exp merge."""
    from . import decode_merge

    def merge(o_all, lse_all):
        return decode_merge(o_all, lse_all, out, lse)
    return merge
