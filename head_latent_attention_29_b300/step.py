"""CUDA-graph runner for one MLA decode step.

A decode step launches four or five short kernels for a bf16 cache (the new
rows appended by the absorb launch, split-KV attention, combine, out-up,
optionally the gate; an fp32 cache takes separate append and absorb kernels and
a one-kernel attention).  At ~tens of microseconds per
step the host-side launch cost matters, so the step is captured once into a CUDA
graph over static buffers and replayed.  Every kernel in the graph is a libmla
kernel; the graph only removes host launch overhead.
"""
from __future__ import annotations

import torch

from . import LatentCache, PagedLatentCache, absorb_q_append, decode_attn, decode_attn_paged, decode_workspace, gate, \
    out_up


class DecodeStep:
    """Static buffers + captured graph of one decode step over `cache` (a
    LatentCache, or a PagedLatentCache whose block table covers every sequence).

    Step inputs (device, static): c_kv [B, d_c], k_r [B, d_r], q_nope [B, H, d_k],
    q_rope [B, H, d_r], optional h [B, d_model]; the new token of sequence b is
    written at position seq_lens[b] - 1 and attends to seq_lens[b] tokens.
    Output: o [B, H, d_v] (gated in place when W_g is given)."""

    def __init__(self, cache: LatentCache | PagedLatentCache, w_uk: torch.Tensor, w_uv: torch.Tensor,
                 seq_lens: torch.Tensor, scale: float, rope_base: float = 10000.0, w_g: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None):
        dev = cache.data.device
        self.cache, self.w_uk, self.w_uv, self.w_g = cache, w_uk, w_uv, w_g
        self.scale, self.rope_base = float(scale), float(rope_base)
        B, H, d_c, d_r = cache.B, w_uk.shape[0], cache.d_c, cache.d_r
        d_k, d_v = w_uk.shape[1], w_uv.shape[1]
        dt = cache.dtype
        self.B, self.H = B, H
        self.seq_lens = seq_lens
        self.seq_idx = torch.arange(B, dtype=torch.int32, device=dev)
        self.pos = (seq_lens - 1).clamp(min=0).to(torch.int32)
        self.inputs = {
            "c_kv": torch.zeros((B, d_c), dtype=dt, device=dev),
            "k_r": torch.zeros((B, max(d_r, 1)), dtype=dt, device=dev)[:, :d_r].contiguous() if d_r else None,
            "q_nope": torch.zeros((B, H, d_k), dtype=dt, device=dev),
            "q_rope": torch.zeros((B, H, d_r), dtype=dt, device=dev) if d_r else None,
        }
        if w_g is not None:
            self.inputs["h"] = torch.zeros((B, w_g.shape[0]), dtype=dt, device=dev)
        self.inputs = {k: v for k, v in self.inputs.items() if v is not None}
        self.q_cat = torch.empty((B, H, d_c + d_r), dtype=dt, device=dev)
        self.ws = decode_workspace(B, H, d_c, dt, dev)
        self.o_lat = torch.empty((B, H, d_c), dtype=dt, device=dev)
        self.lse = torch.empty((B, H), dtype=torch.float32, device=dev)
        self.o = torch.empty((B, H, d_v), dtype=dt, device=dev)
        # bf16: absorb + append, split attention, combine, out-up; fp32: append,
        # absorb, attention, out-up (a bf16 batch of at most four sequences adds the
        # grouped merge's second kernel when each sequence is cut into 16 or more
        # pieces; not counted here)
        self.kernels_per_step = 4 + (1 if w_g is not None else 0)
        self.graph = None
        self.stream = stream

    def launch(self) -> None:
        """Queue the step's kernels on the current stream (no graph)."""
        d = self.inputs
        attend = decode_attn_paged if isinstance(self.cache, PagedLatentCache) else decode_attn
        # the new rows and the absorbed queries in one call (one launch for bf16)
        absorb_q_append(self.cache, d["c_kv"], d.get("k_r"), self.seq_idx, self.pos, d["q_nope"], d.get("q_rope"),
                        self.pos, self.w_uk, self.rope_base, out=self.q_cat)
        attend(self.q_cat, self.cache, self.seq_lens, self.scale, self.ws, self.o_lat, self.lse)
        out_up(self.o_lat, self.w_uv, out=self.o)
        if self.w_g is not None:
            gate(d["h"], self.w_g, self.o.view(self.B, -1))

    def capture(self, host_inputs: dict | None = None, host_out: torch.Tensor | None = None) -> None:
        """Capture the step (optionally with pinned host->device input copies and a
        device->host output copy) into a CUDA graph.  The kernels must have run
        once before capture (launch()) so that one-time host setup is done."""
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            if host_inputs is not None:
                for k, v in host_inputs.items():
                    self.inputs[k].copy_(v, non_blocking=True)
            self.launch()
            if host_out is not None:
                host_out.copy_(self.o, non_blocking=True)

    def replay(self) -> None:
        self.graph.replay()
