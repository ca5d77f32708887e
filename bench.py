"""MLA decode benchmark (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]
                    [--workload decode_h128_b32_n4096] [--paged]

A step is one decode step of the whole hot path for every sequence of the batch:
append the new token's latent row (RoPE on its key), absorb W_UK into the query,
latent attention over the cache (split-KV runs + log-sum-exp combine), and the
W_UV up-projection (plus the output gate for the gated workload).  `value` is
decoded tokens per second over the whole job with inputs resident in HBM; `e2e`
is the same metric with the step's inputs copied from pinned host memory and the
result copied back inside the timed region.

Several copies of the latent cache rotate between steps (total well above the
126 MB L2), so every step reads its cache from HBM.

With --gpus N > 1 (launched by torch.distributed.run) every rank runs an
independent replica of the workload: the decode path has no cross-sequence
exchange, so batches are data-parallel (weak scaling, no collective on the data
path).

`--impl reference` times the float64 CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).

Other workloads (see mla_workloads): ragged and gated decode steps; prefill
steps (`prefill_*`: append the prompt rows, absorb every query, causal prefill
attention, W_UV); and the new tokens' cache rows straight from hidden states
(`kvdown_*`: projection, RMSNorm, RoPE, append).  `--paged` runs a decode
workload over a paged cache (64-row pages of one pool in shuffled order).  The
decode line carries the attention op's roofline (`roofline`, with the ncu DRAM
traffic when the stored counters match the kernel source) and the whole step's
(`step_roofline`).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import mla_workloads as W  # noqa: E402

ROTATE = 4  # default number of cache copies rotated between steps

THROTTLE_BITS = {
    0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
    0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x10: "sync_boost",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)) or None, "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# ---------------------------------------------------------------- clocks (NVML)
class ClockSampler:
    """SM clock and clock-event reasons during the timed region: NVML when the
    Python module is present, else an nvidia-smi sampling subprocess; the GPU is
    selected by UUID (NVML ignores CUDA_VISIBLE_DEVICES).  Every sample carries
    its host time; the sampler is running before the region starts and keeps
    going until a sample after its end has arrived, so a region shorter than the
    sampling period is still bracketed by the samples on either side."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
    SMI_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.02):
        self.samples = []  # (host time, SM MHz, reason names)
        self.max_mhz = None
        self._stop = threading.Event()
        self._period = period_s
        self._mode = None
        self.error = None
        self._uuid = None
        self._t0 = self._t1 = None
        try:
            import torch
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self._uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception as e:
            self.error = repr(e)[:200]
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByUUID(self._uuid) if self._uuid else \
                pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self._reasons_fn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._mode = "nvml"
        except Exception as e:
            self.error = repr(e)[:200]
            import shutil
            if shutil.which("nvidia-smi") and self._uuid:
                self._mode = "smi"

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                mhz = self._nv.nvmlDeviceGetClockInfo(self._h, self._nv.NVML_CLOCK_SM)
                bits = int(self._reasons_fn(self._h))
                self.samples.append((time.perf_counter(), float(mhz),
                                     [n for bit, n in THROTTLE_BITS.items() if bits & bit]))
            except Exception as e:
                self.error = repr(e)[:200]
            time.sleep(self._period)

    def _run_smi(self):
        for line in self._p.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                mhz, self.max_mhz = float(f[0]), float(f[1])
            except ValueError:
                continue
            names = [n for n, v in zip(self.SMI_REASONS, f[3:7]) if v.lower() in ("active", "1", "yes")]
            self.samples.append((time.perf_counter(), mhz, names))

    def _wait_for_sample_after(self, t, limit_s):
        end = time.perf_counter() + limit_s
        while time.perf_counter() < end:
            if self.samples and self.samples[-1][0] > t:
                return
            time.sleep(0.002)

    def __enter__(self):
        if self._mode == "nvml":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
        elif self._mode == "smi":
            import subprocess
            self._p = subprocess.Popen(["nvidia-smi", "-i", self._uuid, f"--query-gpu={self.SMI_FIELDS}",
                                        "--format=csv,noheader,nounits", f"-lms={int(self._period * 1000)}"],
                                       stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._run_smi, daemon=True)
        if self._mode:
            self._t.start()
            self._wait_for_sample_after(0.0, 5.0)  # sampling is live before the region starts
        self._t0 = time.perf_counter()
        return self

    def __exit__(self, *exc):
        self._t1 = time.perf_counter()
        if self._mode:
            self._wait_for_sample_after(self._t1, 2.0)
        if self._mode == "nvml":
            self._stop.set()
            self._t.join()
        elif self._mode == "smi":
            self._p.terminate()
            try:
                self._p.wait(timeout=10)
            except Exception:  # pragma: no cover
                self._p.kill()
            self._t.join(timeout=5)

    def window(self):
        """The samples taken inside the region; if it was shorter than the sampling
        period, the last sample before it and the first after it."""
        inside = [x for x in self.samples if self._t0 <= x[0] <= self._t1]
        if inside:
            return inside, "inside"
        before = [x for x in self.samples if x[0] < self._t0][-1:]
        after = [x for x in self.samples if x[0] > self._t1][:1]
        return before + after, "adjacent"

    def summary(self):
        got, where = self.window() if self._t0 is not None else ([], "none")
        if not got:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "error": self.error}
        names = sorted({n for x in got for n in x[2]})
        return {"sm_mhz": statistics.median(x[1] for x in got), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(got), "window": where, "source": self._mode}


# ---------------------------------------------------------------- workload
ATTN_WARMUP = 20
ATTN_REPS = 200


def time_attention(replay, stream, device, launches_per_replay: int = 10):
    """Median per-launch time (us) of the attention op over ATTN_REPS graph replays
    after ATTN_WARMUP, each replay bracketed by CUDA events on the launching stream;
    also the spread and the SM clock seen during the replays, with the median time
    scaled to the maximum SM clock (time x median MHz / max MHz)."""
    import torch
    for _ in range(ATTN_WARMUP):
        replay()
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(ATTN_REPS + 1)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize(device)
        ev[0].record(stream)
        for i in range(ATTN_REPS):
            replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(device)
    per = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 / launches_per_replay for i in range(ATTN_REPS))
    med = statistics.median(per)
    ck = clk.summary()
    at_max = None
    if ck.get("sm_mhz") and ck.get("sm_max_mhz"):
        at_max = round(med * ck["sm_mhz"] / ck["sm_max_mhz"], 3)
    q = lambda f: round(per[min(len(per) - 1, int(f * len(per)))], 3)
    return {"us": med, "timing": {
        "replays": ATTN_REPS, "launches_per_replay": launches_per_replay, "warmup_replays": ATTN_WARMUP,
        "median_us": round(med, 3), "mean_us": round(statistics.fmean(per), 3), "min_us": round(per[0], 3),
        "p10_us": q(0.1), "p90_us": q(0.9), "max_us": round(per[-1], 3),
        "median_us_at_max_clock": at_max, "clocks": ck}}


def time_seqpar(wl, k: int, stream, device) -> dict:
    """Decode sharded by sequence position on this one GPU: shard 0's partial (its
    share of every sequence's rows, `seqpar.shard_rows`) and the merge of k partials,
    each timed as the attention op is (ten-launch graphs over the rotating caches).
    A k-GPU run adds the all-gather of the partials between the two."""
    import torch
    from head_latent_attention_29_b300.seqpar import shard_rows
    mla, B, H = wl.mla, wl.B, wl.H
    b0, b1 = shard_rows(wl.lens, k, 0)
    begin, end = torch.from_numpy(b0).to(device), torch.from_numpy(b1).to(device)
    scale = wl.cfg["scale"]
    d_c = wl.steps[0].o_lat.shape[-1]
    o_p = [torch.empty((B, H, d_c), dtype=torch.bfloat16, device=device) for _ in wl.steps]
    l_p = [torch.empty((B, H), dtype=torch.float32, device=device) for _ in wl.steps]
    for st, o, l in zip(wl.steps, o_p, l_p):  # eager once: one-time host setup outside capture
        mla.decode_attn_partial(st.q_cat, st.cache, begin, end, scale, st.ws, out=o, lse=l)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(10):
            j = i % len(wl.steps)
            st = wl.steps[j]
            mla.decode_attn_partial(st.q_cat, st.cache, begin, end, scale, st.ws, out=o_p[j], lse=l_p[j])
    part = time_attention(g.replay, stream, device)
    o_parts = torch.stack([o_p[0]] * k)
    l_parts = torch.stack([l_p[0]] * k)
    o_m = torch.empty((B, H, d_c), dtype=torch.bfloat16, device=device)
    l_m = torch.empty((B, H), dtype=torch.float32, device=device)
    mla.decode_merge(o_parts, l_parts, out=o_m, lse=l_m)
    torch.cuda.synchronize(device)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        for _ in range(10):
            mla.decode_merge(o_parts, l_parts, out=o_m, lse=l_m)
    mer = time_attention(g2.replay, stream, device)
    st, word = mla.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} ({word:#x}) in the sequence-sharded timing")
    return {"shards": k, "shard_timed": 0, "rows_of_shard": int(np.sum(b1 - b0)),
            "partial_us": round(part["us"], 3), "merge_us": round(mer["us"], 3),
            "per_gpu_us_without_collective": round(part["us"] + mer["us"], 3),
            "collective": (f"all-gather of {k} partials (o bf16 [B,H,{d_c}] + lse fp32 [B,H]) between the "
                           "partial and the merge: not measured, one GPU per box")}


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over all ranks (the slowest replica sets the job's
    time); no collective for a single process."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds_per_step: float) -> float:
    """Whole-job rate: the units all replicas processed in one step over the
    slowest replica's step time."""
    return units_per_rank * world / seconds_per_step


def decode_metric(workload: str, cfg) -> str:
    """The metric's name: the headline decode shape keeps its published wording, the
    other decode shapes spell out their own sizes."""
    if workload == "decode_h128_b32_n4096":
        return "MLA decode tokens/s at H=128,d_c=512,B=32,N=4K bf16; % of roofline"
    n = f"N={cfg['N']}" if "N" in cfg else f"N={cfg['N_lo']}..{cfg['N_hi']} (ragged)"
    extra = "" if cfg["d_r"] else ", no RoPE"
    extra += ", output gate" if "d_model" in cfg else ""
    return f"MLA decode tokens/s at H={cfg['H']},d_c={cfg['d_c']},B={cfg['B']},{n}{extra} bf16; % of roofline"


def workload_bytes_flops(cfg, lens):
    R = cfg["d_c"] + cfg["d_r"]
    tokens = int(np.sum(lens))
    bytes_attn = tokens * R * 2
    flops_attn = tokens * cfg["H"] * (2 * R + 2 * cfg["d_c"])
    return bytes_attn, flops_attn


def step_bytes_flops(cfg, lens):
    """Algorithmic bytes and FLOPs of the whole decode step: the attention's cache
    read plus the weights the step streams once (W_UK and W_UV, and W_g for the
    gated workload), and the absorb, up-projection and gate contractions."""
    B, H, d_c, d_k, d_v = cfg["B"], cfg["H"], cfg["d_c"], cfg["d_k"], cfg["d_v"]
    nbytes, flops = workload_bytes_flops(cfg, lens)
    nbytes += H * (d_k + d_v) * d_c * 2
    flops += 2 * B * H * (d_k + d_v) * d_c
    if cfg["d_r"] == 0 and "d_model" in cfg:
        nbytes += cfg["d_model"] * H * d_v * 2
        flops += 2 * B * cfg["d_model"] * H * d_v
    return nbytes, flops


def paged_block_table(lens, seed: int, page_rows: int = 64):
    """Block table [B, max_blocks] int32 giving each sequence's 64-row blocks
    distinct pages of one pool in a seeded random order (how pages end up after
    sequences of a serving batch have grown and finished at different times), and
    the pool size (exactly the pages the lengths need)."""
    need = [-(-int(n) // page_rows) for n in lens]
    max_blocks = max(1, max(need))
    num_pages = max(1, sum(need))
    perm = np.random.default_rng([seed, 0x9A6E]).permutation(num_pages).astype(np.int32)
    table = np.zeros((len(lens), max_blocks), dtype=np.int32)
    k = 0
    for b, nb in enumerate(need):
        table[b, :nb] = perm[k:k + nb]
        k += nb
    return table, num_pages


class DeviceWorkload:
    """Resident inputs of one replica: ROTATE latent caches, each with a captured
    decode-step graph, shared weights and the step's pinned host inputs."""

    def __init__(self, name: str, seed: int, device, rotate: int = ROTATE, paged: bool = False):
        import torch
        import head_latent_attention_29_b300 as mla
        from head_latent_attention_29_b300.step import DecodeStep
        self.mla, self.torch = mla, torch
        cfg = dict(W.WORKLOADS[name])
        self.cfg, self.name = cfg, name
        self.lens = W.seq_lens(cfg, seed)
        B, H, d_c, d_r = cfg["B"], cfg["H"], cfg["d_c"], cfg["d_r"]
        self.B, self.H = B, H
        N_max = int(self.lens.max())
        bf = torch.bfloat16
        rb = cfg.get("rope_base", 1e4)

        def up(x):
            return torch.from_numpy(np.ascontiguousarray(W.bf16_bits(x)).view(np.int16)).view(bf).to(device)

        def pin(x):
            return torch.from_numpy(np.ascontiguousarray(W.bf16_bits(x)).view(np.int16)).view(bf).pin_memory()

        # cache copy 0 is filled from the seeded draws through the library's own
        # append (RoPE on the key); the other copies are device-side clones.  The
        # paged variant draws every sequence's pages from one pool in shuffled order.
        self.paged = paged
        if paged:
            table, num_pages = paged_block_table(self.lens, seed)
            table = torch.from_numpy(table).to(device)

            def new_cache(data=None):
                return mla.PagedLatentCache(num_pages, B, table.shape[1], d_c, d_r, dtype=bf, device=device,
                                            block_table=table, data=data)
            append = mla.cache_append_paged
        else:
            def new_cache(data=None):
                return mla.LatentCache(B, N_max, d_c, d_r, dtype=bf, device=device, data=data)
            append = mla.cache_append
        c0 = new_cache()
        for b in range(B):
            n = int(self.lens[b])
            c, k = W.latent_rows(cfg, seed, b, n)
            idx = torch.full((n,), b, dtype=torch.int32, device=device)
            pos = torch.arange(n, dtype=torch.int32, device=device)
            append(c0, up(c), up(k) if d_r else None, idx, pos, rb)
        self.rotate = rotate
        caches = [c0] + [new_cache(c0.data.clone()) for _ in range(rotate - 1)]
        w_uk, w_uv = W.up_weights(cfg, seed)
        w_uk, w_uv = up(w_uk), up(w_uv)
        self.gated = d_r == 0 and "d_model" in cfg
        w_g = None
        q_nope, q_r = W.query(cfg, seed)
        self.host = {"c_kv": pin(W.normal(seed, "step_c_kv", (B, d_c))), "q_nope": pin(q_nope[:, 0])}
        if d_r:
            self.host["k_r"] = pin(W.normal(seed, "step_k_r", (B, d_r)))
            self.host["q_rope"] = pin(q_r[:, 0])
        if self.gated:
            h, wg = W.gate_inputs(cfg, seed)
            self.host["h"] = pin(h)
            w_g = up(wg)
        seq_lens = torch.from_numpy(self.lens).to(device)
        self.steps = [DecodeStep(c, w_uk, w_uv, seq_lens, cfg["scale"], rb, w_g) for c in caches]
        for st in self.steps:
            for k, v in self.host.items():
                st.inputs[k].copy_(v)
            st.launch()  # one eager run: one-time host setup happens outside capture
        torch.cuda.synchronize(device)
        for st in self.steps:
            st.capture()
        # end-to-end variant: H2D of the step inputs and D2H of the output inside the graph
        # (one pinned output per cache copy: two steps may be in flight at once)
        self.o_hosts = [torch.empty(tuple(self.steps[0].o.shape), dtype=bf).pin_memory() for _ in caches]
        self.e2e = [DecodeStep(c, w_uk, w_uv, seq_lens, cfg["scale"], rb, w_g) for c in caches]
        for st in self.e2e:
            st.launch()
        torch.cuda.synchronize(device)
        for st, o_host in zip(self.e2e, self.o_hosts):
            st.capture(self.host, o_host)
        # attention alone, ten launches per graph over the rotating caches
        self.attn_graph = torch.cuda.CUDAGraph()
        s0 = self.steps[0]
        with torch.cuda.graph(self.attn_graph):
            attend = mla.decode_attn_paged if paged else mla.decode_attn
            for i in range(10):
                st = self.steps[i % rotate]
                attend(st.q_cat, st.cache, seq_lens, cfg["scale"], st.ws, st.o_lat, st.lse)
        self.kernels_per_step = s0.kernels_per_step
        # the timed graph: one step per cache copy, back to back, as a model's layers
        # issue them (programmatic launch between steps, no graph launch in between);
        # a replay is `rotate` steps
        self.graph_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_all):
            for st in self.steps:
                st.launch()

    def step(self, i: int):
        """One step alone: its own graph replay."""
        self.steps[i % self.rotate].replay()

    def replay_all(self):
        """`rotate` steps in one graph replay."""
        self.graph_all.replay()


def run_b300(args, rank, world, device):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(device)
    wl = DeviceWorkload(args.workload, args.seed + rank, device, args.rotate, getattr(args, "paged", False))
    cfg = wl.cfg
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            dist.barrier()

    for i in range(max(1, math.ceil(args.warmup / wl.rotate))):
        wl.replay_all()
    torch.cuda.synchronize(device)

    # ---- device-resident throughput: K whole steps, `rotate` per graph replay
    replays = max(1, math.ceil(args.steps / wl.rotate))
    steps_done = replays * wl.rotate
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(replays):
            wl.replay_all()
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, device)
    ms_step = ms_total / steps_done

    # ---- the same steps with one graph replay each (a graph launch between steps)
    n_single = max(4 * wl.rotate, min(args.steps, 400))
    for i in range(wl.rotate):
        wl.step(i)
    torch.cuda.synchronize(device)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(n_single):
        wl.step(i)
    s1.record(stream)
    torch.cuda.synchronize(device)
    ms_single = max_over_ranks(s0.elapsed_time(s1), world, device) / n_single
    tokens_per_step = wl.B * world
    value = job_throughput(wl.B, world, ms_step * 1e-3)

    # ---- dominant op (attention: split-KV kernel + combine), timed alone on its stream:
    # 20 warm-up replays, then ATTN_REPS replays of a ten-launch graph (whatever
    # --steps is), each bracketed by events; the median replay gives the time
    attn = time_attention(wl.attn_graph.replay, stream, device)
    attn_us = attn["us"]
    seqpar = time_seqpar(wl, args.seq_shards, stream, device) if getattr(args, "seq_shards", 0) > 1 else None

    # ---- end to end: pinned inputs in, result out, the host reads every step's result
    n_e2e = 2000  # whatever --steps is: host-side jitter and the pipeline fill average out
    for i in range(3):
        wl.e2e[i % wl.rotate].replay()
    torch.cuda.synchronize(device)
    # (a) one step at a time: the host waits for each step before queueing the next
    barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        wl.e2e[i % wl.rotate].replay()
        torch.cuda.current_stream(device).synchronize()
    barrier()
    e2e_serial_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device)
    # (b) one batch per cache copy in flight, each on its own stream, as a server
    # interleaves independent groups of sequences: the steps' copies overlap other
    # steps' kernels, and the host waits for each step's result `rotate` steps behind.
    # Steps that share a cache copy and its buffers (i = j mod rotate) share a
    # stream, so they stay ordered.
    e2e_s, in_flight = e2e_serial_s, 1
    if wl.rotate > 1:
        streams = [torch.cuda.Stream(device) for _ in range(wl.rotate)]

        def pipelined(n):
            pending = []
            for i in range(n):
                s = streams[i % wl.rotate]
                with torch.cuda.stream(s):
                    wl.e2e[i % wl.rotate].replay()
                ev = torch.cuda.Event()
                ev.record(s)
                pending.append(ev)
                if len(pending) == wl.rotate:
                    pending.pop(0).synchronize()
            for ev in pending:
                ev.synchronize()

        pipelined(4 * wl.rotate)  # warm-up
        torch.cuda.synchronize(device)
        barrier()
        t0 = time.perf_counter()
        pipelined(n_e2e)
        barrier()
        e2e_s, in_flight = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device), wl.rotate
        torch.cuda.synchronize(device)
    h2d = sum(v.numel() * v.element_size() for v in wl.host.values())
    d2h = wl.o_hosts[0].numel() * wl.o_hosts[0].element_size()

    hbm, tc_burst, tc_sust, peak_kind = _peaks()
    bytes_attn, flops_attn = workload_bytes_flops(cfg, wl.lens)
    achieved_gbs = bytes_attn / (attn_us * 1e-6) / 1e9
    t_mem = bytes_attn / (hbm * 1e9)
    t_tc = flops_attn / (tc_burst * 1e12)
    roof_us = max(t_mem, t_tc) * 1e6
    traffic = None if wl.paged else _ncu_traffic(args.workload)  # counters were taken on the contiguous cache
    step_bytes, step_flops = step_bytes_flops(cfg, wl.lens)
    step_roof_us = max(step_bytes / (hbm * 1e9), step_flops / (tc_burst * 1e12)) * 1e6

    out = {
        "metric": decode_metric(args.workload, cfg),
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps_done,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "ms_per_step_single_replay": round(ms_single, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) latents/keys/queries, N(0,1/512) up-projections)",
        "config": {
            "workload": args.workload, "B": cfg["B"], "H": cfg["H"], "d_c": cfg["d_c"], "d_r": cfg["d_r"],
            "d_k": cfg["d_k"], "d_v": cfg["d_v"], "tokens_cached": int(np.sum(wl.lens)),
            "parallelism": f"replicas x{world}",
            "l2": f"{wl.rotate} rotating cache copies ({wl.rotate * bytes_attn / 1e6:.0f} MB vs 126 MB L2)",
            "timing": (f"{wl.rotate} steps per graph replay, each on its own cache copy, back to back as a "
                       "model's layers issue them; ms_per_step_single_replay: one step per graph replay"),
            "step": "absorb_q_append(append + absorb in one launch)+decode_attn(split+combine)+out_up" + ("+gate" if wl.gated else ""),
            "cache": "paged (64-row pages, shuffled block table)" if wl.paged else "contiguous [B, N_max, 576]",
        },
        "gpu_launches": wl.kernels_per_step * steps_done,
        "e2e": {"value": round(tokens_per_step / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps_in_flight": in_flight,
                "value_one_step_at_a_time": round(tokens_per_step / e2e_serial_s, 1),
                "how": ("DecodeStep graphs with the pinned-input copies, the step's kernels and the output "
                        "copy; the host reads every step's result; with several in flight, each step "
                        "(an independent batch on its own cache copy) runs on that copy's stream")},
        "roofline": {
            "bound": "hbm", "kernel": "decode_attn (split-KV tensor-core kernel + combine)",
            "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved_gbs / hbm, 4), "traffic": traffic,
            "peak_source": f"{peak_kind} hbm_gbs",
            "attn_us": round(attn_us, 3), "algorithmic_bytes": bytes_attn, "algorithmic_flops": flops_attn,
            "tflops": round(flops_attn / (attn_us * 1e-6) / 1e12, 1),
            "roofline_us": round(roof_us, 3), "frac_of_roofline": round(roof_us / attn_us, 4),
            "frac_of_roofline_sustained_tc": (round(max(t_mem, flops_attn / (tc_sust * 1e12)) * 1e6 / attn_us, 4)
                                              if tc_sust else None),
            "timing": attn["timing"],
        },
        "step_roofline": {
            "bound": "hbm" if step_bytes / (hbm * 1e9) >= step_flops / (tc_burst * 1e12) else "tensor",
            "algorithmic_bytes": step_bytes, "algorithmic_flops": step_flops,
            "roofline_us": round(step_roof_us, 3), "step_us": round(ms_step * 1e3, 3),
            "frac": round(step_roof_us / (ms_step * 1e3), 4),
        },
        "clocks": clk.summary(),
    }
    if seqpar is not None:
        seqpar["unsharded_attn_us"] = round(attn_us, 3)
        out["seqpar"] = seqpar
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, args.seed, budget_s=args.cpu_seconds)
    return out


# ---------------------------------------------------------------- prefill
def prefill_draws(cfg, seed, b):
    """Seeded prompt inputs of sequence b: c_KV [S, d_c], k_R [S, d_r] (pre-rotation),
    q_nope [S, H, d_k], q_R [S, H, d_r], bf16 bit patterns."""
    S, H = cfg["S"], cfg["H"]
    c, k = W.latent_rows(cfg, seed, b, S)
    q_nope = W.normal(seed, "prefill_q_nope", (S, H, cfg["d_k"]), index=(b,))
    q_r = W.normal(seed, "prefill_q_r", (S, H, cfg["d_r"]), index=(b,))
    return tuple(W.bf16_bits(x) for x in (c, k, q_nope, q_r))


def prefill_flops(cfg):
    """Causal (query, row) pairs x heads x (2 R + 2 d_c)."""
    S, R = cfg["S"], cfg["d_c"] + cfg["d_r"]
    pairs = cfg["B"] * S * (S + 1) // 2
    return pairs * cfg["H"] * (2 * R + 2 * cfg["d_c"]), pairs


def prefill_explicit_flops(cfg):
    """K / V rebuild (2 B S H (d_k + d_v) d_c) plus causal (query, row) pairs x heads x
    (2 (d_k + d_r) + 2 d_v)."""
    B, S, H, d_c, d_r, d_k, d_v = (cfg[k] for k in ("B", "S", "H", "d_c", "d_r", "d_k", "d_v"))
    pairs = B * S * (S + 1) // 2
    return 2 * B * S * H * (d_k + d_v) * d_c + pairs * H * (2 * (d_k + d_r) + 2 * d_v), pairs


class PrefillWorkload:
    """One prompt step over static buffers: append the B x S prompt rows (RoPE at
    0..S-1), absorb every query at its own position, causal prefill attention,
    W_UV.  With explicit=True the step is append + prefill without absorption (K and
    V rebuilt per head, standard causal attention).  Inputs are far larger than L2."""

    def __init__(self, name, seed, device, explicit=False):
        import torch
        import head_latent_attention_29_b300 as mla
        self.mla, self.torch = mla, torch
        cfg = dict(W.WORKLOADS[name])
        self.cfg = cfg
        B, S, H, d_c, d_r, d_k, d_v = (cfg[k] for k in ("B", "S", "H", "d_c", "d_r", "d_k", "d_v"))
        self.B, self.S, self.H = B, S, H
        bf = torch.bfloat16
        self.base, self.scale = cfg["rope_base"], cfg["scale"]
        pin = lambda shape: torch.empty(shape, dtype=bf).pin_memory()
        self.host = {"c_kv": pin((B, S, d_c)), "k_r": pin((B, S, d_r)), "q_nope": pin((B, S, H, d_k)),
                     "q_rope": pin((B, S, H, d_r))}
        for b in range(B):
            for key, x in zip(("c_kv", "k_r", "q_nope", "q_rope"), prefill_draws(cfg, seed, b)):
                self.host[key][b].copy_(torch.from_numpy(x.view(np.int16)).view(bf))
        self.dev = {k: v.to(device) for k, v in self.host.items()}
        w_uk, w_uv = W.up_weights(cfg, seed)
        up = lambda x: torch.from_numpy(np.ascontiguousarray(W.bf16_bits(x)).view(np.int16)).view(bf).to(device)
        self.w_uk, self.w_uv = up(w_uk), up(w_uv)
        self.cache = mla.LatentCache(B, S, d_c, d_r, dtype=bf, device=device)
        self.seq_idx = torch.arange(B, dtype=torch.int32, device=device).repeat_interleave(S)
        self.pos = torch.arange(S, dtype=torch.int32, device=device).repeat(B)
        self.q_start = torch.zeros(B, dtype=torch.int32, device=device)
        if not explicit:  # the explicit form needs neither the absorbed query nor o_lat
            self.q_cat = torch.empty((B, S, H, d_c + d_r), dtype=bf, device=device)
            self.o_lat = torch.empty((B, S, H, d_c), dtype=bf, device=device)
        self.lse = torch.empty((B, S, H), dtype=torch.float32, device=device)
        self.o = torch.empty((B, S, H, d_v), dtype=bf, device=device)
        self.o_host = torch.empty((B, S, H, d_v), dtype=bf).pin_memory()
        self.explicit = explicit
        if explicit:
            self.ws = mla.prefill_explicit_workspace(B, 0, S, H, device)
            self.kernels_per_step = 3  # append, K / V rebuild GEMM, attention
        else:
            self.ws = mla.prefill_workspace(B, S, H, d_c, bf, device)
            self.kernels_per_step = 5  # append, absorb GEMM, split attention, combine, out-up GEMM

    def attn(self):
        if self.explicit:
            d = self.dev
            self.mla.prefill_explicit(d["q_nope"], d["q_rope"], self.cache, self.w_uk, self.w_uv, 0, self.scale,
                                      True, self.base, self.ws, self.o, self.lse)
            return
        self.mla.prefill_attn(self.q_cat, self.cache, self.q_start, self.scale, True, self.ws, self.o_lat, self.lse)

    def step(self, copy_in=False, copy_out=False):
        d, mla, BS = self.dev, self.mla, self.B * self.S
        if copy_in:
            for k, v in self.host.items():
                d[k].copy_(v, non_blocking=True)
        mla.cache_append(self.cache, d["c_kv"].view(BS, -1), d["k_r"].view(BS, -1), self.seq_idx, self.pos,
                         self.base)
        if self.explicit:
            self.attn()
            if copy_out:
                self.o_host.copy_(self.o, non_blocking=True)
            return
        mla.absorb_q(d["q_nope"].view(BS, self.H, -1), d["q_rope"].view(BS, self.H, -1), self.pos, self.w_uk,
                     self.base, out=self.q_cat.view(BS, self.H, -1))
        self.attn()
        mla.out_up(self.o_lat.view(BS, self.H, -1), self.w_uv, out=self.o.view(BS, self.H, -1))
        if copy_out:
            self.o_host.copy_(self.o, non_blocking=True)


def run_b300_prefill(args, rank, world, device):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(device)
    explicit = getattr(args, "explicit", False)
    wl = PrefillWorkload(args.workload, args.seed + rank, device, explicit)
    cfg = wl.cfg
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize(device)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            wl.step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, device)
    ms_step = ms_total / args.steps
    tokens = wl.B * wl.S * world
    value = job_throughput(wl.B * wl.S, world, ms_step * 1e-3)

    # the attention kernel alone (split + combine), on its stream
    n_rep = max(3, min(args.steps, 20))
    wl.attn()
    torch.cuda.synchronize(device)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_rep):
        wl.attn()
    a1.record(stream)
    torch.cuda.synchronize(device)
    attn_us = a0.elapsed_time(a1) * 1e3 / n_rep

    # end to end: prompt inputs in from pinned memory, o back to pinned memory
    n_e2e = max(3, min(args.steps, 10))
    wl.step(True, True)
    torch.cuda.synchronize(device)
    barrier()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        wl.step(True, True)
        stream.synchronize()
    barrier()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device)
    h2d = sum(v.numel() * v.element_size() for v in wl.host.values())
    d2h = wl.o_host.numel() * wl.o_host.element_size()

    hbm, tc_burst, tc_sust, peak_kind = _peaks()
    flops, pairs = prefill_explicit_flops(cfg) if explicit else prefill_flops(cfg)
    R = cfg["d_c"] + cfg["d_r"]
    if explicit:  # queries and rows in, rebuilt K / V out and back in, o out
        kv = cfg["B"] * cfg["S"] * cfg["H"] * (cfg["d_k"] + cfg["d_v"]) * 2
        bytes_alg = (cfg["B"] * cfg["S"] * (cfg["H"] * (cfg["d_k"] + cfg["d_r"]) + R) * 2 + 2 * kv
                     + cfg["B"] * cfg["S"] * cfg["H"] * cfg["d_v"] * 2)
    else:
        bytes_alg = cfg["B"] * cfg["S"] * cfg["H"] * (R + cfg["d_c"]) * 2 + cfg["B"] * cfg["S"] * R * 2
    tflops = flops / (attn_us * 1e-6) / 1e12
    t_tc = flops / (tc_burst * 1e12)
    t_mem = bytes_alg / (hbm * 1e9)
    return {
        "metric": f"MLA causal prefill prompt tokens/s at H={cfg['H']},d_c={cfg['d_c']},B={cfg['B']},S={cfg['S']} bf16; "
                  "% of roofline",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) latents/keys/queries, N(0,1/512) up-projections)",
        "config": {"workload": args.workload, "B": cfg["B"], "S": cfg["S"], "H": cfg["H"], "d_c": cfg["d_c"],
                   "d_r": cfg["d_r"], "causal": True, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (queries, rebuilt K / V or q_cat / o_lat: GBs per step)",
                   "step": ("append(B*S rows)+prefill_explicit(K/V rebuild + causal attention)" if explicit else
                            "append(B*S rows)+absorb_q(B*S queries)+prefill_attn(split+combine)+out_up")},
        "gpu_launches": wl.kernels_per_step * args.steps,
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "roofline": {
            "bound": "tensor",
            "kernel": ("prefill_explicit (K/V rebuild GEMM + causal attention)" if explicit else
                       "prefill_attn (split tensor-core kernel + combine)"),
            "achieved": round(tflops, 1), "peak": tc_burst, "unit": "TFLOP/s", "frac": round(tflops / tc_burst, 4),
            "traffic": None, "peak_source": f"{peak_kind} bf16_tflops (burst)",
            "frac_sustained": round(tflops / tc_sust, 4) if tc_sust else None,
            "attn_us": round(attn_us, 1), "algorithmic_flops": flops, "causal_pairs": pairs,
            "roofline_us": round(max(t_tc, t_mem) * 1e6, 1), "frac_of_roofline": round(max(t_tc, t_mem) * 1e6 / attn_us, 4),
        },
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- cache rows from hidden states
def kvdown_rows_slots(cfg):
    """(sequence, position) of every token a kv_down step writes: the new token at
    position N - 1 of each decode sequence, or a whole prompt per sequence."""
    if "prompt" in cfg:
        B, P = cfg["B"], cfg["prompt"]
        return np.repeat(np.arange(B, dtype=np.int32), P), np.tile(np.arange(P, dtype=np.int32), B), B, P
    B, N, T = cfg["B"], cfg["N"], cfg["T"]
    return np.arange(T, dtype=np.int32) % B, np.full(T, N - 1, dtype=np.int32), B, N


def kvdown_bytes_flops(cfg):
    """Algorithmic bytes (W once, h once, gamma, the rows written) and FLOPs of one step."""
    T, dm, R, d_c = cfg["T"], cfg["d_model"], cfg["d_c"] + cfg["d_r"], cfg["d_c"]
    return 2 * (dm * R + T * dm + d_c + T * R), 2 * T * dm * R


class KvDownWorkload:
    """kv_down_append over static buffers, captured in CUDA graphs.  Decode-sized
    steps rotate through enough weight copies that every step reads W from HBM."""

    def __init__(self, name, seed, device):
        import torch
        import head_latent_attention_29_b300 as mla
        self.mla, self.torch = mla, torch
        cfg = dict(W.WORKLOADS[name])
        self.cfg = cfg
        bf = torch.bfloat16
        T, dm, d_c, d_r = cfg["T"], cfg["d_model"], cfg["d_c"], cfg["d_r"]
        self.T = T
        h, w_dkv, w_kr, gamma = W.kv_down_inputs(cfg, seed)
        up = lambda x: torch.from_numpy(np.ascontiguousarray(W.bf16_bits(x)).view(np.int16)).view(bf)
        self.h_host = up(h).pin_memory()
        self.h = self.h_host.to(device)
        w = up(np.concatenate([w_dkv, w_kr], axis=1)).to(device)
        w_bytes = w.numel() * 2
        self.rotate = max(1, math.ceil(160e6 / w_bytes)) if T * dm * 2 < 126e6 else 1
        self.ws_list = [w] + [w.clone() for _ in range(self.rotate - 1)]
        self.gamma = up(gamma).to(device)
        seq, pos, B, N = kvdown_rows_slots(cfg)
        self.seq, self.pos = torch.from_numpy(seq).to(device), torch.from_numpy(pos).to(device)
        # every device buffer a captured graph touches stays referenced from here: each
        # capture empties the allocator's cache, so a buffer freed earlier would leave a
        # graph with a released address
        self.seq_l, self.pos_l = self.seq.long(), self.pos.long()
        self.cache = mla.LatentCache(B, N, d_c, d_r, dtype=bf, device=device)
        self.ws = mla.kv_down_workspace(T, dm, d_c, d_r, bf, device)
        self.eps, self.base = cfg["eps"], cfg["rope_base"]
        self.rows_host = torch.empty((T, d_c + d_r), dtype=bf).pin_memory()
        self.kernels_per_step = 2  # projection (tensor cores) + partial sums / norm / RoPE / store

        def call(w):
            mla.kv_down_append(self.cache, self.h, w, self.gamma, self.seq, self.pos, self.eps, self.base, self.ws)

        for w in self.ws_list:
            call(w)  # one eager run each: one-time host setup happens outside capture
        torch.cuda.synchronize(device)
        # one graph holds a step per weight copy, back to back as a model's layers
        # would issue them (programmatic launch between steps, no graph-launch gap
        # inside); a replay is `rotate` steps
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            for w in self.ws_list:
                call(w)
        self.e2e = []
        # end to end: h in from pinned memory, the written rows back to pinned memory;
        # decode-sized steps get four independent sets of buffers (h, cache, workspace,
        # rows), so that steps of different sets can be in flight at once
        self.rows_hosts = [self.rows_host]
        self.e2e_sets = []  # (h, cache, workspace, rows) of each set, kept alive with its graph
        n_sets = 4 if T <= 4096 else 1
        for j in range(n_sets):
            h_d = self.h if j == 0 else self.h.clone()
            cache = self.cache if j == 0 else mla.LatentCache(B, N, d_c, d_r, dtype=bf, device=device)
            ws = self.ws if j == 0 else mla.kv_down_workspace(T, dm, d_c, d_r, bf, device)
            rows_dev = torch.empty((T, d_c + d_r), dtype=bf, device=device)
            if j > 0:
                self.rows_hosts.append(torch.empty((T, d_c + d_r), dtype=bf).pin_memory())
            w = self.ws_list[j % len(self.ws_list)]
            self.e2e_sets.append((h_d, cache, ws, rows_dev))
            mla.kv_down_append(cache, h_d, w, self.gamma, self.seq, self.pos, self.eps, self.base, ws)
            torch.cuda.synchronize(device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                h_d.copy_(self.h_host, non_blocking=True)
                mla.kv_down_append(cache, h_d, w, self.gamma, self.seq, self.pos, self.eps, self.base, ws)
                rows_dev.copy_(cache.data[self.seq_l, self.pos_l, : d_c + d_r])
                self.rows_hosts[j].copy_(rows_dev, non_blocking=True)
            self.e2e.append(g)

    def replay(self):
        """`rotate` steps, each on its own weight copy."""
        self.graph.replay()


def run_b300_kvdown(args, rank, world, device):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(device)
    wl = KvDownWorkload(args.workload, args.seed + rank, device)
    cfg = wl.cfg
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            dist.barrier()

    for i in range(max(1, math.ceil(args.warmup / wl.rotate))):
        wl.replay()
    torch.cuda.synchronize(device)
    steps = args.steps if wl.T <= 4096 else max(3, min(args.steps, 200))
    replays = max(1, math.ceil(steps / wl.rotate))
    steps = replays * wl.rotate
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(replays):
            wl.replay()
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
    ms_step = max_over_ranks(e0.elapsed_time(e1), world, device) / steps
    value = job_throughput(wl.T, world, ms_step * 1e-3)

    n_e2e = 2000 if wl.T <= 4096 else 5
    for g in wl.e2e:
        g.replay()
    torch.cuda.synchronize(device)
    # one step at a time: the host waits for each step's rows before the next step
    barrier()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        wl.e2e[0].replay()
        stream.synchronize()
    barrier()
    e2e_serial_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device)
    # one step per buffer set in flight, each set on its own stream (independent
    # batches of new tokens), the host waiting for each step's rows len(sets) behind
    e2e_s, in_flight = e2e_serial_s, 1
    k = len(wl.e2e)
    if k > 1:
        streams = [torch.cuda.Stream(device) for _ in range(k)]

        def pipelined(n):
            pending = []
            for i in range(n):
                s = streams[i % k]
                with torch.cuda.stream(s):
                    wl.e2e[i % k].replay()
                ev = torch.cuda.Event()
                ev.record(s)
                pending.append(ev)
                if len(pending) == k:
                    pending.pop(0).synchronize()
            for ev in pending:
                ev.synchronize()

        pipelined(4 * k)  # warm-up
        torch.cuda.synchronize(device)
        barrier()
        t0 = time.perf_counter()
        pipelined(n_e2e)
        barrier()
        e2e_s, in_flight = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device), k
        torch.cuda.synchronize(device)

    hbm, tc_burst, tc_sust, peak_kind = _peaks()
    bytes_alg, flops = kvdown_bytes_flops(cfg)
    t_mem, t_tc = bytes_alg / (hbm * 1e9), flops / (tc_burst * 1e12)
    us = ms_step * 1e3
    tensor = t_tc > t_mem
    achieved = flops / (us * 1e-6) / 1e12 if tensor else bytes_alg / (us * 1e-6) / 1e9
    peak = tc_burst if tensor else hbm
    R = cfg["d_c"] + cfg["d_r"]
    return {
        "metric": f"MLA cache rows from hidden states tokens/s (RMSNorm(h W_DKV) || RoPE(h W_KR), append) at "
                  f"T={wl.T},d_model={cfg['d_model']},d_c={cfg['d_c']},d_r={cfg['d_r']} bf16; % of roofline",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) hidden states, N(0,1/d_model) projections, gain 1+N(0,0.01))",
        "config": {"workload": args.workload, "T": wl.T, "d_model": cfg["d_model"], "d_c": cfg["d_c"],
                   "d_r": cfg["d_r"], "parallelism": f"replicas x{world}",
                   "l2": (f"{wl.rotate} rotating weight copies ({wl.rotate * cfg['d_model'] * R * 2 / 1e6:.0f} MB "
                          "vs 126 MB L2)" if wl.rotate > 1 else "inputs larger than L2"),
                   "step": "kv_down_append (projection on the tensor cores + norm/RoPE/store)"},
        "gpu_launches": wl.kernels_per_step * steps,
        "e2e": {"value": round(wl.T * world / e2e_s, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.h_host.numel() * 2, "d2h_bytes_per_step": wl.rows_host.numel() * 2,
                "steps_in_flight": in_flight, "value_one_step_at_a_time": round(wl.T * world / e2e_serial_s, 1)},
        "roofline": {
            "bound": "tensor" if tensor else "hbm", "kernel": "kv_down_append (projection + finish)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s" if tensor else "GB/s",
            "frac": round(achieved / peak, 4), "traffic": None,
            "peak_source": f"{peak_kind} " + ("bf16_tflops (burst)" if tensor else "hbm_gbs"),
            "step_us": round(us, 3), "algorithmic_bytes": bytes_alg, "algorithmic_flops": flops,
            "roofline_us": round(max(t_mem, t_tc) * 1e6, 3),
        },
        "clocks": clk.summary(),
    }


def _ncu_traffic(workload):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary, if any."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        v = d.get(workload)
        if v and v.get("kernel_hash") == _kernel_hash():
            return v.get("dram_bytes_per_launch")
    return None


def _kernel_hash():
    """sha256[:16] of the attention kernels' source with comments and blank space
    removed, so that the stored DRAM counters follow code changes, not comment edits."""
    import hashlib
    import re
    p = os.path.join(ROOT, "head_latent_attention_29_b300", "csrc", "k_decode_tc.cu")
    with open(p) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    code = "\n".join(line.strip() for line in src.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


# ---------------------------------------------------------------- CPU oracle baseline
def _cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo), for the baseline's record."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


# The oracle's step runs on every host core this process may use: one spawned
# worker process per core (spawn, not fork: the parent holds a CUDA context), BLAS
# held to one thread in each, the sample's inputs built once inside the workers as
# resident state.  All workers start together and run for the same wall-clock
# window; the rate is the tokens of all of them over that window.
ORACLE_ROW_CAP = 1 << 20  # cached rows a decode sample may hold in all (float64 rows: ~4.8 GB)


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _oracle_sample(kind: str, workload: str, seed: int):
    """(units of work, description) of the bounded sample the oracle is timed on."""
    cfg = dict(W.WORKLOADS[workload])
    if kind == "decode":
        lens = W.seq_lens(cfg, seed)
        k, rows = 0, 0
        while k < cfg["B"] and (k == 0 or rows + int(lens[k]) <= ORACLE_ROW_CAP):
            rows += int(lens[k])
            k += 1
        return list(range(k)), (f"decode steps of sequences 0..{k - 1} of {cfg['B']} "
                                f"({rows} cached rows, N={int(lens[:k].min())}..{int(lens[:k].max())})")
    if kind == "prefill":
        S = cfg["S"]
        order = [int(i) for i in np.random.default_rng(seed).permutation(S)]
        return order, (f"prompt query rows of sequence 0 at random positions of 0..{S - 1} "
                       "(absorb at the row's position, causal prefix, W_UV)")
    n = min(cfg["T"], 32)
    return [n], f"batches of {n} tokens (projection, RMSNorm, RoPE)"


def _oracle_units(kind: str, workload: str, seed: int, mine):
    """Closures, one per unit of this worker's share; each runs the oracle's step on
    its unit and returns the tokens it produced."""
    from oracle import mla_oracle as O
    cfg = dict(W.WORKLOADS[workload])
    if kind == "decode":
        lens = W.seq_lens(cfg, seed)
        q_nope, q_r = W.query(cfg, seed)
        w_uk, w_uv = W.up_weights(cfg, seed)
        wd = lambda x: W.widen(W.as_dtype(x, cfg["dtype"]), cfg["dtype"])
        w_uk, w_uv = wd(w_uk), wd(w_uv)
        q_nope, q_r = wd(q_nope[:, 0]), wd(q_r[:, 0])
        base = cfg.get("rope_base", 1e4)
        units = []
        for b in mine:
            n = int(lens[b])
            c, k = W.latent_rows(cfg, seed, b, n)
            rows = O.cache_rows(wd(c), wd(k), np.arange(n), base)

            def step(b=b, n=n, rows=rows):
                q_cat = O.absorb_q(q_nope[b], q_r[b], n - 1, w_uk, base)
                o_lat, _ = O.decode_absorbed(q_cat, rows, cfg["d_c"], cfg["scale"])
                O.out_up(o_lat, w_uv)
                return 1
            units.append(step)
        return units
    if kind == "prefill":
        S, base = cfg["S"], cfg["rope_base"]
        c, k, q_nope, q_r = prefill_draws(cfg, seed, 0)
        rows = O.cache_rows(W.widen(c, "bf16"), W.widen(k, "bf16"), np.arange(S), base)
        sel = np.asarray(mine, dtype=np.int64)
        qn, qr = W.widen(q_nope[sel], "bf16"), W.widen(q_r[sel], "bf16")
        del q_nope, q_r
        w_uk, w_uv = (W.widen(W.as_dtype(w, "bf16"), "bf16") for w in W.up_weights(cfg, seed))
        units = []
        for j, i in enumerate(mine):
            def step(j=j, i=i):
                q_cat = O.absorb_q(qn[j], qr[j], i, w_uk, base)
                o_lat, _ = O.decode_absorbed(q_cat, rows[: i + 1], cfg["d_c"], cfg["scale"])
                O.out_up(o_lat, w_uv)
                return 1
            units.append(step)
        return units
    n = mine[0]
    d_c = cfg["d_c"]
    h, w_dkv, w_kr, gamma = W.kv_down_inputs(dict(cfg, T=n), seed)
    wd = lambda x: W.widen(W.as_dtype(x, "bf16"), "bf16")
    h, w, g = wd(h), wd(np.concatenate([w_dkv, w_kr], axis=1)), wd(gamma)
    pos = kvdown_rows_slots(cfg)[1][:n]

    def step():
        O.kv_down_rows(h, w[:, :d_c], w[:, d_c:], g, cfg["eps"], pos, cfg["rope_base"])
        return n
    return [step]


def _oracle_worker(kind, workload, seed, share, n_workers, cmd, res):
    """One host core of the oracle timing: build this share's units, report ready,
    then on each ("run", start, seconds) run units round-robin from the common wall
    clock start until the window has passed."""
    try:
        from threadpoolctl import threadpool_info, threadpool_limits
        threadpool_limits(1)
        blas = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
    except Exception:  # pragma: no cover
        blas = [int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0)]
    units_all, _ = _oracle_sample(kind, workload, seed)
    mine = units_all if kind == "kvdown" else units_all[share::n_workers]
    units = _oracle_units(kind, workload, seed, mine)
    res.put(("ready", share, max(blas) if blas else 1))
    while True:
        m = cmd.get()
        if m[0] != "run":
            return
        _, t_start, seconds = m
        while time.time() < t_start:
            time.sleep(0.0005)
        tokens, i = 0, 0
        while True:
            tokens += units[i % len(units)]()
            i += 1
            now = time.time()
            if now >= t_start + seconds:
                break
        res.put(("done", share, tokens, now))


class OracleHost:
    """The float64 oracle timed on the host cores (test infrastructure: only the CPU
    baseline and the reference arm use it)."""

    def __init__(self, kind: str, workload: str, seed: int):
        import multiprocessing as mp
        units, self.sample = _oracle_sample(kind, workload, seed)
        cores = _host_cores()
        self.n = cores if kind != "decode" else max(1, min(cores, len(units)))
        self.cores_available = cores
        ctx = mp.get_context("spawn")
        self.res = ctx.Queue()
        self.cmd = [ctx.Queue() for _ in range(self.n)]
        # BLAS in the workers held to one thread from their first import on
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        try:
            for k in saved:
                os.environ[k] = "1"
            self.procs = [ctx.Process(target=_oracle_worker, args=(kind, workload, seed, i, self.n, self.cmd[i],
                                                                    self.res), daemon=True)
                          for i in range(self.n)]
            for p in self.procs:
                p.start()
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        ready = [self.res.get(timeout=900) for _ in range(self.n)]
        self.blas_threads = max(r[2] for r in ready)

    def measure(self, seconds: float) -> float:
        t_start = time.time() + 0.05
        for q in self.cmd:
            q.put(("run", t_start, float(seconds)))
        done = [self.res.get(timeout=seconds + 900) for _ in range(self.n)]
        self.tokens = sum(d[2] for d in done)
        self.wall = max(d[3] for d in done) - t_start
        return self.tokens / self.wall

    def record(self, value: float) -> dict:
        return {"value": round(value, 3), "unit": "tokens/s", "cores": self.n * self.blas_threads,
                "kind": "oracle", "workers": self.n, "blas_threads_per_worker": self.blas_threads,
                "host_cpus": os.cpu_count(), "cpus_usable": self.cores_available, "cpu_model": _cpu_model(),
                "sample": f"{self.sample}, float64 numpy; {self.tokens} tokens in {self.wall:.1f} s of wall time "
                          f"on {self.n} worker processes"}

    def close(self):
        for q in self.cmd:
            q.put(("stop",))
        for p in self.procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()


def _oracle_kind(workload: str) -> str:
    cfg = W.WORKLOADS[workload]
    return "kvdown" if "T" in cfg else ("prefill" if "S" in cfg else "decode")


def cpu_baseline(workload: str, seed: int, budget_s: float = 12.0):
    """The float64 oracle's step (decode: absorb_q, attention over the prebuilt cache
    rows, out_up; prefill: the same per prompt row; rows from hidden states: the
    projection, norm and rotation) on the host cores for a bounded sample."""
    host = OracleHost(_oracle_kind(workload), workload, seed)
    try:
        host.measure(min(1.0, budget_s))  # warm-up
        return host.record(host.measure(budget_s))
    finally:
        host.close()


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cfg = W.WORKLOADS[args.workload]
    prefill = "S" in cfg
    kvdown = "T" in cfg
    host = OracleHost(_oracle_kind(args.workload), args.workload, args.seed)
    try:
        for _ in range(max(1, args.warmup)):
            host.measure(0.5)
        per = max(1.0, min(10.0, 60.0 / max(args.steps, 1)))
        vals = [host.measure(per) for _ in range(args.steps)]
        v = statistics.median(vals)
        cb = host.record(v)
    finally:
        host.close()
    if kvdown:
        metric = (f"MLA cache rows from hidden states tokens/s (RMSNorm(h W_DKV) || RoPE(h W_KR), append) at "
                  f"T={cfg['T']},d_model={cfg['d_model']},d_c={cfg['d_c']},d_r={cfg['d_r']} bf16; % of roofline")
    elif prefill:
        metric = (f"MLA causal prefill prompt tokens/s at H={cfg['H']},d_c={cfg['d_c']},B={cfg['B']},S={cfg['S']} bf16; "
                  "% of roofline")
    else:
        metric = decode_metric(args.workload, cfg)
    tokens_per_step = cfg["T"] if kvdown else cfg["B"] * cfg.get("S", 1)
    return {
        "impl": "reference",
        "metric": metric,
        "value": round(v, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tokens_per_step / v, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": cfg["B"], "H": cfg.get("H"), "d_c": cfg["d_c"], "d_r": cfg["d_r"],
                   "parallelism": "host cores (oracle)"},
        "cpu_baseline": cb,
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--workload", default="decode_h128_b32_n4096", choices=sorted(W.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rotate", type=int, default=ROTATE, help="cache copies rotated between steps (>= 1)")
    ap.add_argument("--explicit", action="store_true",
                    help="prefill workloads: the non-absorbed form (K and V rebuilt per head)")
    ap.add_argument("--paged", action="store_true",
                    help="decode workloads: 64-row pages of one pool in shuffled order behind a block table")
    ap.add_argument("--seq-shards", type=int, default=0,
                    help="decode workloads: also time one shard's partial and the merge of this many "
                         "sequence-position shards (one GPU; the collective between them is not timed)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.explicit and "S" not in W.WORKLOADS[args.workload]:
        ap.error("--explicit applies to prefill workloads")
    if args.paged and ("S" in W.WORKLOADS[args.workload] or "T" in W.WORKLOADS[args.workload]):
        ap.error("--paged applies to decode workloads")
    if args.seq_shards and (args.paged or "S" in W.WORKLOADS[args.workload] or "T" in W.WORKLOADS[args.workload]):
        ap.error("--seq-shards applies to decode workloads on a contiguous cache")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    import torch
    import torch.distributed as dist
    device = torch.device("cuda", local)
    if world > 1:
        torch.cuda.set_device(device)
        dist.init_process_group("nccl", device_id=device)
    try:
        if "T" in W.WORKLOADS[args.workload]:
            out = run_b300_kvdown(args, rank, world, device)
            if rank == 0 and not args.no_cpu_baseline:
                out["cpu_baseline"] = cpu_baseline(args.workload, args.seed, budget_s=args.cpu_seconds)
        elif "S" in W.WORKLOADS[args.workload]:
            out = run_b300_prefill(args, rank, world, device)
            if rank == 0 and not args.no_cpu_baseline:
                out["cpu_baseline"] = cpu_baseline(args.workload, args.seed, budget_s=args.cpu_seconds)
        else:
            out = run_b300(args, rank, world, device)
        if rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
