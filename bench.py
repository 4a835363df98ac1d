"""Benchmark of one paged decode step on GB300.

A step is the whole decode hot path for one batch: each sequence's newest
token is stored in its slot and paged GQA decode attention attends every
cached token.  With one new token per sequence at its last position (the
default workload) both happen in one call, pa_decode_ex with new_k / new_v:
the stream-K decode kernel stores each token just before it fetches the
block holding it, and its merge kernel follows; otherwise the slot writer
(pa_reshape_and_cache) runs first and pa_decode after it.  The default
workload is the Llama-3.1-70B-shaped single layer: 64 sequences of 600-850
tokens, 64 query / 8 KV heads, head_dim 128, bf16, 16-token blocks placed at
random in a 16,384-block pool.

Prints one JSON line.  ``value`` is tokens/s (decoded tokens, i.e. sequences
per step, over device time with inputs resident in HBM).  A model runs one
such step per layer, each on its own slice of the KV cache, so the timed
loop runs K steps back to back over 8 layers' pools (and q), layer i % 8 at
step i: a layer's K/V are touched again only after the other seven layers'
(over 1.3 GB for the default workload, far beyond the 129 MB L2) have passed
through, so every step reads its K/V from HBM; no flush kernel sits between
steps.  The K steps are captured as CUDA graphs of 256 steps and replayed
(the launches keep their programmatic overlap inside a graph), bracketed by
one pair of CUDA events, so they run at device speed whatever the rate at
which Python issues calls; the default K keeps the timed region near three
seconds, long enough for the clock sampler.  ``per_step_flushed`` is one
step between CUDA events after an L2 flush by a 256 MiB read; it adds a
fixed few microseconds of event and launch latency to every step.  ``e2e``
is the same metric through the C ABI from pinned host buffers (per-step
inputs copied in and the output copied back inside the timed region; the KV
pool is device-resident state).  ``roofline`` reports the attention call
alone (pa_decode, no stores) against the measured HBM copy bandwidth.
``configs`` reports the other decode workloads the same way (the long-context
batch in its 512-token-partition launch, beside the automatic plan; the
shared-prompt and beam batches plain and as a cascade; the beams'
copy-on-write copies).  ``prefill`` times chunked prefill (16 sequences x
4,096 cached + 512 new tokens) against the measured bf16 tensor peak.
``cpu_baseline`` times the CPU oracle on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch one process per GPU with torch.distributed.run; every rank
decodes its own batch (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import pa_workloads as wl  # noqa: E402

METRIC = "paged decode attention tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20   # twice the 129 MB L2


def log(msg: str) -> None:
    print(msg, file=sys.stderr, flush=True)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


FALLBACK_BF16_TFLOPS = 1900.0


def measured_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, 'measured' | 'fallback')."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def prefill_flops(w: wl.Workload) -> int:
    """Algorithmic FLOPs of chunked causal prefill: for every (sequence, query,
    head) 2*d multiply-adds per visible key in Q.K and again in P.V."""
    visible = w.ctx_lens.astype(np.int64)[:, None] + np.arange(w.chunk, dtype=np.int64)[None, :] + 1
    return 4 * w.head_dim * int(visible.sum()) * w.num_q_heads


def unique_decode_bytes(w: wl.Workload) -> int:
    """decode_bytes with every physical block's K/V counted once however many
    tables share it (the slots read of a shared block: the most any of its
    sequences reads)."""
    b = w.block_size
    fill = {}
    for s, L in enumerate(w.seq_lens.astype(np.int64)):
        for i in range(int(-(-L // b))):
            blk = int(w.tables[s, i])
            fill[blk] = max(fill.get(blk, 0), int(min(b, L - i * b)))
    kv = sum(fill.values()) * w.num_kv_heads * w.head_dim * 2 * 2
    return decode_bytes(w) - int(w.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 4 + kv


def cascade_group_size(w: wl.Workload):
    """Sequences per group that share a prefix, for the workloads built that
    way (one prompt shared by the whole batch; the beams of a prompt)."""
    if w.name == "shared_prefix":
        return w.batch
    if w.name == "beam_fork":
        return int(w.notes["beams"])
    return None


def decode_bytes(w: wl.Workload) -> int:
    """Algorithmic bytes of one decode call: every attended K and V row once,
    q and out once, the table entries used and the lengths."""
    L = w.seq_lens.astype(np.int64)
    kv = int(L.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    qo = 2 * w.batch * w.num_q_heads * w.head_dim * 2
    tables = 4 * int((-(-L // w.block_size)).sum())
    return kv + qo + tables + 4 * w.batch


def traffic_record(workload: str):
    """DRAM bytes per decode launch for a workload from the committed ncu
    summary, if it was taken on the current decode kernel source; else None.
    Keys are workload names, with '@auto' for a batch on the automatic plan
    that is specified with partitions."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256") != kernel_source_sha():
        return None
    r = rec.get("records", {}).get(workload)
    return r["dram_bytes_per_launch"] if r else None


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for name in ("pa_decode_kernel.cuh", "pa_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_167_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class GraphLoop:
    """fn(i) for i = 0 .. K-1, back to back on the device: captured as CUDA
    graphs of up to `chunk` calls (programmatic launches keep their
    overlap inside a graph) and replayed, so the steps run at device speed
    whatever the rate at which Python issues calls.  fn must have run
    eagerly before (the library does its one-time set-up outside capture)."""

    def __init__(self, fn, K: int, chunk: int = 256):
        self.K = K
        self.n = max(1, min(K, chunk))
        self.full, self.rem = divmod(K, self.n)
        self.g_full = self._capture(fn, 0, self.n) if self.full else None
        self.g_rem = self._capture(fn, self.full * self.n, self.rem) if self.rem else None

    @staticmethod
    def _capture(fn, start: int, count: int):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(start, start + count):
                    fn(i)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def run(self):
        for _ in range(self.full):
            self.g_full.replay()
        if self.g_rem is not None:
            self.g_rem.replay()


def timed_graph(fn, K: int, warmup: int, barrier=lambda: None) -> float:
    """Milliseconds of K calls fn(0 .. K-1) replayed from CUDA graphs,
    bracketed by one pair of CUDA events on the launching stream after
    `warmup` eager calls and one untimed replay."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    loop = GraphLoop(fn, K)
    loop.run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    loop.run()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    del loop
    return e0.elapsed_time(e1)


def measure_prefill(pa, dev, flush_fn, K: int = 20, warmup: int = 3, iters: int = 5):
    """Device time of pa_prefill_chunk on the 16 x (4096 + 512) chunk: K
    launches replayed from a CUDA graph between one pair of CUDA events (each
    launch reads 302 MB of K/V, more than L2 holds), and beside it the median
    of single launches between events after an L2 flush, which includes the
    host's launch work (argument checks, tensor-map encoding)."""
    w = wl.prefill_chunk()
    t = wl.make_tensors(w, dev)
    tables = torch.as_tensor(w.tables, device=dev)
    ctx = torch.as_tensor(w.ctx_lens, device=dev)
    out = torch.empty_like(t["q"])
    run = lambda: pa.prefill_chunk(out, t["q"], t["pool"], tables, ctx, int(w.ctx_lens.max()), w.scale)
    ms = timed_graph(lambda i: run(), K, warmup) / K
    ts = []
    stream = torch.cuda.current_stream()
    for _ in range(iters):
        flush_fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    assert pa.get_device_error() == 0, "device error during prefill"
    return w, ms, prefill_flops(w), float(np.median(ts)), K


def measure_swap(pa, step, iters: int = 5):
    """Median device time of pa_swap_blocks moving 1,024 blocks of the decode
    pool (64 MiB) to pinned host memory and back."""
    n = min(1024, step.w.num_blocks)
    w = step.w
    host = torch.empty((n, 2, w.num_kv_heads, w.block_size, w.head_dim), dtype=torch.bfloat16, pin_memory=True)
    pairs = torch.stack([torch.arange(n, dtype=torch.int32), torch.arange(n, dtype=torch.int32)], 1).to(step.dev)
    stream = torch.cuda.current_stream()
    res = {}
    for name, direction in (("out", pa.PA_SWAP_OUT), ("in", pa.PA_SWAP_IN)):
        pa.swap_blocks(step.pool, host, pairs, direction)
        ts = []
        for _ in range(iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            pa.swap_blocks(step.pool, host, pairs, direction)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = float(np.median(ts))
        res[name] = {"ms": round(ms, 4), "gbs": round(host.numel() * 2 / (ms / 1e3) / 1e9, 1)}
    assert pa.get_device_error() == 0, "device error during swap"
    return {"blocks": n, "bytes": host.numel() * 2, **res}


def measure_paging_overhead(pa, step, K: int, warmup: int):
    """The attention call (as the roofline times it) on copies of the layers'
    pools whose blocks are placed sequence after sequence in table order;
    None when blocks are shared or the plan is split-context."""
    w, dev = step.w, step.dev
    nb = (-(-w.seq_lens.astype(np.int64) // w.block_size)).astype(np.int64)
    ids = np.full_like(w.tables, -1)
    base = 0
    for s in range(w.batch):
        ids[s, :nb[s]] = np.arange(base, base + nb[s])
        base += int(nb[s])
    old = w.tables[ids >= 0]
    if step.part != 0 or base > w.num_blocks or len(np.unique(old)) != len(old):
        return None
    src = torch.as_tensor(old.astype(np.int64), device=dev)
    dst = torch.as_tensor(ids[ids >= 0].astype(np.int64), device=dev)
    pools = torch.zeros_like(step.pools)
    for layer in range(step.layers):
        pools[layer][dst] = step.pools[layer][src]
    tables = torch.as_tensor(ids.astype(np.int32), device=dev)

    def call(i):
        pa.decode(step.out, step.qs[i % step.layers], pools[i % step.layers], tables, step.seq_lens, w.max_seq_len,
                  w.scale, 0, step.ws, flags=pa.PA_DECODE_EARLY_METADATA)

    ms = timed_graph(call, K, warmup) / K
    assert pa.get_device_error() == 0, "device error during the identity-placement calls"
    del pools
    return {"identity_ms": round(ms, 5)}


def measure_cascade(pa, step, K: int, warmup: int):
    """The same decode step as a cascade: pa_prefix_attention over each
    group's shared prefix (read once for the group), then pa_decode_cascade
    over the private suffixes with the new tokens stored by the call.  Replayed
    over the layers, as the step is timed.  None for workloads without shared
    prefixes or off the balanced schedule."""
    w, dev = step.w, step.dev
    gsz = cascade_group_size(w)
    if gsz is None or not step.fused:
        return None
    plan = pa.cascade_plan(w.tables, w.seq_lens, gsz, w.block_size)
    pt = torch.as_tensor(plan["prefix_tables"], device=dev)
    pl = torch.as_tensor(plan["prefix_lens"], device=dev)
    order = torch.as_tensor(plan["group_order"], device=dev)   # longest prefix first
    st = torch.as_tensor(plan["suffix_tables"], device=dev)
    sl = torch.as_tensor(plan["suffix_lens"], device=dev)
    max_p, max_s = int(plan["prefix_lens"].max()), max(1, int(plan["suffix_lens"].max()))
    o_part = torch.empty(step.q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device=dev)
    nbytes = pa.decode_workspace_size(step.pool, w.batch, w.num_q_heads, max_s, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None

    def prefix(i):
        pa.prefix_attention(o_part, lse, step.qs[i % step.layers], step.pools[i % step.layers], pt, pl, gsz, max_p,
                            w.scale, group_order=order)

    def suffix(i):
        pa.decode_cascade(step.out, step.qs[i % step.layers], step.pools[i % step.layers], st, sl, max_s, w.scale,
                          o_part, lse, 0, ws, flags=pa.PA_DECODE_EARLY_METADATA, new_k=step.new_k, new_v=step.new_v)

    def both(i):
        prefix(i)
        suffix(i)

    def grouped(i):
        pa.decode_grouped(step.out, step.qs[i % step.layers], step.pools[i % step.layers], pt, pl, st, sl, gsz, max_p,
                          max_s, w.scale, group_order=order, new_k=step.new_k, new_v=step.new_v,
                          flags=pa.PA_DECODE_EARLY_METADATA)

    step_ms = timed_graph(both, K, warmup) / K
    prefix_ms = timed_graph(prefix, K, warmup) / K
    suffix_ms = timed_graph(suffix, K, warmup) / K
    try:   # the one-call form, where every member's suffix fits the suffix tile
        grouped(0)
        grouped_ms = timed_graph(grouped, K, warmup) / K
    except pa.PagedAttentionError as e:
        if e.status != 2:
            raise
        grouped_ms = None
    assert pa.get_device_error() == 0, "device error during the cascade calls"
    return {"group_size": gsz, "groups": int(len(plan["prefix_lens"])),
            "prefix_tokens_mean": float(plan["prefix_lens"].mean()),
            "step_ms": step_ms, "prefix_ms": prefix_ms, "suffix_ms": suffix_ms, "grouped_ms": grouped_ms}


def measure_copy_blocks(pa, step, K: int, warmup: int):
    """pa_copy_blocks on the workload's copy-on-write pairs (each copies a
    whole block, K and V of every kv-head), alternating between two layers'
    pools; None without pairs."""
    w = step.w
    if w.copy_pairs is None or not len(w.copy_pairs):
        return None
    pairs = torch.as_tensor(w.copy_pairs, device=step.dev)
    ms = timed_graph(lambda i: pa.copy_blocks(step.pools[i % step.layers], pairs), K, warmup) / K
    assert pa.get_device_error() == 0, "device error during copy_blocks"
    nbytes = 2 * len(w.copy_pairs) * 2 * w.num_kv_heads * w.block_size * w.head_dim * 2   # read + write
    return {"pairs": int(len(w.copy_pairs)), "ms": ms, "bytes": nbytes}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class DecodeStep:
    """Device-resident inputs of one decode step per layer and the calls that
    run it.  Every layer has its own pool and q (copies of the workload's);
    tables, lengths and slots are shared, as in a model."""

    LAYERS = 8

    def __init__(self, pa, w: wl.Workload, dev: torch.device, tensors, layers: int = LAYERS):
        self.pa, self.w, self.dev, self.layers = pa, w, dev, layers
        pool0 = tensors["pool"].to(dev)
        self.pools = torch.empty((layers,) + tuple(pool0.shape), dtype=pool0.dtype, device=dev)
        for layer in range(layers):
            self.pools[layer].copy_(pool0)
        del pool0
        q0 = tensors["q"].to(dev)
        self.qs = torch.empty((layers,) + tuple(q0.shape), dtype=q0.dtype, device=dev)
        for layer in range(layers):
            self.qs[layer].copy_(q0)
        self.pool, self.q = self.pools[0], self.qs[0]
        self.new_k = tensors["new_k"].to(dev)
        self.new_v = tensors["new_v"].to(dev)
        self.tables = torch.as_tensor(w.tables, device=dev)
        self.seq_lens = torch.as_tensor(w.seq_lens, device=dev)
        self.slots_host = pa.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size, w.num_blocks)
        self.slots = torch.as_tensor(self.slots_host, device=dev)
        self.out = torch.empty_like(self.q)
        self.part = pa.decode_partition_tokens(self.pool, w.batch, w.num_q_heads, w.max_seq_len, w.partition_tokens)
        nbytes = pa.decode_workspace_size(self.pool, w.batch, w.num_q_heads, w.max_seq_len, w.partition_tokens)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
        # part == 0: the balanced (stream-K) schedule, a persistent kernel plus its merge kernel
        self.num_parts = -(-w.max_seq_len // self.part) if self.part > 0 else 1
        decode_launches = 2 if self.part == 0 or self.num_parts > 1 else 1
        # one new token per sequence, at its last position: the decode call
        # stores it itself (pa_decode_ex with new_k / new_v)
        self.fused = (self.part == 0 and len(w.new_seq_idx) == w.batch
                      and np.array_equal(w.new_seq_idx, np.arange(w.batch))
                      and np.array_equal(w.new_positions, w.seq_lens.astype(np.int64) - 1))
        self.decode_launches = decode_launches
        self.launches_per_step = decode_launches + (0 if self.fused else 1)

    def write(self, layer: int = 0):
        self.pa.reshape_and_cache(self.pools[layer], self.new_k, self.new_v, self.slots)

    def step(self, layer: int = 0):
        """One decode step: store the new tokens' K/V, attend."""
        if not self.fused:
            self.write(layer)
            self.decode(layer)
            return
        w = self.w
        self.pa.decode(self.out, self.qs[layer], self.pools[layer], self.tables, self.seq_lens, w.max_seq_len,
                       w.scale, w.partition_tokens, self.ws, flags=self.pa.PA_DECODE_EARLY_METADATA,
                       new_k=self.new_k, new_v=self.new_v)

    def decode(self, layer: int = 0, partition_tokens=None, ws=None):
        w = self.w
        part = w.partition_tokens if partition_tokens is None else partition_tokens
        # lengths and tables are host copies, never written by the slot writer
        # that each decode call follows: the early-metadata launch applies
        self.pa.decode(self.out, self.qs[layer], self.pools[layer], self.tables, self.seq_lens, w.max_seq_len,
                       w.scale, part, self.ws if ws is None else ws, flags=self.pa.PA_DECODE_EARLY_METADATA)


def rank_workload(name: str, rank: int) -> wl.Workload:
    """The batch one rank decodes: every rank its own Llama-shaped batch (same
    shapes, its own lengths, placement and values: weak scaling); the other
    workloads are the same on every rank."""
    if name == "llama70b_decode":
        return wl.CONFIGS[name](seed=wl.SEED_BASE + 1 + 1000 * rank)
    return wl.CONFIGS[name]()


def reduce_max(values, world: int, device) -> list:
    """Element-wise maximum of each rank's timings over all ranks (the job's
    time is its slowest rank's); a plain list on one rank."""
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def roofline_hbm(alg: int, ms: float, peak: float, peak_kind: str, kernel: str, traffic=None, unique=None) -> dict:
    achieved = alg / (ms / 1e3) / 1e9
    r = {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic, "algorithmic_bytes": alg,
         "decode_ms": round(ms, 5)}
    if unique is not None:
        r["unique_bytes"] = unique
        r["unique_frac"] = round(unique / (ms / 1e3) / 1e9 / peak, 4)
    return r


# Decode workloads reported besides the headline one, in the launch
# configuration each is specified with (the long-context batch with its
# 512-token partitions and the reduce kernel).
CONFIG_NAMES = ("tiny", "long_context", "shared_prefix", "beam_fork")
CONFIG_STEPS = 2048


def measure_config(pa, name: str, dev, K: int, warmup: int):
    """Timings of one decode workload: the step (new tokens stored, then
    attention), the attention call alone, and for the long-context batch the
    automatic plan beside its partitions; the cascade and the copy-on-write
    copies where the workload has them.  Raw milliseconds (reduced over ranks
    by the caller)."""
    w = wl.CONFIGS[name]()
    tensors = wl.make_tensors(w, dev)
    step = DecodeStep(pa, w, dev, tensors)
    del tensors
    res = {}
    copies = measure_copy_blocks(pa, step, K, warmup)
    if copies is not None:   # the forks' copies first, as the workload's recipe
        pairs = torch.as_tensor(w.copy_pairs, device=dev)
        for layer in range(step.layers):
            pa.copy_blocks(step.pools[layer], pairs)
        res["copy_ms"] = copies["ms"]
    res["step_ms"] = timed_graph(lambda i: step.step(i % step.layers), K, warmup) / K
    res["decode_ms"] = timed_graph(lambda i: step.decode(i % step.layers), K, warmup) / K
    if step.part != 0:   # the same batch on the automatic plan
        nb = pa.decode_workspace_size(step.pool, w.batch, w.num_q_heads, w.max_seq_len, 0)
        ws0 = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        res["auto_decode_ms"] = timed_graph(lambda i: step.decode(i % step.layers, 0, ws0), K, warmup) / K
    casc = measure_cascade(pa, step, K, warmup)
    if casc is not None:
        for k in ("step_ms", "prefix_ms", "suffix_ms", "grouped_ms"):
            if casc[k] is not None:
                res["cascade_" + k] = casc[k]
    assert pa.get_device_error() == 0, f"device error during {name}"
    meta = {"w": w, "part": step.part, "num_parts": step.num_parts, "fused": step.fused,
            "launches": step.launches_per_step, "cascade": casc, "copies": copies}
    del step
    torch.cuda.empty_cache()
    return res, meta


def config_line(name, res, meta, peak, peak_kind, world):
    """The JSON object of one decode workload."""
    w = meta["w"]
    alg, uniq = decode_bytes(w), unique_decode_bytes(w)
    part = meta["part"]
    kernel = ("paged_decode_kernel + paged_decode_reduce_kernel" if part and meta["num_parts"] > 1
              else "paged_decode_kernel" if part else "paged_decode_sk_kernel + paged_decode_sk_merge_kernel")
    out = {"workload": w.name, "global_batch": world * w.batch, "num_q_heads": w.num_q_heads,
           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
           "seq_len_min": int(w.seq_lens.min()), "seq_len_max": int(w.seq_lens.max()),
           "seq_len_mean": round(float(w.seq_lens.mean()), 1), "pool_blocks": w.num_blocks,
           "schedule": f"split-context, {part}-token partitions x {meta['num_parts']}" + (" + reduce" if meta["num_parts"] > 1 else "")
           if part else "balanced stream-K (persistent, 2 CTAs/SM), early-metadata launch",
           "step": "new tokens stored by the decode call, then attention" if meta["fused"]
           else "slot writer (pa_reshape_and_cache), then pa_decode",
           "steps_timed": CONFIG_STEPS,
           "step_ms": round(res["step_ms"], 5),
           "tokens_per_s": round(world * w.batch / (res["step_ms"] / 1e3), 1),
           "roofline": roofline_hbm(alg, res["decode_ms"], peak, peak_kind, kernel, traffic_record(w.name),
                                    uniq if uniq != alg else None)}
    if "auto_decode_ms" in res:
        out["auto_plan"] = {"schedule": "balanced stream-K (the automatic plan) on the same batch",
                            "roofline": roofline_hbm(alg, res["auto_decode_ms"], peak, peak_kind,
                                                     "paged_decode_sk_kernel + paged_decode_sk_merge_kernel",
                                                     traffic_record(w.name + "@auto"))}
    casc = meta["cascade"]
    if casc is not None:
        ms = res["cascade_step_ms"]
        out["cascade"] = {"group_size": casc["group_size"], "groups": casc["groups"],
                          "prefix_tokens_mean": round(casc["prefix_tokens_mean"], 1),
                          "step_ms": round(ms, 5), "prefix_ms": round(res["cascade_prefix_ms"], 5),
                          "suffix_ms": round(res["cascade_suffix_ms"], 5),
                          "tokens_per_s": round(world * w.batch / (ms / 1e3), 1),
                          "speedup_vs_step": round(res["step_ms"] / ms, 3),
                          "roofline": {"bound": "hbm", "achieved": round(uniq / (ms / 1e3) / 1e9, 1), "peak": peak,
                                       "peak_kind": peak_kind, "unit": "GB/s",
                                       "frac": round(uniq / (ms / 1e3) / 1e9 / peak, 4), "traffic": None,
                                       "algorithmic_bytes": uniq,
                                       "note": "unique bytes (each shared block once) over the whole cascade step"},
                          "note": "pa_prefix_attention over each group's shared prefix (tensor cores, read once per "
                                  "group), then pa_decode_cascade over the private suffixes with the new tokens "
                                  "stored by the call"}
        if "cascade_grouped_ms" in res:
            gms = res["cascade_grouped_ms"]
            out["cascade"]["grouped"] = {
                "step_ms": round(gms, 5), "tokens_per_s": round(world * w.batch / (gms / 1e3), 1),
                "speedup_vs_step": round(res["step_ms"] / gms, 3),
                "roofline": {"bound": "hbm", "kernel": "prefill_kernel, grouped (prefix tiles + one suffix tile), persistent",
                             "achieved": round(uniq / (gms / 1e3) / 1e9, 1), "peak": peak, "peak_kind": peak_kind,
                             "unit": "GB/s", "frac": round(uniq / (gms / 1e3) / 1e9 / peak, 4), "traffic": None,
                             "algorithmic_bytes": uniq, "note": "unique bytes over the one-call step"},
                "note": "pa_decode_grouped: each group's queries over its shared prefix and then one tile of every "
                        "member's suffix blocks, the new tokens stored by the call; one launch"}
    if meta["copies"] is not None:
        cp = meta["copies"]
        out["copy_blocks"] = {"pairs": cp["pairs"], "ms": round(res["copy_ms"], 5),
                              "roofline": {"bound": "hbm", "achieved": round(cp["bytes"] / (res["copy_ms"] / 1e3) / 1e9, 1),
                                           "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                                           "frac": round(cp["bytes"] / (res["copy_ms"] / 1e3) / 1e9 / peak, 4),
                                           "algorithmic_bytes": cp["bytes"]}}
    return out


def run_ours(args, world, rank, local):
    import paged_kv_cache_167_gb300 as pa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = rank_workload(args.config, rank)
    tensors = wl.make_tensors(w, "cpu")
    step = DecodeStep(pa, w, dev, tensors, layers=args.layers)
    stream = torch.cuda.current_stream()
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = lambda: flush.view(torch.int32).sum()     # evicts L2, leaves no dirty lines
    flush_write = lambda: flush.fill_(1)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for i in range(args.warmup):
        step.step(i % step.layers)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0, "device error during warm-up"

    K = args.steps
    # ---- the headline: K steps back to back over the layers, replayed from CUDA graphs
    loop = GraphLoop(lambda i: step.step(i % step.layers), K)
    loop.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        e0.record(stream)
        loop.run()
        e1.record(stream)
        torch.cuda.synchronize()
    total_ms = e0.elapsed_time(e1)
    barrier()
    del loop
    K_dec = min(K, 8192)   # the attention call alone, for the roofline
    decode_total_ms = timed_graph(lambda i: step.decode(i % step.layers), K_dec, args.warmup, barrier)

    K_flush = min(K, 50)

    def timed_flushed(flush_fn, write=True):
        # one step between events after an L2 flush; no event between the two
        # calls: it would serialise the decode kernel's programmatic launch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K_flush)]
        barrier()
        torch.cuda.synchronize()
        for i in range(K_flush):
            flush_fn()
            ev[i][0].record(stream)
            if write:
                step.step()
            else:
                step.decode()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        return [ev[i][0].elapsed_time(ev[i][1]) for i in range(K_flush)]

    flushed_ms = timed_flushed(flush_read)
    flushed_decode_ms = timed_flushed(flush_read, write=False)
    wstep_ms = timed_flushed(flush_write)
    assert pa.get_device_error() == 0, "device error during the timed steps"

    # ---- end to end through the C ABI from pinned host buffers
    host_q = tensors["q"].pin_memory()
    host_k = tensors["new_k"].pin_memory()
    host_v = tensors["new_v"].pin_memory()
    host_tables = torch.as_tensor(w.tables).pin_memory()
    host_lens = torch.as_tensor(w.seq_lens).pin_memory()
    host_slots = torch.empty(len(step.slots_host), dtype=torch.int64).pin_memory()
    host_out = torch.empty_like(tensors["q"]).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (host_q, host_k, host_v, host_tables, host_lens) +
              (() if step.fused else (host_slots,)))
    d2h = host_out.numel() * host_out.element_size()

    staging = None
    if step.fused:   # one call: inputs from host buffers, the step, the output back (pa_decode_host)
        nb = pa.decode_host_staging_size(step.pool, w.batch, w.num_q_heads, w.tables.shape[1])
        staging = torch.empty(nb, dtype=torch.uint8, device=dev)

    def e2e_step():
        if staging is not None:
            pa.decode_host(host_out, host_q, step.pool, host_tables, host_lens, w.max_seq_len, w.scale, staging,
                           w.partition_tokens, step.ws, new_k_host=host_k, new_v_host=host_v)
            torch.cuda.current_stream().synchronize()
            return
        step.q.copy_(host_q, non_blocking=True)
        step.new_k.copy_(host_k, non_blocking=True)
        step.new_v.copy_(host_v, non_blocking=True)
        step.tables.copy_(host_tables, non_blocking=True)
        step.seq_lens.copy_(host_lens, non_blocking=True)
        if not step.fused:   # the slot writer needs the slots
            host_slots.numpy()[:] = pa.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size,
                                                    w.num_blocks)
            step.slots.copy_(host_slots, non_blocking=True)
        step.step()
        host_out.copy_(step.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    K_e2e = min(K, 400)
    for _ in range(args.warmup):
        e2e_step()
    barrier()
    e2e_s = 0.0
    for _ in range(K_e2e):
        flush_read()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_s += time.perf_counter() - t0
    barrier()

    K_side = min(K, CONFIG_STEPS)
    paging = measure_paging_overhead(pa, step, K_side, args.warmup)
    casc = measure_cascade(pa, step, K_side, args.warmup)
    prefill = None if args.no_prefill else measure_prefill(pa, dev, flush_read)
    swap = measure_swap(pa, step)
    head_launches = step.launches_per_step
    head_fused, head_part, head_parts = step.fused, step.part, step.num_parts
    del step
    torch.cuda.empty_cache()

    configs = []
    if not args.no_configs:
        for name in CONFIG_NAMES:
            if name != args.config:
                configs.append((name,) + measure_config(pa, name, dev, min(K, CONFIG_STEPS), args.warmup))

    flat = [total_ms, e2e_s * 1e3, decode_total_ms / K_dec, sum(wstep_ms), sum(flushed_ms),
            float(np.mean(flushed_decode_ms))]
    keys = []
    for name, res, _ in configs:
        for k in sorted(res):
            keys.append((name, k))
            flat.append(res[k])
    if casc is not None:
        for k in ("step_ms", "prefix_ms", "suffix_ms"):
            flat.append(casc[k])
        casc.pop("grouped_ms", None)
    red = reduce_max(flat, world, dev)
    total_ms, e2e_ms, decode_avg_ms, wtotal_ms, ftotal_ms, fdecode_ms = red[:6]
    off = 6
    for (name, k) in keys:
        for cname, res, _ in configs:
            if cname == name:
                res[k] = red[off]
        off += 1
    if casc is not None:
        for k in ("step_ms", "prefix_ms", "suffix_ms"):
            casc[k] = red[off]
            off += 1

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    tokens = world * w.batch * K
    value = tokens / (total_ms / 1e3)
    alg = decode_bytes(w)
    peak, bf16_peak, peak_kind = measured_peaks()
    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded bf16 N(0,1) K/V/q, random physical block placement",
        "config": {"workload": w.name, "global_batch": world * w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                   "seq_len_min": int(w.seq_lens.min()), "seq_len_max": int(w.seq_lens.max()),
                   "seq_len_mean": float(w.seq_lens.mean()), "pool_blocks": w.num_blocks,
                   "schedule": "balanced stream-K (persistent, 2 CTAs/SM), early-metadata launch" if head_part == 0
                   else f"split-context, {head_part}-token partitions x {head_parts}",
                   "step": "new tokens stored by the decode call (pa_decode_ex new_k/new_v), then attention"
                   if head_fused else "slot writer (pa_reshape_and_cache), then pa_decode",
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "layers": args.layers,
                   "timing": "K steps replayed from CUDA graphs of 256 steps, one CUDA event pair around all K",
                   "l2": f"inputs larger than L2: steps rotate over {args.layers} layers' pools and q, "
                         f"{(args.layers - 1) * alg / 1e9:.2f} GB of other layers' K/V between reuses of a layer; no flush"},
        "per_step_flushed": {"steps": K_flush, "ms_per_step": round(ftotal_ms / K_flush, 5),
                             "tokens_per_s": round(world * w.batch * K_flush / (ftotal_ms / 1e3), 1),
                             "decode_ms": round(fdecode_ms, 5),
                             "decode_frac": round(alg / (fdecode_ms / 1e3) / 1e9 / peak, 4),
                             "tokens_per_s_after_write_flush": round(world * w.batch * K_flush / (wtotal_ms / 1e3), 1),
                             "l2": "flushed before each step by reading a 256 MiB buffer; one event pair per step"},
        "roofline": roofline_hbm(alg, decode_avg_ms, peak, peak_kind, "pa_decode (decode kernel + merge kernel)",
                                 traffic_record(w.name), unique_decode_bytes(w)),
        "kv_read_gbs": round(alg / (decode_avg_ms / 1e3) / 1e9, 1),
        "derived": {"full_model_80_layers_tokens_per_s": round(value / 80, 1),
                    "note": "value / 80: one such step per layer of an 80-layer model, attention only"},
        "e2e": {"value": round(world * w.batch * K_e2e / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K_e2e,
                "call": "pa_decode_host (pinned host q, new K/V, tables, lengths in; output back; one call)"
                if staging is not None else "host-to-device copies, pa_reshape_and_cache, pa_decode, copy back"},
        "gpu_launches": head_launches * K,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples_under_load": clk["samples"], "window_s": round(total_ms / 1e3, 3)},
    }
    if prefill is not None:
        pw, pms, pflop, psingle, pK = prefill
        line["prefill"] = {"workload": f"{pw.batch} seqs x ({int(pw.ctx_lens[0])} cached + {pw.chunk} chunk) tokens, "
                                       f"{pw.num_q_heads}/{pw.num_kv_heads} heads, d={pw.head_dim}",
                           "ms": round(pms, 4), "tflops": round(pflop / (pms / 1e3) / 1e12, 1),
                           "timing": f"{pK} launches replayed from a CUDA graph, one CUDA event pair around them; "
                                     "each reads 302 MB of K/V (more than L2)",
                           "single_flushed_ms": round(psingle, 4),
                           "roofline": {"bound": "tensor", "kernel": "prefill_kernel (tcgen05)",
                                        "achieved": round(pflop / (pms / 1e3) / 1e12, 1),
                                        "peak": bf16_peak, "peak_kind": peak_kind, "unit": "TFLOP/s",
                                        "frac": round(pflop / (pms / 1e3) / 1e12 / bf16_peak, 4),
                                        "flops": pflop}}
    if paging is not None:
        line["paging_overhead"] = dict(paging, random_ms=round(decode_avg_ms, 5),
                                       ratio=round(decode_avg_ms / paging["identity_ms"], 4),
                                       note="the attention call on the same K/V with every sequence's blocks "
                                            "consecutive in the pool (identity placement) against random placement")
    if casc is not None:
        ub = unique_decode_bytes(w)
        line["cascade"] = dict(casc, tokens_per_s=round(world * w.batch / (casc["step_ms"] / 1e3), 1),
                               speedup_vs_step=round((total_ms / K) / casc["step_ms"], 3),
                               unique_gbs=round(ub / (casc["step_ms"] / 1e3) / 1e9, 1),
                               unique_frac=round(ub / (casc["step_ms"] / 1e3) / 1e9 / peak, 4))
    line["swap"] = dict(swap, note="pa_swap_blocks between the decode pool and pinned host memory, one kernel "
                                   "over the CPU-GPU link")
    if configs:
        line["configs"] = {name: config_line(name, res, meta, peak, peak_kind, world) for name, res, meta in configs}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, tensors, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_pass(orc, w, tensors_bits, seqs):
    """The oracle's decode step for sequences `seqs`: write their new tokens,
    then attend every query head."""
    rows = np.stack(np.meshgrid(seqs, np.arange(w.num_q_heads), indexing="ij"), axis=-1).reshape(-1, 2)
    oracle_rows(orc, w, tensors_bits, rows)


def oracle_rows(orc, w, tensors_bits, rows):
    """The oracle's decode step for query rows (sequence, head): write those
    sequences' new tokens, then attend the rows."""
    import oracle
    pool, q, k, v = tensors_bits
    geom = oracle.dense_geom(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    sel = np.isin(w.new_seq_idx, rows[:, 0])
    slots = orc.slot_mapping(w.tables, w.new_seq_idx[sel], w.new_positions[sel], w.block_size)
    orc.reshape_and_cache(pool, geom, k[sel], v[sel], slots)
    orc.paged_decode(q, pool, geom, w.tables, w.seq_lens, w.num_q_heads, w.scale, rows=rows)


def cpu_baseline(w, tensors, budget_s: float = 10.0):
    import oracle
    orc = oracle.load()
    tb = (wl.bf16_bits(tensors["pool"]).copy(), wl.bf16_bits(tensors["q"]), wl.bf16_bits(tensors["new_k"]),
          wl.bf16_bits(tensors["new_v"]))
    t0 = time.perf_counter()
    oracle_pass(orc, w, tb, np.arange(w.batch))
    first = time.perf_counter() - t0
    passes, elapsed = 1, first
    while elapsed < budget_s and passes < 1000:
        t0 = time.perf_counter()
        oracle_pass(orc, w, tb, np.arange(w.batch))
        elapsed += time.perf_counter() - t0
        passes += 1
    cores = orc.num_threads()
    # the same oracle on one thread, over whole passes for about half the budget
    orc.set_num_threads(1)
    try:
        p1, e1 = 0, 0.0
        while p1 == 0 or (e1 < budget_s / 2 and p1 < 1000):
            t0 = time.perf_counter()
            oracle_pass(orc, w, tb, np.arange(w.batch))
            e1 += time.perf_counter() - t0
            p1 += 1
    finally:
        orc.set_num_threads(cores)
    return {"value": round(w.batch * passes / elapsed, 2), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{passes} full passes over the {w.batch}-sequence batch ({w.batch * w.num_q_heads} "
                      f"query rows each), fp64, {elapsed:.1f} s",
            "single_thread": {"value": round(w.batch * p1 / e1, 2), "unit": "tokens/s", "cores": 1,
                              "sample": f"{p1} full passes, {e1:.1f} s"}}


def run_reference(args, world, rank, local):
    """The oracle as it stands on the host cores, on this arm's workload: each
    step a random sample of the batch's query rows (a decoded token is one
    sequence's num_q_heads rows), sized so the run takes about a minute."""
    if rank != 0:
        return
    import oracle
    orc = oracle.load()
    w = wl.CONFIGS[args.config]()
    tensors = wl.make_tensors(w, "cpu")
    tb = (wl.bf16_bits(tensors["pool"]).copy(), wl.bf16_bits(tensors["q"]), wl.bf16_bits(tensors["new_k"]),
          wl.bf16_bits(tensors["new_v"]))
    all_rows = np.stack(np.meshgrid(np.arange(w.batch), np.arange(w.num_q_heads), indexing="ij"),
                        axis=-1).reshape(-1, 2).astype(np.int32)
    rng = np.random.default_rng(0)
    probe = all_rows[rng.choice(len(all_rows), min(len(all_rows), 64), replace=False)]
    t0 = time.perf_counter()
    oracle_rows(orc, w, tb, probe)
    per_row = max((time.perf_counter() - t0) / len(probe), 1e-6)
    per_step = int(max(1, min(len(all_rows), 60.0 / (args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        oracle_rows(orc, w, tb, all_rows[rng.choice(len(all_rows), per_step, replace=False)])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rows(orc, w, tb, all_rows[rng.choice(len(all_rows), per_step, replace=False)])
    elapsed = time.perf_counter() - t0
    value = per_step * args.steps / w.num_q_heads / elapsed
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded bf16 N(0,1) K/V/q, random physical block placement",
        "config": {"workload": w.name, "global_batch": w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                   "query_rows_per_step": per_step},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": orc.num_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step} random query rows (sequence, head) of the batch per step; "
                                   f"a token is {w.num_q_heads} rows"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=81920)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama70b_decode",
                    choices=["tiny", "llama70b_decode", "long_context", "shared_prefix", "beam_fork"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other decode workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=DecodeStep.LAYERS,
                    help="layers' pools the timed steps rotate over (1 keeps one pool, e.g. for profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if world != args.gpus and rank == 0:
        log(f"note: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE")
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
