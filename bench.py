#!/usr/bin/env python3
"""Benchmark of one paged decode step on GB300.

A step is one pass of the hot path over one batch: the new token of every
sequence is written into its slot, then decode attention runs over the whole
paged context.  By default both happen in one call, pa_decode_append (the
write folded into the decode kernel; plus the split-KV merge kernel when
contexts are split); ``--step write+decode`` times pa_write_kv followed by
pa_decode instead.  Block tables and slots come from the host block pool
(pa_pool), built before the timed region; the pool's slots are checked to be
the slots of positions L - 1 that pa_decode_append derives.

Prints one JSON line (rank 0).  ``value`` is KV GB/s over the algorithmic
bytes (K+V of the valid tokens + q + out + block-table entries + lengths, plus
the write's bytes), device-timed with CUDA events with inputs resident in HBM;
``e2e`` is the same metric through the Python API with the step's inputs
copied from pinned host memory and the output copied back inside the timed
region.  ``--impl reference`` times the fp64 CPU oracle instead.

Under torchrun each rank runs its own batch of the same shape (weak scaling,
no collective on the data path); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged-decode KV GB/s and % of GB300 HBM peak; decode queries/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES_DEFAULT = 129 * 1024 * 1024

# pa_decode_plan.schedule values
SCHEDULE_NAMES = {0: "partitioned grid", 1: "lean persistent wave + merge",
                  2: "persistent row-split wave + merge"}

# Timed beside the headline in the default run, one side record each.
SIDE_WORKLOADS = ("qwen_gqa_fp8", "qwen_gqa_verify4", "mha_short_bs16", "long_context_fp8")

WORKLOAD_DESCRIPTIONS = {
    "qwen_gqa": "Qwen-style GQA layer: batch 64, 28 q / 4 kv heads, head_dim 128, bf16, block_size 16, "
                "context_lens uniform in [512,4096], pool 20000 blocks shuffled, q/K/V ~ N(0,1), "
                "one new token per sequence written via slot_mapping before the decode",
    "long_context": "long-context split-KV: batch 8, 32 q / 8 kv heads, head_dim 128, bf16, block_size 16, "
                    "context_lens uniform in [32768,131072], pool sized to fit (+1%), shuffled",
    "mha_short_bs16": "many short requests, MHA: batch 256, 32/32 heads, head_dim 128, fp16, block_size 16, "
                      "context_lens lognormal(median 256, sigma 1) clipped to [16,2048]",
    "mha_short_bs32": "many short requests, MHA: batch 256, 32/32 heads, head_dim 128, fp16, block_size 32, "
                      "context_lens lognormal(median 256, sigma 1) clipped to [16,2048]",
    "qwen_gqa_verify4": "speculative verify on the Qwen-style GQA layer: batch 64, 28 q / 4 kv heads, head_dim 128, "
                        "bf16, block_size 16, context_lens uniform in [512,4096] (including the 4 new tokens), pool "
                        "20000 blocks shuffled; 4 new tokens per sequence written via slot_mapping, then every one "
                        "attends its prefix causally (pa_decode_multi, q_len 4)",
    "prefix_cow": "prefix sharing: 64 sequences (one parent + 63 forks through the block pool) share a "
                  "2048-token prefix (full shared tail: no copy-on-write), private tails uniform in [1,256], "
                  "28 q / 4 kv heads, head_dim 128, bf16, block_size 16; value = effective GB/s (every "
                  "sequence's K/V counted), roofline over the unique pages",
    "prefix_cow_2056": "prefix sharing, copy-on-write variant: as prefix_cow with a 2056-token prefix, so the "
                       "first append of 63 sequences copies the shared partial block (pa_copy_blocks)",
    "qwen_gqa_fp8": "the Qwen-style GQA layer with an FP8 (E4M3) KV cache: batch 64, 28 q / 4 kv heads, head_dim 128, "
                    "bf16 queries, block_size 16, context_lens uniform in [512,4096], pool 20000 blocks shuffled; "
                    "q/K/V ~ N(0,1) in bf16, K/V quantised with one scale per (block, kv head) = block max / 448; "
                    "one new token per sequence quantised into the slot of position L - 1 inside the decode "
                    "(pa_decode_fp8_append)",
    "long_context_fp8": "long-context split-KV with an FP8 (E4M3) KV cache: batch 8, 32 q / 8 kv heads, head_dim 128, "
                        "bf16 queries, block_size 16, context_lens uniform in [32768,131072]; scales per (block, kv "
                        "head) = block max / 448",
    "mha_short_bs16_fp8": "many short requests, MHA, FP8 (E4M3) KV cache: batch 256, 32/32 heads, head_dim 128, "
                          "fp16 queries, block_size 16, context_lens lognormal(median 256, sigma 1) clipped to "
                          "[16,2048]; scales per (block, kv head) = block max / 448",
    "qwen_gqa_layers28": "a whole-model decode step over 28 Qwen-style GQA layers (each: batch 64, 28 q / 4 kv "
                         "heads, head_dim 128, bf16, block_size 16, context_lens uniform in [512,4096], pool 20000 "
                         "blocks): every layer's new token written in one pa_write_kv_layers launch, then one "
                         "pa_decode per layer",
    "swap_qwen": "preemption swap on the Qwen-style GQA layer's cache (4 kv heads, head_dim 128, bf16, "
                 "block_size 16, pool 20000 blocks, 64 sequences with context_lens uniform in [512,4096] "
                 "built through the block pool): each step swaps 16 sequences out to a page-locked host pool "
                 "while the 16 swapped out the step before come back in (pa_seq_swap + pa_swap_blocks, one "
                 "launch per direction, the two on separate streams)",
}
SWAP_GROUP = 16  # sequences preempted per swap step
DTYPE_NAMES = {"f32": "f32", "f16": "f16", "bf16": "bf16"}


# ---- host-side pieces (no GPU needed; covered by the gloo tests) ------------------------------
def rank_seed(base_seed: int, rank: int) -> int:
    """Every rank decodes its own batch of the same shape: the seed is offset by the rank."""
    return base_seed + 1000003 * rank


def decode_bytes(context_lens, num_heads: int, num_kv_heads: int, head_dim: int, elem_bytes: int,
                 block_size: int, q_len: int = 1) -> int:
    """Algorithmic bytes of one decode call: K+V of the valid tokens, q, out, table entries, lengths
    (q_len query tokens per sequence: the context is read once for all of them)."""
    lens = np.asarray(context_lens, dtype=np.int64)
    kv = 2 * int(lens.sum()) * num_kv_heads * head_dim * elem_bytes
    qo = 2 * len(lens) * q_len * num_heads * head_dim * elem_bytes
    tables = 4 * int(((lens + block_size - 1) // block_size).sum())
    return kv + qo + tables + 4 * len(lens)


def decode_bytes_fp8(context_lens, num_heads: int, num_kv_heads: int, head_dim: int, q_bytes: int,
                     block_size: int) -> int:
    """Algorithmic bytes of one FP8 decode call: K+V codes of the valid tokens (one byte each), the K and V
    scale of every (page, kv head), q, out, table entries, lengths."""
    lens = np.asarray(context_lens, dtype=np.int64)
    pages = int(((lens + block_size - 1) // block_size).sum())
    kv = 2 * int(lens.sum()) * num_kv_heads * head_dim
    scales = 8 * pages * num_kv_heads
    qo = 2 * len(lens) * num_heads * head_dim * q_bytes
    return kv + scales + qo + 4 * pages + 4 * len(lens)


def write_bytes_fp8(num_tokens: int, num_kv_heads: int, head_dim: int, src_bytes: int) -> int:
    """Read new K and V, write their codes, read the slots and the scales."""
    return (2 * src_bytes + 2) * num_tokens * num_kv_heads * head_dim + 8 * num_tokens + 8 * num_tokens * num_kv_heads


def pages_touched_bytes(context_lens, num_kv_heads: int, head_dim: int, elem_bytes: int, block_size: int) -> int:
    lens = np.asarray(context_lens, dtype=np.int64)
    pages = int(((lens + block_size - 1) // block_size).sum())
    return 2 * pages * block_size * num_kv_heads * head_dim * elem_bytes


def write_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Read new K and V, write them into the caches, read the slots."""
    return 4 * num_tokens * num_kv_heads * head_dim * elem_bytes + 8 * num_tokens


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def kernel_sources_digest() -> str:
    """sha256 over the decode kernel's sources: ties a stored ncu traffic figure to the code it measured."""
    h = hashlib.sha256()
    for name in ("decode_kernel.cuh", "pa_common.cuh", "decode_launch.h", "decode_bf16.cu", "decode_f16.cu",
                 "decode_f32.cu", "decode_fp8.cu"):
        with open(os.path.join(ROOT, "paged_kv_cache_129_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def stored_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it measured the current sources."""
    path = os.path.join(ROOT, "profiles", f"ncu_paged_decode_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_sources_sha256") != kernel_sources_digest():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def gpu_selector(device) -> str:
    """nvidia-smi -i argument for a torch device (its UUID; CUDA_VISIBLE_DEVICES may renumber)."""
    import torch

    try:
        uid = str(torch.cuda.get_device_properties(device).uuid)
        return uid if uid.startswith("GPU-") else "GPU-" + uid
    except (AttributeError, RuntimeError):
        return str(device.index or 0)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: str, period_s: float = 0.1):
        self.device_index = device_index
        self.period_s = period_s
        self.samples = []
        self._stop = threading.Event()
        self._thread = None
        self.window = None

    def _one(self):
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
        except (OSError, subprocess.SubprocessError):
            return None
        if r.returncode != 0 or not r.stdout.strip():
            return None
        return [x.strip() for x in r.stdout.strip().splitlines()[0].split(",")]

    def _loop(self):
        while not self._stop.is_set():
            t0 = time.monotonic()
            s = self._one()
            t1 = time.monotonic()
            if s:
                self.samples.append(((t0 + t1) / 2, s))
            self._stop.wait(max(0.0, self.period_s - (t1 - t0)))

    def start(self):
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=10)

    def summary(self, t_begin: float, t_end: float, windows=None) -> dict:
        """Clocks seen between t_begin and t_end (or inside any of ``windows``, a list of (begin, end))."""
        windows = windows or [(t_begin, t_end)]
        inside = [s for t, s in self.samples if any(a <= t <= b for a, b in windows)]
        used = inside if inside else [s for _, s in self.samples]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in used if num(s[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in used:
            for name, flag in zip(names, s[4:8]):
                if flag.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(used[0][1]),
                "reasons": sorted(reasons), "samples": len(used),
                "samples_inside_timed_region": len(inside),
                "power_w_max": max((num(s[2]) or 0.0) for s in used)}


# ---- the CPU oracle leg -------------------------------------------------------------------------
def cpu_model() -> str:
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        parts = [f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields]
        return " ".join(parts) or os.uname().machine
    except OSError:
        return os.uname().machine


def time_oracle_parallel(inp, budget_s: float, threads: int, fp8=None):
    """Time the fp64 oracle over whole sequences (all heads) on `threads` host threads.

    One sequence is timed alone first; then as many sequences as fit in about
    `budget_s` of wall time are decoded, one task per sequence (the C oracle
    releases the GIL).  Returns the seconds, the sequences and rows done, the
    algorithmic bytes, and the single-thread figure of the first sequence.
    """
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    eb = inp.elem_bytes

    q_len = inp.q.shape[1] if inp.q.ndim == 4 else 1

    def seq_bytes(b):
        if fp8 is not None:
            return decode_bytes_fp8([int(inp.context_lens[b])], inp.num_heads, inp.num_kv_heads, inp.head_dim, eb,
                                    inp.block_size)
        return decode_bytes([int(inp.context_lens[b])], inp.num_heads, inp.num_kv_heads, inp.head_dim, eb,
                            inp.block_size, q_len)

    def run(b):
        if fp8 is not None:  # (key codes, value codes, key scales, value scales)
            oracle.decode_fp8(inp.q, inp.dtype, fp8[0], fp8[1], fp8[2], fp8[3], inp.block_tables, inp.context_lens,
                              inp.scale, rows=[(b, h) for h in range(inp.num_heads)])
        elif q_len == 1:
            oracle.decode_inputs(inp, rows=[(b, h) for h in range(inp.num_heads)])
        else:
            oracle.decode_multi(inp.q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, inp.dtype,
                                inp.scale, rows=[(b, t, h) for t in range(q_len) for h in range(inp.num_heads)])

    t0 = time.perf_counter()
    run(0)
    t_one = max(time.perf_counter() - t0, 1e-6)
    single = seq_bytes(0) / t_one
    n = int(min(inp.num_seqs, max(threads, budget_s * threads / t_one)))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        list(ex.map(run, range(n)))
        dt = time.perf_counter() - t0
    return {"seconds": dt, "seqs": n, "rows": n * inp.num_heads, "bytes": sum(seq_bytes(b) for b in range(n)),
            "single_thread_gbs": single / 1e9, "single_thread_seconds": t_one}


def time_oracle(inp, budget_s: float, rows_cap: int = 0):
    """Time the fp64 oracle on the first sequences of the batch (all heads), about `budget_s` seconds."""
    import oracle

    per_seq = []
    rows_done = 0
    seqs = 0
    bytes_done = 0
    t_total = 0.0
    eb = inp.elem_bytes
    for b in range(inp.num_seqs):
        rows = [(b, h) for h in range(inp.num_heads)]
        if rows_cap:
            rows = rows[:rows_cap]
        t0 = time.perf_counter()
        oracle.decode_inputs(inp, rows=rows)
        dt = time.perf_counter() - t0
        t_total += dt
        per_seq.append(dt)
        rows_done += len(rows)
        seqs += 1
        L = int(inp.context_lens[b])
        frac = len(rows) / inp.num_heads
        bytes_done += frac * decode_bytes([L], inp.num_heads, inp.num_kv_heads, inp.head_dim, eb, inp.block_size)
        if t_total >= budget_s:
            break
    return {"seconds": t_total, "seqs": seqs, "rows": rows_done, "bytes": bytes_done}


# ---- GPU arm ---------------------------------------------------------------------------------------
def build_batch(workload: str, seed: int):
    from paged_kv_cache_129_gb300 import workloads as wl

    gen = {"qwen_gqa": lambda s: wl.qwen_gqa(s), "qwen_gqa_verify4": lambda s: wl.qwen_gqa_verify(s, q_len=4),
           "qwen_gqa_layers28": lambda s: wl.qwen_gqa(s),  # every layer has the Qwen layer's shape
           "qwen_gqa_fp8": lambda s: wl.qwen_gqa(s), "long_context_fp8": lambda s: wl.long_context(s),
           "mha_short_bs16_fp8": lambda s: wl.mha_short(16, s),
           "long_context": lambda s: wl.long_context(s),
           "mha_short_bs16": lambda s: wl.mha_short(16, s), "mha_short_bs32": lambda s: wl.mha_short(32, s)}[workload]
    return gen(seed)


def prefix_batch(workload: str, seed: int, model: bool = False):
    """The prefix-sharing workload built through the product block pool (``model``: the
    oracle's allocator model, for the reference arm; both give the same tables).

    A parent appends the shared prefix, 63 forks share it; every sequence then
    appends its tail but the last token (copy-on-write pairs are copied, tail
    tokens written, on the host copy of the caches), and the step's new token
    (each tail's last) is appended for all sequences at once.  Returns the
    decode inputs, tables, lengths, new-token slots, the number of copy-on-write
    copies, and the bytes of the distinct pages the decode reads.
    """
    from paged_kv_cache_129_gb300 import workloads as wl

    prefix = 2056 if workload == "prefix_cow_2056" else 2048
    w = wl.prefix_cow(seed, prefix_len=prefix)
    bs = w.block_size
    pool = make_pool(w.num_blocks, bs, np.random.default_rng(12345).permutation(w.num_blocks), model)
    parent = pool.create()
    for _ in range(prefix):
        pool.append(parent)
    seqs = [parent] + [pool.fork(parent) for _ in range(w.num_seqs - 1)]
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    cum = np.concatenate([[0], np.cumsum(w.tail_lens)]).astype(np.int64)
    n_cow = 0

    def cow(pair):
        kc[pair[1]] = kc[pair[0]]
        vc[pair[1]] = vc[pair[0]]

    for i, sid in enumerate(seqs):
        for t in range(int(w.tail_lens[i]) - 1):
            slot, pair = pool.append(sid)
            if pair:
                cow(pair)
                n_cow += 1
            kc[slot // bs, :, slot % bs, :] = w.tail_key[cum[i] + t]
            vc[slot // bs, :, slot % bs, :] = w.tail_value[cum[i] + t]
    slots, pairs = pool.append_batch(seqs)
    for pair in pairs:
        cow(pair)
    n_cow += len(pairs)
    last = cum[1:] - 1
    tables, lens = pool.block_tables(seqs, int((int(max(prefix + t for t in w.tail_lens)) + bs - 1) // bs))
    pool.check_invariants()
    inp = wl.DecodeInputs(name=workload, dtype="bf16", num_heads=w.num_heads, num_kv_heads=w.num_kv_heads,
                          head_dim=w.head_dim, block_size=bs, num_blocks=w.num_blocks, q=w.q, key_cache=kc,
                          value_cache=vc, block_tables=tables, context_lens=lens,
                          scale=wl.default_scale(w.head_dim), new_key=w.tail_key[last], new_value=w.tail_value[last],
                          new_token_pos=lens.astype(np.int64) - 1)
    used = {int(tables[b, j]) for b in range(len(seqs)) for j in range((int(lens[b]) + bs - 1) // bs)}
    unique_bytes = len(used) * 2 * w.num_kv_heads * bs * w.head_dim * 2
    return inp, tables, lens, np.asarray(slots, dtype=np.int64), n_cow, unique_bytes


class _ModelPool:
    """The oracle's allocator model behind the product pool's method names (reference arm only)."""

    def __init__(self, num_blocks: int, block_size: int, free_order):
        from oracle.block_pool import SequencePool

        self.m = SequencePool(num_blocks, block_size, free_order=free_order)

    def create(self):
        return self.m.create()

    def fork(self, sid):
        return self.m.fork(sid)

    def append(self, sid):
        res = self.m.append(sid)
        return res.slot, res.cow

    def append_batch(self, ids):
        slots, pairs = [], []
        for sid in ids:
            slot, pair = self.append(sid)
            slots.append(slot)
            if pair:
                pairs.append(pair)
        return np.asarray(slots, dtype=np.int64), pairs

    def block_tables(self, ids, width):
        return self.m.block_tables(ids, width)

    def swap_to(self, dst, sid):
        new_sid, pairs = self.m.swap_to(dst.m, sid)
        return new_sid, np.asarray(pairs, dtype=np.int64).reshape(-1, 2)

    def check_invariants(self):
        bad = self.m.invariants()
        assert not bad, bad


def make_pool(num_blocks: int, block_size: int, free_order, model: bool = False):
    """The product block pool, or (``model``) the oracle's allocator model with the same free order."""
    if model:
        return _ModelPool(num_blocks, block_size, free_order)
    import paged_kv_cache_129_gb300 as pa

    return pa.BlockPool(num_blocks, block_size, free_order=free_order)


def pool_tables(inp, model: bool = False):
    """Block tables and new-token slots from the host block pool (a shuffled free list).

    Each sequence appends its L-1 context tokens, then the step's new token is
    appended for all sequences at once; the decode attends over L tokens.  With
    ``model`` the oracle's allocator model stands in for the product pool (the
    reference arm maps no product code); both give the same tables and slots.
    """
    rng = np.random.default_rng(12345)
    pool = make_pool(inp.num_blocks, inp.block_size, rng.permutation(inp.num_blocks), model)
    ids = [pool.create() for _ in range(inp.num_seqs)]
    q_len = inp.q.shape[1] if inp.q.ndim == 4 else 1
    for sid, L in zip(ids, inp.context_lens):
        for _ in range(int(L) - q_len):
            pool.append(sid)
    if inp.new_key is not None:
        rounds = []
        for _ in range(q_len):  # the step's new tokens, one batch append per token
            slots, pairs = pool.append_batch(ids)
            assert len(pairs) == 0
            rounds.append(np.asarray(slots, dtype=np.int64))
        slots = rounds[0] if q_len == 1 else np.stack(rounds, axis=1).reshape(-1)  # [B, q_len] order
    else:
        for sid in ids:
            pool.append(sid)
        slots = None
    width = int((int(inp.context_lens.max()) + inp.block_size - 1) // inp.block_size)
    tables, lens = pool.block_tables(ids, width)
    assert np.array_equal(lens, inp.context_lens)
    pool.check_invariants()
    return tables, lens, slots


def rep_times(torch, stream, call, reps: int, steps_per_rep: int, first: int = 0):
    """Per-rep device times (ms per step): ``reps`` sub-regions of ``steps_per_rep`` calls back to back,
    one event at each sub-region boundary only (an event between two launches breaks their programmatic
    dependent launch, so there is one such break per sub-region, not per call)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    i = first
    for r in range(reps):
        for _ in range(steps_per_rep):
            call(i)
            i += 1
        evs[r + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[r].elapsed_time(evs[r + 1]) / steps_per_rep for r in range(reps)]


def rep_summary(per_step_ms, bytes_per_step: float, steps_per_rep: int, what: str) -> dict:
    s = sorted(per_step_ms)
    med = statistics.median(s)
    return {"reps": len(s), "steps_per_rep": steps_per_rep, "median_ms_per_step": round(med, 5),
            "min_ms_per_step": round(s[0], 5), "max_ms_per_step": round(s[-1], 5),
            "median_value": round(bytes_per_step / (med / 1e3) / 1e9, 2),
            "best_value": round(bytes_per_step / (s[0] / 1e3) / 1e9, 2), "unit": UNIT,
            "timing": f"{what}: CUDA events at the {len(s) + 1} sub-region boundaries only, on the launch stream"}


def long_context_leg(args, device, peak: float, steps: int, warmup: int) -> dict:
    """The long-context split-KV configuration (8 sequences, 32 q / 8 kv heads, d 128, bf16, L in
    [32768, 131072]) timed in the same run as the headline: one pa_decode_ex call per step on inputs
    resident in HBM (2.2 GB of pages per step, far above L2), lean schedule + merge."""
    import torch

    import paged_kv_cache_129_gb300 as pa

    inp = build_batch("long_context", rank_seed(args.seed, 0))
    tables, lens, _ = pool_tables(inp)
    B, Hq, Hkv, d, bs = inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    kc, vc, q = up(inp.key_cache), up(inp.value_cache), up(inp.q)
    del inp.key_cache, inp.value_cache
    bt, dl = torch.from_numpy(tables).to(device), torch.from_numpy(lens).to(device)
    out = torch.empty_like(q)
    max_ctx = int(lens.max())
    plan = pa.decode_plan(B, Hq, Hkv, d, bs, tables.shape[1], torch.bfloat16, max_context_len=max_ctx)
    ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    lib = pa.library()
    stream = torch.cuda.current_stream(device)
    a = [out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), dl.data_ptr(), B, Hq, Hkv, d,
         bs, tables.shape[1], inp.num_blocks, float(inp.scale), 2, ws.data_ptr(), ws.numel(), max_ctx, 0,
         pa.KERNELS["auto"], int(stream.cuda_stream)]

    def call(i):
        if lib.pa_decode_ex(*a) != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())

    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    pa.check_error()
    nbytes = decode_bytes(lens, Hq, Hkv, d, 2, bs)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_begin = time.monotonic()
    e0.record(stream)
    for i in range(steps):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    pa.check_error()
    ms = e0.elapsed_time(e1) / steps
    # >= 50 reps of about 30 ms each (the clock sampler sees this region)
    per_rep = max(1, int(math.ceil(30.0 / ms)))
    reps = rep_times(torch, stream, call, 50, per_rep)
    t_end = time.monotonic()
    pa.check_error()
    value = nbytes / (ms / 1e3) / 1e9
    return {"window": (t_begin, t_end), "workload": WORKLOAD_DESCRIPTIONS["long_context"], "name": "long_context", "step": "pa_decode",
            "schedule": SCHEDULE_NAMES[plan.schedule],
            "value": round(value, 2), "unit": UNIT, "pct_of_hbm_peak": round(100 * value / peak, 2),
            "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 5),
            "queries_per_s": round(B / (ms / 1e3), 1),
            "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(value / peak, 4), "traffic": stored_traffic("long_context"),
                         "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": round(ms, 5),
                         "kernel": "pa_decode call (paged_decode_lean_kernel + lean_merge_kernel)"
                                   if plan.schedule == 1 else "pa_decode call (paged_decode_kernel)"},
            "per_rep": rep_summary(reps, nbytes, per_rep, "pa_decode calls"),
            "gpu_launches": steps * (2 if (plan.schedule in (1, 2) or plan.max_parts > 1) else 1),
            "l2": f"pages touched per step {pages_touched_bytes(lens, Hkv, d, 2, bs) / 1e6:.0f} MB, above L2"}


def run_ours(args, rank: int, world: int, local_rank: int, sub: bool = False):
    """Time one workload. sub=False: the headline run (prints the JSON line); sub=True: a side
    record for the headline line (returned as a dict: no clock sampler, e2e or CPU leg of its own)."""
    import torch

    import paged_kv_cache_129_gb300 as pa

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    pa.library()

    prefix = args.workload.startswith("prefix_cow")
    n_cow, unique_bytes = 0, None
    if prefix:
        inp, tables, lens, slots, n_cow, unique_bytes = prefix_batch(args.workload, rank_seed(args.seed, rank))
    else:
        inp = build_batch(args.workload, rank_seed(args.seed, rank))
        tables, lens, slots = pool_tables(inp)
    inp.block_tables = tables
    tdtype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[inp.dtype]

    def up(a):
        a = np.ascontiguousarray(a)
        if inp.dtype in ("bf16", "f16"):
            return torch.from_numpy(a.view(np.int16)).to(device).view(tdtype)
        return torch.from_numpy(a).to(device)

    eb = inp.elem_bytes
    B, Hq, Hkv, d, bs = inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size
    q_len = inp.q.shape[1] if inp.q.ndim == 4 else 1  # query tokens per sequence (verify step: > 1)
    fp8 = args.workload.endswith("_fp8")  # E4M3 caches with a scale per (block, kv head)
    dec_bytes = decode_bytes(lens, Hq, Hkv, d, eb, bs, q_len)
    ntok = 0 if slots is None else len(slots)
    wr_bytes = write_bytes(ntok, Hkv, d, eb)
    if fp8:
        dec_bytes = decode_bytes_fp8(lens, Hq, Hkv, d, eb, bs)
        wr_bytes = write_bytes_fp8(ntok, Hkv, d, eb)
    step_bytes = dec_bytes + wr_bytes
    touched = pages_touched_bytes(lens, Hkv, d, 1 if fp8 else eb, bs)
    if prefix:
        touched = unique_bytes  # shared pages are read once per step

    l2 = L2_BYTES_DEFAULT
    try:
        l2 = torch.cuda.get_device_properties(device).L2_cache_size or l2
    except AttributeError:
        pass
    # Rotate over cache replicas so that a step never finds its pages in L2 from the previous one.
    replicas = 1 if touched >= 3 * l2 else max(2, math.ceil(2 * l2 / touched) + 1)
    kc0, vc0 = up(inp.key_cache), up(inp.value_cache)
    if fp8:
        # quantise the whole pool through the product writer (every slot once), then drop the sources
        from paged_kv_cache_129_gb300 import workloads as wl

        ks_np, vs_np = wl.fp8_scales(inp.key_cache, inp.dtype), wl.fp8_scales(inp.value_cache, inp.dtype)
        ksd, vsd = torch.from_numpy(ks_np).to(device), torch.from_numpy(vs_np).to(device)
        nb_ = inp.num_blocks
        all_slots = torch.arange(nb_ * bs, dtype=torch.int64, device=device)
        interleaved = args.fp8_layout == "interleaved"
        if interleaved:  # [N, H_kv, 2, bs, d]: one record per (block, kv head), K rows then V rows
            q8k, q8v = torch.empty(nb_, Hkv, 2, bs, d, dtype=torch.uint8, device=device), None
        else:
            q8k = torch.empty(nb_, Hkv, bs, d, dtype=torch.uint8, device=device)
            q8v = torch.empty_like(q8k)
        pa.write_kv_fp8(kc0.permute(0, 2, 1, 3).reshape(nb_ * bs, Hkv, d).contiguous(),
                        vc0.permute(0, 2, 1, 3).reshape(nb_ * bs, Hkv, d).contiguous(), q8k, q8v, ksd, vsd, all_slots)
        torch.cuda.synchronize()
        del kc0, vc0, all_slots
        kc0, vc0 = q8k, q8v  # q8v None: the interleaved layout
    kcs, vcs = [kc0], [vc0]
    for _ in range(replicas - 1):
        kcs.append(kc0.clone())
        vcs.append(vc0.clone() if vc0 is not None else None)
    q = up(inp.q)
    bt = torch.from_numpy(tables).to(device)
    dl = torch.from_numpy(lens).to(device)
    out = torch.empty_like(q)
    has_write = slots is not None
    if has_write:
        nk, nv = up(inp.new_key), up(inp.new_value)
        sl = torch.from_numpy(slots).to(device)
    max_ctx = int(lens.max())
    if fp8:
        plan = pa.DecodePlan()
        plan.kernel, plan.schedule, plan.partition_pages, plan.max_parts = 1, 1, 0, 0
        plan.workspace_bytes = pa.decode_fp8_workspace_size(B, Hq, Hkv, d, bs, tables.shape[1], tdtype)
        plan.grid_ctas = 0
    else:
        plan = pa.decode_plan(B, Hq, Hkv, d, bs, tables.shape[1], tdtype, max_context_len=max_ctx,
                              partition_pages=args.partition_pages, kernel=args.kernel, q_len=q_len)
    ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    lib = pa.library()
    stream = torch.cuda.current_stream(device)
    sptr = int(stream.cuda_stream)
    code = {"f32": 0, "f16": 1, "bf16": 2}[inp.dtype]
    kern = pa.KERNELS[args.kernel]

    fused = has_write and args.step == "append" and q_len == 1
    if fused:
        # pa_decode_append / pa_decode_fp8_append write at the slot of position L - 1: the pool handed
        # out exactly those
        live = lens >= 1
        derived = tables[np.arange(B), (lens - 1) // bs].astype(np.int64) * bs + (lens - 1) % bs
        assert np.array_equal(np.asarray(slots)[live], derived[live])

    # Pre-marshalled C-ABI argument lists (the timed loop only calls the library).
    def ptr(t):
        return t.data_ptr() if t is not None else None

    dec_args = [[out.data_ptr(), q.data_ptr(), kcs[r].data_ptr(), ptr(vcs[r]), bt.data_ptr(), dl.data_ptr(),
                 B] + ([q_len] if q_len > 1 else []) + [Hq, Hkv, d, bs, tables.shape[1], inp.num_blocks,
                 float(inp.scale), code, ws.data_ptr(), ws.numel(), max_ctx, args.partition_pages, kern, sptr]
                for r in range(replicas)]
    decode_fn = lib.pa_decode_multi if q_len > 1 else lib.pa_decode_ex
    wr_args = ([[nk.data_ptr(), nv.data_ptr(), kcs[r].data_ptr(), ptr(vcs[r]), sl.data_ptr(), ntok, Hkv, d, bs,
                 inp.num_blocks, code, sptr] for r in range(replicas)] if has_write else None)
    if fp8:
        decode_fn = lib.pa_decode_fp8
        vptr = [vcs[r].data_ptr() if vcs[r] is not None else None for r in range(replicas)]
        dec_args = [[out.data_ptr(), q.data_ptr(), kcs[r].data_ptr(), vptr[r], ksd.data_ptr(),
                     vsd.data_ptr(), bt.data_ptr(), dl.data_ptr(), B, Hq, Hkv, d, bs, tables.shape[1], inp.num_blocks,
                     float(inp.scale), code, ws.data_ptr(), ws.numel(), sptr] for r in range(replicas)]
        write_fn = lib.pa_write_kv_fp8
        if has_write:
            wr_args = [[nk.data_ptr(), nv.data_ptr(), kcs[r].data_ptr(), vptr[r], ksd.data_ptr(),
                        vsd.data_ptr(), sl.data_ptr(), ntok, Hkv, d, bs, inp.num_blocks, code, sptr]
                       for r in range(replicas)]
    else:
        write_fn = lib.pa_write_kv
    app_args = ([[out.data_ptr(), q.data_ptr(), nk.data_ptr(), nv.data_ptr(), kcs[r].data_ptr(), ptr(vcs[r]),
                  bt.data_ptr(), dl.data_ptr(), B, Hq, Hkv, d, bs, tables.shape[1], inp.num_blocks, float(inp.scale),
                  code, ws.data_ptr(), ws.numel(), max_ctx, args.partition_pages, kern, sptr]
                 for r in range(replicas)] if fused else None)
    append_fn = lib.pa_decode_append
    if fused and fp8:
        append_fn = lib.pa_decode_fp8_append
        app_args = [[out.data_ptr(), q.data_ptr(), nk.data_ptr(), nv.data_ptr(), kcs[r].data_ptr(), ptr(vcs[r]),
                     ksd.data_ptr(), vsd.data_ptr(), bt.data_ptr(), dl.data_ptr(), B, Hq, Hkv, d, bs, tables.shape[1],
                     inp.num_blocks, float(inp.scale), code, ws.data_ptr(), ws.numel(), sptr]
                    for r in range(replicas)]
    # the decode kernel, plus the merge kernel (always for the lean schedule, when split for
    # the grid one), plus the write kernel when it is a call of its own
    merge_launches = 1 if (plan.schedule in (1, 2) or plan.max_parts > 1) else 0
    launches_per_step = (1 if (has_write and not fused) else 0) + 1 + merge_launches

    def step(i):
        r = i % replicas
        if fused:
            if append_fn(*app_args[r]) != 0:
                raise RuntimeError(lib.pa_last_error_string().decode())
            return
        if has_write and write_fn(*wr_args[r]) != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())
        if decode_fn(*dec_args[r]) != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())

    def decode_call(i):
        # the step's decode call: pa_decode_append / pa_decode_fp8_append (rewriting the same rows),
        # pa_decode_ex, pa_decode_multi or pa_decode_fp8
        status = append_fn(*app_args[i % replicas]) if fused else decode_fn(*dec_args[i % replicas])
        if status != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())

    sampler = None if sub else ClockSampler(gpu_selector(device))
    if sampler is not None:
        sampler.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    pa.check_error()

    K = args.steps
    # Timed region 1, the headline: K whole steps back to back, events only around them
    # (an event between two launches would break their programmatic dependent launch).
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_begin = time.monotonic()
    ev_start.record(stream)
    for i in range(K):
        step(i)
    ev_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    pa.check_error()
    elapsed_ms = ev_start.elapsed_time(ev_end)
    # Timed region 2, for the roofline: the pa_decode call alone, K calls back to back on
    # the same stream; its average duration is the region's time / K.
    ev_d0, ev_d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev_d0.record(stream)
    for i in range(K):
        decode_call(i)
    ev_d1.record(stream)
    torch.cuda.synchronize()
    pa.check_error()
    dec_avg_ms = ev_d0.elapsed_time(ev_d1) / K
    # Timed region 3, the spread: 50 reps of whole steps (about 30 ms each, so the clock sampler
    # sees this region too), events at the rep boundaries only.
    per_rep = max(1, int(math.ceil(30.0 / max(elapsed_ms / K, 1e-3))))
    rep_ms = rep_times(torch, stream, step, 50, per_rep, first=K)
    windows = [(t_begin, time.monotonic())]
    pa.check_error()
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "of measured (MEASURED_PEAKS.json hbm_gbs)" if peak else "of fallback"
    peak = float(peak or FALLBACK_HBM_GBS)
    # The long-context configuration (the other >= 70 % of HBM target), timed in the same run.
    long_leg = None
    if not sub and args.workload == "qwen_gqa" and not args.no_long_context and world == 1:
        long_leg = long_context_leg(args, device, peak, steps=max(K, 20), warmup=args.warmup)
        windows.append(long_leg.pop("window"))
    # The other hot-path rows (FP8 cache, speculative verify, many short MHA requests), each a
    # side record timed the same way in the same run.
    side = []
    if not sub and args.workload == "qwen_gqa" and not args.no_side_workloads and world == 1:
        for w in SIDE_WORKLOADS:
            sargs = argparse.Namespace(**vars(args))
            sargs.workload, sargs.kernel, sargs.partition_pages = w, "auto", 0
            sargs.no_e2e = sargs.no_cpu_baseline = sargs.no_long_context = sargs.no_side_workloads = True
            sargs.steps = max(K, 20)
            rec = run_ours(sargs, rank, world, local_rank, sub=True)
            windows.append(rec.pop("window"))
            side.append(rec)
    t_end = time.monotonic()
    barrier(world)
    if sampler is not None:
        sampler.stop()
    elapsed_ms_max = max_over_ranks(elapsed_ms, world)
    total_bytes = sum_over_ranks(float(step_bytes) * K, world)
    total_seqs = sum_over_ranks(float(B) * K, world)
    value = total_bytes / (elapsed_ms_max / 1e3) / 1e9
    ms_per_step = elapsed_ms_max / K

    # e2e: the public step runner (pa.DecodeStepper): every step one packed upload of the step's inputs
    # from pinned host memory, the decode call, one download of the output; two slots, so the upload of
    # step i + 1 overlaps the decode of step i.
    e2e = None
    # the step runner does one decode call per step (no separate write, one query token)
    if not args.no_e2e and (fused or fp8 or not has_write) and q_len == 1:
        step_append = fused or (fp8 and has_write)
        if fp8:
            stepper = pa.DecodeStepper(kcs[0], vcs[0], B, Hq, tables.shape[1], scale=inp.scale, append=step_append,
                                       tables="deltas", k_scale=ksd, v_scale=vsd, query_dtype=tdtype,
                                       fp8_write="fused" if fused else "separate")
        else:
            stepper = pa.DecodeStepper(kcs[0], vcs[0], B, Hq, tables.shape[1], scale=inp.scale, append=fused,
                                       max_context_len=max_ctx, partition_pages=args.partition_pages,
                                       kernel=args.kernel, tables="deltas")
        # the device tables are kept by delta uploads: the first step sends every entry, later steps
        # re-send the tail entry of B / bs rows (the rate at which one token a step opens new blocks)
        nblk = (lens + bs - 1) // bs
        full_deltas = np.array([(r, j, tables[r, j]) for r in range(B) for j in range(nblk[r])],
                               np.int32).reshape(-1, 3)
        churn = max(1, B // bs)
        tail = np.maximum(nblk - 1, 0).astype(np.int32)

        def fill(view, arr):
            a = np.ascontiguousarray(arr)
            t = torch.from_numpy(a.view(np.int16) if inp.dtype in ("bf16", "f16") else a)
            view.copy_(t.view(view.dtype) if inp.dtype in ("bf16", "f16") else t)

        for sl in range(stepper.slots):
            v = stepper.inputs(sl)
            fill(v.query, inp.q)
            v.context_lens.copy_(torch.from_numpy(lens))
            if step_append:
                fill(v.new_key, inp.new_key)
                fill(v.new_value, inp.new_value)
            if fp8 and step_append and not fused:
                v.slots.copy_(torch.from_numpy(np.asarray(slots, dtype=np.int64)))

        def e2e_run(n, first=False):
            for i in range(n):
                dv = stepper.inputs(i).deltas.numpy()
                if first and i == 0:
                    k = len(full_deltas)
                    dv[:k] = full_deltas
                else:
                    rows = (i * churn + np.arange(churn)) % B
                    k = churn
                    dv[:k, 0], dv[:k, 1], dv[:k, 2] = rows, tail[rows], tables[rows, tail[rows]]
                stepper.launch(i, kcs[i % replicas], vcs[i % replicas], num_deltas=k)
                if i >= 1:
                    stepper.result(i - 1)
            stepper.result(n - 1)

        e2e_run(min(args.warmup, 20) + 1, first=True)
        torch.cuda.synchronize()
        Ke = max(1, args.e2e_steps)  # a steady-state run, whatever K is (K = 20 would be mostly pipeline fill)
        # three timed runs of Ke steps each; the line reports the median run (the host thread paces
        # this leg, and one run can lose its core to another process)
        runs = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            torch.cuda.synchronize()
            e0.record(stream)
            stepper.upload.wait_event(e0)
            e2e_run(Ke)
            e1.record(stream)
            torch.cuda.synchronize()
            barrier(world)
            pa.check_error()
            runs.append(max_over_ranks(e0.elapsed_time(e1), world))
        e_ms = sorted(runs)[1]
        e_bytes = sum_over_ranks(float(step_bytes) * Ke, world)
        e2e = {"value": round(e_bytes / (e_ms / 1e3) / 1e9, 2), "unit": UNIT, "steps": Ke,
               "ms_per_step": round(e_ms / Ke, 5), "statistic": "median of 3 timed runs",
               "runs_ms_per_step": [round(r / Ke, 5) for r in runs],
               "h2d_bytes_per_step": int(stepper.h2d_bytes),
               "d2h_bytes_per_step": int(stepper.d2h_bytes),
               "note": f"pa.DecodeStepper ({'pa_decode_fp8_append' if fused and fp8 else 'pa_decode_append' if fused else 'pa_write_kv_fp8 + pa_decode_fp8' if fp8 and step_append else 'pa_decode_fp8' if fp8 else 'pa_decode'}, tables kept on the "
                       "device by deltas): every step one upload of the packed inputs (queries" +
                       (", new K/V" if step_append else "") + (", slots" if fp8 and step_append and not fused else "") +
                       f", lengths, {churn} block-table deltas) from pinned host "
                       "memory, pa_apply_table_deltas and the decode on the compute stream, one download of the "
                       "output, inside the timed region; two slots, the next upload overlapping the current decode"}

    call_bytes = step_bytes if fused else dec_bytes  # the appending call also does the write
    if prefix:
        # every sequence's K/V would exceed HBM peak through L2 hits on the shared prefix:
        # the roofline counts each distinct page once (plus q, out, tables, lengths, write)
        call_bytes = unique_bytes + (call_bytes - 2 * int(lens.sum()) * Hkv * d * eb)
    achieved = call_bytes / (dec_avg_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": stored_traffic(args.workload),
                "kernel": (("pa_decode_fp8_append" if fused and fp8 else "pa_decode_append" if fused else
                            "pa_decode_multi" if q_len > 1 else
                            "pa_decode_fp8" if fp8 else "pa_decode") +
                           " call (" +
                           ("paged_decode_lean_kernel + lean_merge_kernel)" if plan.schedule == 1 else
                            "paged_decode_rs_lean_kernel + rs_lean_merge_kernel)" if plan.schedule == 2 else
                            "paged_decode_kernel" + (" + splitkv_merge_kernel)" if plan.max_parts > 1 else ")"))),
                "algorithmic_bytes_per_launch": call_bytes, "pages_touched_bytes": touched,
                "avg_launch_ms": round(dec_avg_ms, 5),
                "timing": f"CUDA events around {K} back-to-back calls on the launch stream",
                "peak_source": peak_src}

    if sub:
        return {"window": windows[0], "workload": WORKLOAD_DESCRIPTIONS[args.workload], "name": args.workload,
                "step": roofline["kernel"].split(" call")[0], "dtype": DTYPE_NAMES[inp.dtype],
                "value": round(value, 2), "unit": UNIT, "pct_of_hbm_peak": round(100 * value / peak, 2),
                "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
                "queries_per_s": round(total_seqs / (elapsed_ms_max / 1e3), 1),
                "step_bytes": step_bytes, "roofline": roofline,
                "per_rep": rep_summary(rep_ms, step_bytes, per_rep, "whole steps"),
                "gpu_launches": launches_per_step * K,
                "l2": f"{replicas} cache replicas rotated per step (pages touched per step "
                      f"{touched / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        fp8_host = None
        if fp8:
            # the oracle quantises its own copy of the pool (every slot), then the step's new tokens
            nb_ = inp.num_blocks
            kq, vq = np.zeros((nb_, Hkv, bs, d), np.uint8), np.zeros((nb_, Hkv, bs, d), np.uint8)
            oracle.write_kv_fp8(np.ascontiguousarray(inp.key_cache.transpose(0, 2, 1, 3).reshape(nb_ * bs, Hkv, d)),
                                np.ascontiguousarray(inp.value_cache.transpose(0, 2, 1, 3).reshape(nb_ * bs, Hkv, d)),
                                inp.dtype, kq, vq, ks_np, vs_np, np.arange(nb_ * bs, dtype=np.int64))
            if has_write:
                oracle.write_kv_fp8(inp.new_key.reshape(-1, Hkv, d), inp.new_value.reshape(-1, Hkv, d), inp.dtype,
                                    kq, vq, ks_np, vs_np, slots)
            fp8_host = (kq, vq, ks_np, vs_np)
        elif has_write:
            oracle.write_kv(inp.new_key.reshape(-1, Hkv, d), inp.new_value.reshape(-1, Hkv, d), inp.key_cache,
                            inp.value_cache, slots)
        threads = os.cpu_count() or 1
        r = time_oracle_parallel(inp, args.cpu_budget, threads, fp8_host)
        cpu = {"value": round(r["bytes"] / r["seconds"] / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {r['seqs']} of {B} sequences, all {Hq} heads ({r['rows']} output rows), "
                         f"fp64 C oracle, one sequence per task on {threads} threads, {r['seconds']:.1f} s",
               "seconds": round(r["seconds"], 2), "cpu_model": cpu_model(),
               "single_thread": {"value": round(r["single_thread_gbs"], 4), "unit": UNIT,
                                 "sample": f"sequence 0, all heads, {r['single_thread_seconds']:.2f} s"}}

    clocks = sampler.summary(t_begin, t_end, windows)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAMES[inp.dtype], "data": "synthetic",
        "config": {"workload": WORKLOAD_DESCRIPTIONS[args.workload], "name": args.workload,
                   "step": ("pa_decode_fp8_append (new token per sequence quantised at L - 1, then decode)"
                            if fused and fp8
                            else "pa_decode_append (new token per sequence written at L - 1, then decode)" if fused
                            else "pa_write_kv_fp8 (new token per sequence) + pa_decode_fp8" if fp8 and has_write
                            else "pa_decode_fp8" if fp8
                            else "pa_write_kv (new token per sequence) + pa_decode" if has_write
                            else "pa_decode_multi" if q_len > 1 else "pa_decode"),
                   "l2": f"{replicas} cache replicas rotated per step (pages touched per step "
                         f"{touched / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)",
                   **({"copy_on_write_copies": n_cow, "unique_page_bytes": unique_bytes,
                       "value_kind": "effective GB/s: every sequence's K/V counted, shared pages once per "
                                     "sequence (above HBM peak through L2 hits)"} if prefix else {}),
                   "kernel": {1: "mma", 2: "simt"}[plan.kernel],
                   "schedule": SCHEDULE_NAMES[plan.schedule],
                   "partition_pages": plan.partition_pages,
                   "max_parts": plan.max_parts, "grid_ctas": plan.grid_ctas,
                   "parallelism": f"{world} independent replicas (one batch per GPU)"},
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "queries_per_s": round(total_seqs / (elapsed_ms_max / 1e3), 1),
        "head_queries_per_s": round(total_seqs * Hq / (elapsed_ms_max / 1e3), 1),
        "step_bytes": step_bytes,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "per_rep": rep_summary(rep_ms, step_bytes, per_rep, "whole steps"),
        "clocks": clocks,
    }
    if long_leg is not None:
        line["long_context"] = long_leg
    if side:
        line["side_workloads"] = {r["name"]: r for r in side}
        line["gpu_launches_side_workloads"] = sum(r["gpu_launches"] for r in side)
    print(json.dumps(line), flush=True)


LAYERS = 28


def run_layers(args, rank: int, world: int, local_rank: int) -> None:
    """Whole-model step: pa_write_kv_layers for all layers, then pa_decode_ex per layer."""
    import torch

    import paged_kv_cache_129_gb300 as pa

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    lib = pa.library()
    seed = rank_seed(args.seed, rank)
    inp = build_batch("qwen_gqa", seed)  # lengths, tables and slots of the layer batch
    tables, lens, slots = pool_tables(inp)
    B, Hq, Hkv, d, bs, nb = inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size, inp.num_blocks
    gen = torch.Generator(device=device).manual_seed(seed)

    def randn(*shape):
        return torch.randn(*shape, device=device, generator=gen).to(torch.bfloat16)

    kcs = [randn(nb, Hkv, bs, d) for _ in range(LAYERS)]
    vcs = [randn(nb, Hkv, bs, d) for _ in range(LAYERS)]
    qs = [randn(B, Hq, d) for _ in range(LAYERS)]
    nks = [randn(B, Hkv, d) for _ in range(LAYERS)]
    nvs = [randn(B, Hkv, d) for _ in range(LAYERS)]
    outs = [torch.empty_like(q) for q in qs]
    bt = torch.from_numpy(tables).to(device)
    dl = torch.from_numpy(lens).to(device)
    sl = torch.from_numpy(slots).to(device)
    max_ctx = int(lens.max())
    plan = pa.decode_plan(B, Hq, Hkv, d, bs, tables.shape[1], torch.bfloat16, max_context_len=max_ctx)
    ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sptr = int(stream.cuda_stream)
    import ctypes

    arr = ctypes.c_void_p * LAYERS
    wl_args = [arr(*[t.data_ptr() for t in nks]), arr(*[t.data_ptr() for t in nvs]),
               arr(*[t.data_ptr() for t in kcs]), arr(*[t.data_ptr() for t in vcs]), LAYERS, sl.data_ptr(), B, Hkv,
               d, bs, nb, 2, sptr]
    dec_args = [[outs[l].data_ptr(), qs[l].data_ptr(), kcs[l].data_ptr(), vcs[l].data_ptr(), bt.data_ptr(),
                 dl.data_ptr(), B, Hq, Hkv, d, bs, tables.shape[1], nb, float(inp.scale), 2, ws.data_ptr(),
                 ws.numel(), max_ctx, 0, 0, sptr] for l in range(LAYERS)]

    def write_all():
        if lib.pa_write_kv_layers(*wl_args) != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())

    def decode_all():
        for l in range(LAYERS):
            if lib.pa_decode_ex(*dec_args[l]) != 0:
                raise RuntimeError(lib.pa_last_error_string().decode())

    def region(fn, k):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(k):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    sampler = ClockSampler(gpu_selector(device))
    sampler.start()
    for _ in range(args.warmup):
        write_all()
        decode_all()
    torch.cuda.synchronize()
    pa.check_error()
    K = args.steps
    barrier(world)
    t_begin = time.monotonic()
    step_ms = region(lambda: (write_all(), decode_all()), K)
    write_ms = region(write_all, K)
    t_end = time.monotonic()
    barrier(world)
    sampler.stop()
    pa.check_error()
    dec_bytes = decode_bytes(lens, Hq, Hkv, d, 2, bs)
    wr_bytes = write_bytes(B, Hkv, d, 2)
    step_bytes = LAYERS * (dec_bytes + wr_bytes)
    ms = max_over_ranks(step_ms, world)
    value = sum_over_ranks(float(step_bytes) * K, world) / (ms / 1e3) / 1e9
    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
    dec_avg_ms = (step_ms - write_ms) / (K * LAYERS)
    write_avg_ms = write_ms / K
    clocks = sampler.summary(t_begin, t_end)
    if rank != 0:
        return
    merge = 1 if (plan.schedule in (1, 2) or plan.max_parts > 1) else 0
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESCRIPTIONS["qwen_gqa_layers28"], "name": "qwen_gqa_layers28",
                   "layers": LAYERS, "step": "pa_write_kv_layers (28 layers, one launch) + 28 x pa_decode_ex",
                   "l2": f"28 layers' pages per step ({LAYERS * pages_touched_bytes(lens, Hkv, d, 2, bs) / 1e9:.1f} "
                         "GB) pass through L2 once",
                   "parallelism": f"{world} independent replicas (one model per GPU)"},
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "queries_per_s": round(B * K / (ms / 1e3), 1),
        "step_bytes": step_bytes,
        "roofline": {"bound": "hbm", "achieved": round(dec_bytes / (dec_avg_ms / 1e3) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(dec_bytes / (dec_avg_ms / 1e3) / 1e9 / peak, 4),
                     "traffic": None, "kernel": "pa_decode call per layer (decode step time minus the write's)",
                     "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_ms": round(dec_avg_ms, 5),
                     "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)",
                     "write_kv_layers": {"bytes_per_launch": LAYERS * wr_bytes, "avg_launch_ms": round(write_avg_ms, 5),
                                         "achieved_gbs": round(LAYERS * wr_bytes / (write_avg_ms / 1e3) / 1e9, 1),
                                         "timing": f"CUDA events around {K} back-to-back launches"}},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": K * (1 + LAYERS * (1 + merge)),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def swap_plan(seed: int, steps: int, num_blocks: int = 20000, num_seqs: int = 64, group: int = SWAP_GROUP,
              block_size: int = 16, model: bool = False):
    """Host side of the swap workload (no GPU).  Sequences are built through the product block pool (the
    oracle's allocator model with ``model``, for the reference arm: the same pairs); the
    groups of ``group`` sequences take turns: step k swaps group k out to host pool k % 2 and group k - 1
    back in from host pool (k - 1) % 2, so the two copies of a step can run at once.  Per step the pool
    decides the swap-in first (its device blocks come from blocks free before this step's swap-out
    releases any) and then the swap-out (into the other host pool), so the two copies touch disjoint
    blocks on both sides.  Returns (per-step (out pairs, out host pool, in pairs, in host pool), host pool
    size, seconds of pool work per step, lengths)."""
    assert 2 * group <= num_seqs
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 4097, size=num_seqs)
    dev = make_pool(num_blocks, block_size, rng.permutation(num_blocks), model)
    ids = [dev.create() for _ in range(num_seqs)]
    for t in range(int(lens.max())):
        dev.append_batch([sid for sid, n in zip(ids, lens) if n > t])
    host_blocks = int(np.sort((lens + block_size - 1) // block_size)[-group:].sum())
    hosts = [make_pool(host_blocks, block_size, np.arange(host_blocks), model) for _ in range(2)]
    away = {}  # sequence index -> id in its host pool
    plan, t_pool = [], 0.0
    none = np.zeros((0, 2), np.int64)
    for k in range(steps):
        t0 = time.perf_counter()
        ins = []
        if k > 0:
            for j in range(group):
                i = ((k - 1) * group + j) % num_seqs
                ids[i], pairs = hosts[(k - 1) % 2].swap_to(dev, away.pop(i))
                ins.append(pairs)
        outs = []
        for j in range(group):
            i = (k * group + j) % num_seqs
            away[i], pairs = dev.swap_to(hosts[k % 2], ids[i])
            outs.append(pairs)
        t_pool += time.perf_counter() - t0
        plan.append((np.concatenate(outs), k % 2, np.concatenate(ins) if ins else none, (k - 1) % 2))
    for p in [dev] + hosts:
        p.check_invariants()
    return plan, host_blocks, t_pool / max(steps, 1), lens


def run_swap(args, rank: int, world: int, local_rank: int) -> None:
    """The swap workload: device time of each step's swap-out and swap-in launches, on two streams."""
    import torch

    import paged_kv_cache_129_gb300 as pa

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    lib = pa.library()
    nb, hkv, bs, d = 20000, 4, 16, 128
    n_steps = args.warmup + args.steps
    plan, host_blocks, pool_s, lens = swap_plan(rank_seed(args.seed, rank), n_steps)
    gen = torch.Generator(device=device).manual_seed(rank_seed(args.seed, rank))
    kc = torch.randn(nb, hkv, bs, d, device=device, generator=gen).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, device=device, generator=gen).to(torch.bfloat16)
    hk = [torch.empty(host_blocks, hkv, bs, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hv = [torch.empty(host_blocks, hkv, bs, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    # every step's pairs in page-locked host memory: the kernel reads them there
    offs, flat, pos = [], [], 0
    for out_p, _, in_p, _ in plan:
        offs.append((pos, len(out_p), pos + len(out_p), len(in_p)))
        flat += [out_p, in_p]
        pos += len(out_p) + len(in_p)
    pairs = torch.from_numpy(np.concatenate(flat)).pin_memory()
    main = torch.cuda.current_stream(device)
    s_out, s_in = torch.cuda.Stream(device), torch.cuda.Stream(device)
    block_bytes = hkv * bs * d * 2
    base = pairs.data_ptr()
    done_out, done_in = torch.cuda.Event(), torch.cuda.Event()

    def step(k):
        o0, no, i0, ni = offs[k]
        _, ho, _, hi = plan[k]
        # a step's copies start when both copies of the previous step are done (their blocks are reused)
        s_out.wait_event(done_in)
        s_in.wait_event(done_out)
        if lib.pa_swap_blocks(hk[ho].data_ptr(), hv[ho].data_ptr(), kc.data_ptr(), vc.data_ptr(), base + 16 * o0,
                              no, hkv, d, bs, nb, host_blocks, 2, int(s_out.cuda_stream)) != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())
        if ni and lib.pa_swap_blocks(kc.data_ptr(), vc.data_ptr(), hk[hi].data_ptr(), hv[hi].data_ptr(),
                                     base + 16 * i0, ni, hkv, d, bs, host_blocks, nb, 2,
                                     int(s_in.cuda_stream)) != 0:
            raise RuntimeError(lib.pa_last_error_string().decode())
        done_out.record(s_out)
        done_in.record(s_in)
        return (no + ni) * 2 * block_bytes, no * 2 * block_bytes, ni * 2 * block_bytes, 1 + (ni > 0)

    def join():
        main.wait_stream(s_out)
        main.wait_stream(s_in)

    sampler = ClockSampler(gpu_selector(device))
    sampler.start()
    done_out.record(main)
    done_in.record(main)
    for k in range(args.warmup):
        step(k)
    join()
    torch.cuda.synchronize()
    pa.check_error()
    link = measure_link(torch, device)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_begin = time.monotonic()
    moved = d2h = h2d = launches = 0
    ev0.record(main)
    s_out.wait_stream(main)
    s_in.wait_stream(main)
    for k in range(args.warmup, n_steps):
        m, o, i, n = step(k)
        moved, d2h, h2d, launches = moved + m, d2h + o, h2d + i, launches + n
    join()
    ev1.record(main)
    torch.cuda.synchronize()
    t_end = time.monotonic()
    barrier(world)
    sampler.stop()
    pa.check_error()
    K = args.steps
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    value = sum_over_ranks(float(moved), world) / (ms / 1e3) / 1e9
    e2e_ms = ms + pool_s * 1e3 * K  # plus the host pool's decisions, made before the timed region
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_swap_oracle(plan[1], host_blocks, budget_s=min(args.cpu_budget, 10.0))
        cpu = {"value": r["gbs"], "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"step 1's {r['pairs']} pairs (out and in), oracle byte copy between two numpy pools, "
                         f"repeated {r['reps']} times ({r['seconds']:.1f} s)"}
    clocks = sampler.summary(t_begin, t_end)
    if rank != 0:
        return
    peak = link["both_gbs"]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESCRIPTIONS["swap_qwen"], "name": "swap_qwen",
                   "step": f"pa_swap_blocks out ({SWAP_GROUP} sequences' blocks, device -> host) on one stream and "
                           f"pa_swap_blocks in (the previous {SWAP_GROUP}, host -> device) on another, at once; "
                           "pairs read from page-locked host memory",
                   "l2": "host side of every copy crosses the link; device blocks change each step",
                   "host_pool_blocks": host_blocks, "mean_context": float(lens.mean()),
                   "parallelism": f"{world} independent replicas (one pool per GPU)"},
        "roofline": {"bound": "host_link", "achieved": round(value, 1), "peak": round(peak, 1), "unit": "GB/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "kernel": "swap_blocks_kernel (one launch per direction per step, two streams)",
                     "algorithmic_bytes_per_step": int(moved / K), "avg_step_ms": round(ms / K, 5),
                     "timing": f"CUDA events around {K} steps back to back",
                     "peak_source": "of measured in this run: cudaMemcpyAsync of one 256 MiB page-locked buffer "
                                    "to the device and one from it, at once on two streams (best of 5)",
                     "link_gbs": link},
        "e2e": {"value": round(sum_over_ranks(float(moved), world) / (e2e_ms / 1e3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d / K), "d2h_bytes_per_step": int(d2h / K),
                "note": "device time of the launches plus the host pool's swap decisions (pa_seq_swap for "
                        f"2 x {SWAP_GROUP} sequences, {pool_s * 1e6:.0f} us per step, measured before the "
                        "timed region); every copied byte crosses the host link"},
        "cpu_baseline": cpu,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def measure_link(torch, device, nbytes: int = 256 << 20, reps: int = 5) -> dict:
    """The host link's rate as the CUDA runtime reaches it: one contiguous page-locked buffer copied to the
    device, from it, and both at once on two streams (best of ``reps``, CUDA events)."""
    hbuf = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dbuf = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(2)]
    main = torch.cuda.current_stream(device)
    s2 = torch.cuda.Stream(device)

    def best(fn, moved):
        t = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(main)
            fn()
            b.record(main)
            torch.cuda.synchronize()
            t = min(t, a.elapsed_time(b))
        return round(moved / (t / 1e3) / 1e9, 1)

    def both():
        s2.wait_stream(main)
        dbuf[0].copy_(hbuf[0], non_blocking=True)
        with torch.cuda.stream(s2):
            hbuf[1].copy_(dbuf[1], non_blocking=True)
        main.wait_stream(s2)

    r = {"h2d_gbs": best(lambda: dbuf[0].copy_(hbuf[0], non_blocking=True), nbytes),
         "d2h_gbs": best(lambda: hbuf[1].copy_(dbuf[1], non_blocking=True), nbytes),
         "both_gbs": best(both, 2 * nbytes)}
    del hbuf, dbuf
    return r


_SWAP_POOLS: dict = {}


def time_swap_oracle(pairs_step, host_blocks: int, budget_s: float, nb: int = 20000):
    """The oracle's byte copy of one swap step (out and in) between two numpy pools of the workload's
    geometry, repeated for about ``budget_s`` seconds."""
    import oracle

    out_p, _, in_p, _ = pairs_step
    key = (nb, host_blocks)
    if _SWAP_POOLS.get("key") != key:
        rng = np.random.default_rng(0)
        _SWAP_POOLS.update(key=key, pools=(rng.integers(0, 2**16, (nb, 4, 16, 128), dtype=np.uint16),
                                           rng.integers(0, 2**16, (nb, 4, 16, 128), dtype=np.uint16),
                                           np.zeros((host_blocks, 4, 16, 128), np.uint16),
                                           np.zeros((host_blocks, 4, 16, 128), np.uint16)))
    dev_k, dev_v, host_k, host_v = _SWAP_POOLS["pools"]
    block_bytes = 4 * 16 * 128 * 2
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.swap_blocks(host_k, host_v, dev_k, dev_v, out_p)
        oracle.swap_blocks(dev_k, dev_v, host_k, host_v, in_p)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or reps >= 1000:
            break
    moved = reps * 2 * (len(out_p) + len(in_p)) * block_bytes
    return {"gbs": round(moved / dt / 1e9, 3), "pairs": len(out_p) + len(in_p), "reps": reps, "seconds": dt}


def run_reference(args, rank: int, world: int) -> None:
    """The oracle as the reference arm: each step decodes a bounded sample of the batch on the host cores."""
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    if args.workload == "swap_qwen":
        plan, host_blocks, _, _ = swap_plan(rank_seed(args.seed, 0), 2, model=True)
        _, _, in_p, _ = plan[1]
        out_p = plan[1][0]
        probe = time_swap_oracle((out_p[:64], None, in_p[:64], None), host_blocks, budget_s=0.5)
        s_per_pair = probe["seconds"] / (probe["reps"] * probe["pairs"])
        n_steps = args.warmup + args.steps
        # pairs per step (out and in each) so that warmup + steps take about a minute
        n = int(max(1, min(len(out_p), len(in_p), 60.0 / n_steps / s_per_pair / 2)))
        step_pairs = (out_p[:n], None, in_p[:n], None)
        for _ in range(args.warmup):
            time_swap_oracle(step_pairs, host_blocks, budget_s=0.0)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            time_swap_oracle(step_pairs, host_blocks, budget_s=0.0)
        dt = time.perf_counter() - t0
        value = round(args.steps * 2 * n * 2 * 4 * 16 * 128 * 2 / dt / 1e9, 4)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": WORKLOAD_DESCRIPTIONS[args.workload],
                                                "name": args.workload},
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                 "sample": f"{n} of {len(out_p)} pairs of swap step 1, out and in, per step; "
                                           "oracle byte copy between two numpy pools", "cpu_model": cpu_model()},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.workload.startswith("prefix_cow"):
        inp, tables, lens, slots, _, _ = prefix_batch(args.workload, rank_seed(args.seed, 0), model=True)
    else:
        inp = build_batch(args.workload, rank_seed(args.seed, 0))
        tables, lens, slots = pool_tables(inp, model=True)
    inp.block_tables = tables
    q_len = inp.q.shape[1] if inp.q.ndim == 4 else 1
    if slots is not None:
        oracle.write_kv(inp.new_key.reshape(-1, inp.num_kv_heads, inp.head_dim),
                        inp.new_value.reshape(-1, inp.num_kv_heads, inp.head_dim), inp.key_cache, inp.value_cache,
                        slots)

    fp8 = None
    if args.workload.endswith("_fp8"):
        # the oracle's own quantised pool (every slot through its writer), as the GPU arm's
        from paged_kv_cache_129_gb300 import workloads as wl

        nb_, hkv_, bs_, d_ = inp.key_cache.shape
        ks_, vs_ = wl.fp8_scales(inp.key_cache, inp.dtype), wl.fp8_scales(inp.value_cache, inp.dtype)
        kq, vq = np.zeros(inp.key_cache.shape, np.uint8), np.zeros(inp.key_cache.shape, np.uint8)
        oracle.write_kv_fp8(np.ascontiguousarray(inp.key_cache.transpose(0, 2, 1, 3).reshape(nb_ * bs_, hkv_, d_)),
                            np.ascontiguousarray(inp.value_cache.transpose(0, 2, 1, 3).reshape(nb_ * bs_, hkv_, d_)),
                            inp.dtype, kq, vq, ks_, vs_, np.arange(nb_ * bs_, dtype=np.int64))
        fp8 = (kq, vq, ks_, vs_)

    def one_row(h):
        if fp8 is not None:
            oracle.decode_fp8(inp.q, inp.dtype, fp8[0], fp8[1], fp8[2], fp8[3], inp.block_tables, inp.context_lens,
                              inp.scale, rows=[(0, h)])
        elif q_len == 1:
            oracle.decode_inputs(inp, rows=[(0, h)])
        else:  # one head, every query token
            oracle.decode_multi(inp.q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, inp.dtype,
                                inp.scale, rows=[(0, t, h) for t in range(q_len)])

    threads = os.cpu_count() or 1
    # size the per-step sample (heads of sequence 0, one task per head) so that warmup + steps
    # fit in about two minutes on `threads` threads
    t0 = time.perf_counter()
    one_row(0)
    t_row = max(time.perf_counter() - t0, 1e-4)
    n_steps = args.steps + args.warmup
    rows_per_step = int(max(1, min(inp.num_heads, 120.0 * threads / n_steps / t_row)))
    L0 = int(inp.context_lens[0])
    eb = inp.elem_bytes
    seq_bytes = (decode_bytes_fp8([L0], inp.num_heads, inp.num_kv_heads, inp.head_dim, eb, inp.block_size)
                 if fp8 is not None else
                 decode_bytes([L0], inp.num_heads, inp.num_kv_heads, inp.head_dim, eb, inp.block_size, q_len))
    bytes_per_step = rows_per_step / inp.num_heads * seq_bytes
    used = min(threads, rows_per_step)
    with ThreadPoolExecutor(max_workers=used) as ex:
        def one_step():
            list(ex.map(one_row, range(rows_per_step)))

        for _ in range(args.warmup):
            one_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            one_step()
        dt = time.perf_counter() - t0
    value = bytes_per_step * args.steps / dt / 1e9
    sample = (f"sequence 0 (L={L0}), {rows_per_step} of {inp.num_heads} heads per step, one head per task, "
              f"fp64 C oracle{' over its own E4M3 pool' if fp8 is not None else ''} on {used} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAMES[inp.dtype],
            "data": "synthetic",
            "config": {"workload": WORKLOAD_DESCRIPTIONS[args.workload], "name": args.workload},
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_DESCRIPTIONS), default="qwen_gqa")
    ap.add_argument("--kernel", choices=["auto", "mma", "simt"], default="auto")
    ap.add_argument("--partition-pages", type=int, default=0)
    ap.add_argument("--step", choices=["append", "write+decode"], default="append",
                    help="one fused call per step, or the write and the decode as two calls")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=5000)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="qwen_gqa: skip the FP8, verify and MHA side records of the default line")
    ap.add_argument("--no-long-context", action="store_true",
                    help="qwen_gqa: skip the long-context configuration timed in the same run")
    ap.add_argument("--fp8-layout", choices=["interleaved", "separate"], default="interleaved",
                    help="FP8 workloads: K and V of a (block, kv head) in one record, or two caches")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.workload == "swap_qwen":
            run_swap(args, rank, world, local_rank)
        elif args.workload == "qwen_gqa_layers28":
            run_layers(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
