"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any computation.

Recipe (shared by tests and the benchmark):

* ``numpy.random.default_rng(seed)`` draws the context lengths (where random)
  and then the block permutation. Each tensor (key cache, value cache, query,
  new-token keys, new-token values, in that order) gets its own child of
  ``SeedSequence(seed)``; its flattened elements are drawn in fixed chunks of
  2**20, chunk i from the i-th grandchild, so the values do not depend on how
  many threads fill them.
* q, K and V are drawn in float32 from N(0, 1) and cast to the workload dtype
  (round to nearest even). Every pool block is filled, including unused ones,
  so that unused blocks never act as zeros.
* Physical blocks come from a seeded permutation of the pool; each sequence's
  block table is filled in logical order from that permutation, so the pages of
  a sequence are scattered over the pool. Unused table entries hold -1.
* The cache layout is ``[num_blocks, num_kv_heads, block_size, head_dim]``
  (MiniPaged-Qwen page, section 8.2).

bf16 values are stored as their uint16 bit patterns (numpy has no bf16 type).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def _bf16_bits_inplace(x: np.ndarray) -> np.ndarray:
    """Round a finite float32 array to bfloat16 (nearest even), overwriting it; return the bits."""
    u = x.view(np.uint32)
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest even); return the uint16 bits."""
    x = np.array(x, dtype=np.float32, copy=True)
    if not np.isfinite(x).all():
        raise ValueError("bf16 input generation expects finite values")
    return _bf16_bits_inplace(x)


def cast_from_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Cast a float32 array to the storage form of ``dtype``."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x.astype(np.float16))
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def fp8_scales(cache: np.ndarray, dtype: str) -> np.ndarray:
    """Input construction for FP8 caches: a float32 scale per (block, kv head) that maps the
    largest magnitude of that block's source values onto 448, the largest E4M3 code
    (``cache`` is a source cache ``[N, H_kv, bs, d]`` in ``dtype`` storage form).  Choosing the
    scales is the caller's policy; this is the one the tests and the benchmark use."""
    if dtype == "bf16":
        vals = (cache.astype(np.uint32) << np.uint32(16)).view(np.float32)
    else:
        vals = cache.astype(np.float32)
    amax = np.abs(vals).max(axis=(2, 3))
    return (np.maximum(amax, np.float32(2.0 ** -10)) / np.float32(448.0)).astype(np.float32)


def default_scale(head_dim: int) -> float:
    """1/sqrt(d), rounded to float32 (the value the C ABI receives)."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


@dataclass
class DecodeInputs:
    """One batch of paged decode-attention inputs, in host (numpy) storage form."""

    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q: np.ndarray  # [B, Hq, d]
    key_cache: np.ndarray  # [num_blocks, Hkv, bs, d]
    value_cache: np.ndarray  # [num_blocks, Hkv, bs, d]
    block_tables: np.ndarray  # int32 [B, max_blocks_per_seq]
    context_lens: np.ndarray  # int32 [B]
    scale: float
    # Optional step write: the new token of every sequence (written before decode).
    new_key: Optional[np.ndarray] = None  # [B, Hkv, d]
    new_value: Optional[np.ndarray] = None  # [B, Hkv, d]
    new_token_pos: Optional[np.ndarray] = None  # int64 [B], logical position of the new token
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]


_CHUNK = 1 << 20
_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}


def _normal(ss: np.random.SeedSequence, shape, dtype: str) -> np.ndarray:
    """N(0,1) in float32, cast to ``dtype``; chunked and filled by a thread pool."""
    total = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(total, dtype=_STORAGE[dtype])
    n_chunks = (total + _CHUNK - 1) // _CHUNK
    children = ss.spawn(n_chunks)

    def fill(i: int) -> None:
        lo, hi = i * _CHUNK, min(total, (i + 1) * _CHUNK)
        x = np.random.Generator(np.random.PCG64(children[i])).standard_normal(hi - lo, dtype=np.float32)
        if dtype == "bf16":
            out[lo:hi] = _bf16_bits_inplace(x)  # a fresh N(0,1) draw is finite
        else:
            out[lo:hi] = x.astype(_STORAGE[dtype])

    if n_chunks <= 2:
        for i in range(n_chunks):
            fill(i)
    else:
        workers = max(1, min(n_chunks, os.cpu_count() or 1))
        with ThreadPoolExecutor(workers) as pool:
            list(pool.map(fill, range(n_chunks)))
    return out.reshape(shape)


def tables_from_permutation(perm: np.ndarray, context_lens: np.ndarray, block_size: int,
                            max_blocks: Optional[int] = None) -> np.ndarray:
    """Hand out ``perm`` in order: sequence 0 takes the first ceil(L0/bs) ids, and so on."""
    need = [(int(n) + block_size - 1) // block_size for n in context_lens]
    width = max(1, max(need) if need else 1) if max_blocks is None else max_blocks
    if sum(need) > len(perm):
        raise ValueError("pool too small for the requested context lengths")
    tables = np.full((len(context_lens), width), -1, dtype=np.int32)
    cursor = 0
    for b, n in enumerate(need):
        tables[b, :n] = perm[cursor:cursor + n]
        cursor += n
    return tables


def make_decode_inputs(name: str, *, context_lens, num_heads: int, num_kv_heads: int,
                       head_dim: int, block_size: int, dtype: str, num_blocks: Optional[int] = None,
                       pool_slack: float = 0.0, seed: int = 0,
                       with_new_token: bool = False, max_blocks: Optional[int] = None,
                       scale: Optional[float] = None, q_len: int = 1) -> DecodeInputs:
    """Build a seeded decode batch.

    ``context_lens`` may be a sequence of ints, or a callable that draws them
    from the workload's generator. Lengths are drawn first because they decide
    the pool size when ``num_blocks`` is None.
    """
    rng = np.random.default_rng(seed)
    streams = np.random.SeedSequence(seed).spawn(5)
    if callable(context_lens):
        lens = np.asarray(context_lens(rng), dtype=np.int32)
    else:
        lens = np.asarray(context_lens, dtype=np.int32)
    need = int(sum((int(n) + block_size - 1) // block_size for n in lens))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(need * (1.0 + pool_slack))))
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = tables_from_permutation(perm, lens, block_size, max_blocks)
    cache_shape = (num_blocks, num_kv_heads, block_size, head_dim)
    key_cache = _normal(streams[0], cache_shape, dtype)
    value_cache = _normal(streams[1], cache_shape, dtype)
    # q_len > 1: the queries of the last q_len positions of every sequence, [B, q_len, H_q, d]
    q_shape = (len(lens), num_heads, head_dim) if q_len == 1 else (len(lens), q_len, num_heads, head_dim)
    q = _normal(streams[2], q_shape, dtype)
    inp = DecodeInputs(name=name, dtype=dtype, num_heads=num_heads, num_kv_heads=num_kv_heads,
                       head_dim=head_dim, block_size=block_size, num_blocks=num_blocks, q=q,
                       key_cache=key_cache, value_cache=value_cache, block_tables=tables,
                       context_lens=lens, scale=default_scale(head_dim) if scale is None else scale)
    if with_new_token:
        # The new token of sequence b sits at logical position L_b - 1 (write, then attend);
        # with q_len > 1 the q_len new tokens sit at L_b - q_len .. L_b - 1 ([B, q_len, H_kv, d]).
        # Their slots are derived by the caller (a block pool, or a test's own translation).
        b_count = len(lens)
        shape = (b_count, num_kv_heads, head_dim) if q_len == 1 else (b_count, q_len, num_kv_heads, head_dim)
        inp.new_key = _normal(streams[3], shape, dtype)
        inp.new_value = _normal(streams[4], shape, dtype)
        inp.new_token_pos = (lens.astype(np.int64) - 1) if q_len == 1 else (
            lens.astype(np.int64)[:, None] - q_len + np.arange(q_len, dtype=np.int64)[None, :])
    return inp


# --- The five workloads -------------------------------------------------------------------

def tiny(seed: int = 0) -> DecodeInputs:
    """4 sequences with context lengths {1, 15, 16, 33}, 4 q / 2 kv heads, d 64, fp32, pool 16."""
    return make_decode_inputs("tiny", context_lens=[1, 15, 16, 33], num_heads=4, num_kv_heads=2,
                              head_dim=64, block_size=16, dtype="f32", num_blocks=16, seed=seed)


def qwen_gqa_verify(seed: int = 0, num_seqs: int = 64, q_len: int = 4) -> DecodeInputs:
    """The Qwen-style GQA batch in a speculative verify step: q_len new tokens per sequence
    (written, then attended causally), the same context-length distribution and pool."""
    return make_decode_inputs(f"qwen_gqa_verify{q_len}", context_lens=lambda r: r.integers(512, 4097, size=num_seqs),
                              num_heads=28, num_kv_heads=4, head_dim=128, block_size=16, dtype="bf16",
                              num_blocks=20000, seed=seed, with_new_token=True, q_len=q_len)


def qwen_gqa(seed: int = 0, num_seqs: int = 64) -> DecodeInputs:
    """Qwen-style GQA layer: 28 q / 4 kv heads, d 128, bf16, bs 16, L ~ U[512, 4096], pool 20000.

    One new token per sequence is written through ``slot_mapping`` before the
    decode; the context length includes it.
    """
    return make_decode_inputs("qwen_gqa", context_lens=lambda r: r.integers(512, 4097, size=num_seqs),
                              num_heads=28, num_kv_heads=4, head_dim=128, block_size=16, dtype="bf16",
                              num_blocks=20000, seed=seed, with_new_token=True)


def long_context(seed: int = 0, num_seqs: int = 8) -> DecodeInputs:
    """Long-context split-KV: 32 q / 8 kv heads, d 128, bf16, bs 16, L ~ U[32768, 131072].

    The pool holds exactly the blocks needed plus 1 %.
    """
    return make_decode_inputs("long_context", context_lens=lambda r: r.integers(32768, 131073, size=num_seqs),
                              num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16",
                              pool_slack=0.01, seed=seed)


def mha_lengths(rng: np.random.Generator, num_seqs: int) -> np.ndarray:
    """Lognormal context lengths, median 256 (mu = ln 256), sigma 1.0, clipped to [16, 2048]."""
    raw = rng.lognormal(mean=math.log(256.0), sigma=1.0, size=num_seqs)
    return np.clip(np.rint(raw), 16, 2048).astype(np.int32)


def mha_short(block_size: int = 16, seed: int = 0, num_seqs: int = 256) -> DecodeInputs:
    """Many short requests, MHA (LLaMA-7B layer): 32/32 heads, d 128, fp16, bs 16 or 32."""
    return make_decode_inputs(f"mha_short_bs{block_size}", context_lens=lambda r: mha_lengths(r, num_seqs),
                              num_heads=32, num_kv_heads=32, head_dim=128, block_size=block_size,
                              dtype="f16", pool_slack=0.25, seed=seed)


@dataclass
class PrefixWorkload:
    """Random payloads for the prefix-sharing + COW workload.

    The block tables come from a BlockPool: one parent sequence appends the
    shared prefix, 63 forks share it (refcount 64), then every sequence appends
    its private tail.
    """

    num_seqs: int
    prefix_len: int
    tail_lens: np.ndarray  # int32 [num_seqs], in [1, 256]
    num_blocks: int
    num_heads: int = 28
    num_kv_heads: int = 4
    head_dim: int = 128
    block_size: int = 16
    dtype: str = "bf16"
    key_cache: Optional[np.ndarray] = None  # initial cache (prefix tokens are written here)
    value_cache: Optional[np.ndarray] = None
    tail_key: Optional[np.ndarray] = None  # [sum(tail_lens), Hkv, d] in sequence order
    tail_value: Optional[np.ndarray] = None
    q: Optional[np.ndarray] = None


def prefix_cow(seed: int = 0, prefix_len: int = 2048, num_seqs: int = 64) -> PrefixWorkload:
    """64 sequences sharing a prefix (2048 tokens; the COW variant uses 2056) plus tails of 1..256."""
    rng = np.random.default_rng(seed)
    streams = np.random.SeedSequence(seed).spawn(5)
    tails = rng.integers(1, 257, size=num_seqs).astype(np.int32)
    bs, hkv, d = 16, 4, 128
    shared_blocks = (prefix_len + bs - 1) // bs
    # Private blocks: each tail needs at most ceil((prefix%bs + tail)/bs) + 1 blocks.
    private = int(sum((prefix_len % bs + int(t) + bs - 1) // bs + 1 for t in tails))
    num_blocks = shared_blocks + private + 8
    w = PrefixWorkload(num_seqs=num_seqs, prefix_len=prefix_len, tail_lens=tails, num_blocks=num_blocks)
    shape = (num_blocks, hkv, bs, d)
    w.key_cache = _normal(streams[0], shape, "bf16")
    w.value_cache = _normal(streams[1], shape, "bf16")
    w.q = _normal(streams[2], (num_seqs, w.num_heads, d), "bf16")
    total_tail = int(tails.sum())
    w.tail_key = _normal(streams[3], (total_tail, hkv, d), "bf16")
    w.tail_value = _normal(streams[4], (total_tail, hkv, d), "bf16")
    return w


WORKLOADS = {
    "tiny": tiny,
    "qwen_gqa": qwen_gqa,
    "long_context": long_context,
    "mha_short_bs16": lambda seed=0: mha_short(16, seed),
    "mha_short_bs32": lambda seed=0: mha_short(32, seed),
}
